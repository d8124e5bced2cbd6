// Shared device helpers and the context layout of the ofrl library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ofrl.h"

namespace ofrl {

constexpr int kMaxNets = 2;
constexpr int kMaxSrc = 4;        // primary + up to three auxiliary sources
constexpr int kGramPairs = 10;    // upper triangle of a 4x4 Gram matrix
constexpr int kGramStride = 16;   // floats per block's Gram partial (padded: four 16-byte loads)
constexpr int kMaxGramBlocks = 2048;   // cap of the reduce grid: Gram partials any scratch must hold per network
constexpr int kScalars = 32;      // per-network scalar slots (see Scalar)
constexpr int kMaxActions = 16;
constexpr int kMaxStateDim = 64;

// Per-network scalar slots written by the reduction's last block.
enum Scalar {
    SC_NORM0 = 0,     // n_0 .. n_3 (pre-clip source norms)
    SC_COEF0 = 4,     // alpha_k * s_k .. (4 slots)
    SC_COMBINED = 8,  // ||G||
    SC_LOSS = 9,      // mean expectile loss
};

// Upper-triangle index of the pair (j, k), j <= k < 4.
__host__ __device__ constexpr int gram_index(int j, int k) {
    return j * 4 - (j * (j - 1)) / 2 + (k - j);
}

struct Workspace {
    float* partials;      // [max_nets][max_tiles][P] per-tile gradient partials
    float* tile_loss;     // [max_nets][max_tiles] per-tile sum of w d^2
    float* g0;            // [max_nets][P] primary gradient when the caller gives no buffer
    float* gram_part;     // [max_nets][max_gram_blocks][kGramStride]
    float* scalars;       // [max_nets][kScalars]
    unsigned int* counter;  // [max_nets] last-block tickets (reset by the last block)
    int32_t* status;      // [OFRL_STAT_WORDS]
    uint8_t* img;         // [max_nets] packed bf16 weight images for the tensor-core kernels
    uint8_t* ximg;        // [128-row tiles] bf16 images of the relabelled state tiles
    uint8_t* act[3];      // layered tensor-core path: h1, dz2, dz1 images [max_nets][128-row tiles]
    float* tvec;          // layered path: per-tile dW3, db2 column sums and db3 [max_nets][tiles][tvec_stride]
    float* qbuf;          // [max_batch][A] Q staged from host memory by the relabel (train step)
    unsigned long long* barrier;  // grid-barrier arrival counter of the fused reduce + Adam (only grows)
};

}  // namespace ofrl

namespace ofrl {

// Which V forward/backward implementation a step uses.
enum VnetPath : int32_t {
    PATH_AUTO = 0,      // fused tensor-core kernel for H <= 128, layered for H = 256, else CUDA cores
    PATH_FUSED = 1,     // vnet_tc.cu: one CTA per tile does all five GEMMs (H = 128; 64 padded)
    PATH_LAYERED = 2,   // vnet_wide.cu: per-tile forward/backward, then split-K weight gradients
    PATH_SIMT = 3,      // vnet_simt.cu: CUDA cores
};

// Tensor maps of the layered path (5-D: core matrix, chunk, row group,
// plane, tile or network), each with the box one of its loads uses.
struct alignas(128) WideMaps {
    CUtensorMap h1k, dz2k;      // activation K-chunks: all 128 rows x 16 columns
    CUtensorMap dz2h, dz1h;     // activation MN-chunks: 16 rows x 128 columns (a half of H)
    CUtensorMap h1n;            // activation MN-chunks: 16 rows x H columns
    CUtensorMap xk;             // state-image MN-chunks: 16 rows x 64 columns
    CUtensorMap w2k, w2n;       // W2 image: K-chunks (H rows x 16) and MN-chunks (16 rows x H)
};

}  // namespace ofrl

struct ofrl_ctx {
    int device;
    int num_sms;
    ofrl_vshape shape;
    int32_t max_batch;
    int32_t max_nets;
    int32_t max_tiles;
    int32_t max_gram_blocks;
    int64_t n_params;
    void* base;           // the single cudaMalloc of the context
    int64_t bytes;
    ofrl::Workspace ws;
    int32_t vnet_path;          // ofrl::VnetPath requested (PATH_AUTO unless selected)
    // the last launch of this context was the optimizer kernel of a train
    // step on early_stream: the next step's relabel rows may start early
    int32_t early_ok;
    void* early_stream;
    int32_t act_tiles;          // 128-row tiles per network in ws.act / ws.tvec
    int32_t tvec_stride;
    ofrl::WideMaps* maps;       // tensor maps of the layered path (null: not available)
    uint64_t barrier_arrivals;  // arrivals the launched fused kernels add to ws.barrier
    // self-test of the bounded grid barrier (ofrl_selftest_barrier): its wait
    // limit, and 1 to give the next fused reduce + Adam launches a target one
    // above the arrivals their grid can make
    uint64_t barrier_wait_ns;
    int32_t barrier_unreachable;
    // measurement hooks: events[step][OFRL_PHASES + 1] while profiling
    cudaEvent_t* prof_events;
    int32_t prof_max;
    int32_t prof_count;
};

namespace ofrl {

// ---- counter-based RNG: SplitMix64 (Steele, Lea & Flood 2014) -----------
__host__ __device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
// Output number (counter + 1) of SplitMix64 seeded with `seed`.
__host__ __device__ __forceinline__ uint64_t sm64_at(uint64_t seed, uint64_t counter) {
    return sm64_mix(seed + (counter + 1ull) * 0x9E3779B97F4A7C15ull);
}
// Lemire multiply-shift on the top 32 bits: uniform-ish in [0, n), n <= 2^32.
__host__ __device__ __forceinline__ uint32_t below(uint64_t r, uint64_t n) {
    return (uint32_t)(((r >> 32) * n) >> 32);
}

__device__ __forceinline__ float to_bf16_rn(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Column sums over the 32 rows of a warp: v[j] (16 columns per lane) ->
// lane l returns the sum of column (l >> 1) & 15 (lanes l and l ^ 1 agree).
__device__ __forceinline__ float colsum16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16, n = 16; o >= 2; o >>= 1, n >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float give = up ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Clip scale of the pages' formula: (n > c && n > 0) ? c / n : 1.
__device__ __forceinline__ float clip_scale(float n, float c) {
    return (n > c && n > 0.0f) ? c / n : 1.0f;
}

// Programmatic dependent launch: a kernel launched with launch_pdl may start
// while the previous kernel in the stream finishes; pdl_wait() blocks until
// that kernel has completed and its writes are visible (a no-op when there is
// no such kernel), so everything that reads or writes global memory comes
// after it.  pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Every kernel of the library asks for the largest shared-memory carveout,
// so consecutive kernels never make an SM reconfigure its L1 / shared split
// (the tensor-core kernel needs ~200 KB of shared memory).
template <typename K>
inline cudaError_t set_max_shared_carveout(K kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

template <typename Arg>
inline cudaError_t launch_pdl(void (*kernel)(Arg), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Arg arg) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, arg);
}

template <typename Arg0, typename Arg1>
inline cudaError_t launch_pdl(void (*kernel)(Arg0, Arg1), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Arg0 a0, Arg1 a1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a0, a1);
}

// Launch with programmatic dependent launch and, optionally, thread-block
// clusters of `cluster` CTAs along x (cluster > 1) or a cooperative launch
// (every CTA resident at once; the two are exclusive here).
template <typename... Params, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             unsigned cluster, bool cooperative, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned n = 1;
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    } else if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

inline int64_t n_params_of(int s, int h) {
    return (int64_t)h * s + h + (int64_t)h * h + h + h + 1;
}
// Per-tile stride of the gradient partials: P rounded up to 32 floats, so
// every tile's slice starts on a 128-byte boundary.
inline int64_t part_stride_of(int64_t p) { return (p + 31) / 32 * 32; }

// Offsets of the six tensors inside the flat parameter / gradient buffer.
struct Offsets {
    int64_t w1, b1, w2, b2, w3, b3, total;
};
__host__ __device__ inline Offsets offsets_of(int s, int h) {
    Offsets o;
    o.w1 = 0;
    o.b1 = o.w1 + (int64_t)h * s;
    o.w2 = o.b1 + h;
    o.b2 = o.w2 + (int64_t)h * h;
    o.w3 = o.b2 + h;
    o.b3 = o.w3 + h;
    o.total = o.b3 + 1;
    return o;
}

}  // namespace ofrl

// Launch helpers (defined in the .cu files), called from api.cu.
namespace ofrl {

struct HerLaunch {
    const float* states;
    const float* next_states;
    const int32_t* actions;
    const float* rewards;
    const float* dones;
    const int32_t* episode_ends;
    int32_t capacity;
    int32_t num_episodes;
    int32_t state_dim;
    int32_t in_stride;
    int32_t goal_dim;
    int32_t batch;
    int32_t first_her;
    int32_t strategy;
    float threshold;
    uint64_t seed;
    uint64_t step;
    float* out_states;
    float* out_next_states;
    int32_t* out_actions;
    float* out_rewards;
    float* out_dones;
    int32_t* out_src;
    int32_t* out_donor;
    int32_t out_stride;
    int32_t copy_cols;      // columns copied per row (multiple of 4, <= 64)
    int32_t search_rounds;  // 16-ary search rounds that shrink num_episodes to <= 16
    int32_t* status;
    // optional: bf16 images of the relabelled states per 128-row tile, for
    // the tensor-core V kernel (rows past the batch are zero), and packed
    // weight images made by extra blocks of the same grid
    uint8_t* ximg;          // null: no images
    int32_t img_planes;     // 3 (fp32 workloads) or 1 (bf16)
    int32_t img_rows;       // batch rounded up to a whole tile
    int32_t relabel_blocks; // blocks doing rows; the rest pack weights
    int32_t pack_blocks;
    int32_t pack_nets;
    const float* pack_params[kMaxNets];
    uint8_t* wimg;          // per network: W1 image then W2 image
    int32_t early;          // 1: the row blocks do not wait for the previous kernel (see her_relabel_kernel)
    int32_t pack_hidden;    // H of the network
    int32_t pack_width;     // units of the packed images (>= H; the rest zero)
    // optional: caller-given sources (e.g. PER-sampled) and importance
    // weights; HER rows get weight 1
    const int32_t* src_in;  // [batch] or null: sources drawn here
    const float* isw_in;    // [batch] or null: weight 1 for every row
    float* isw_out;         // [batch] or null
    // optional: Q [batch][q_cols] in host memory, copied to q_dst by the row
    // blocks (the train step's V kernel then reads device memory)
    const float* q_src;
    float* q_dst;
    int32_t q_cols;
};
cudaError_t launch_episode_ends_append(const float* dones, int64_t first_index, int32_t n, int32_t* episode_ends,
                                       int32_t* num_episodes, int32_t max_episodes, int32_t* status,
                                       cudaStream_t st);
cudaError_t launch_her_relabel(const HerLaunch& a, cudaStream_t st);

struct VnetLaunch {
    const float* params[kMaxNets];
    float tau[kMaxNets];
    int n_nets;
    int state_dim, hidden, num_actions, prec;
    const float* states;
    int32_t stride;
    int32_t batch;
    const float* q_taken;      // [B] (standalone) or null
    const float* q;            // [B, A] (fused step) or null
    const int32_t* actions;    // [B] with q
    float beta;
    float* v_out;              // [n_nets, B] or null
    float* pi_out;             // [n_nets, B, A] or null
    int32_t* argmax_out;       // [n_nets, B] or null
    float* partials;           // [n_nets][n_tiles][part_stride]
    float* tile_loss;          // [n_nets][n_tiles]
    const uint8_t* ximg;       // tensor-core kernel: state tile images from the relabel (or null)
    int64_t part_stride;       // floats between tiles in partials (P rounded up to 32)
    int64_t net_partial_stride;  // floats between networks in partials
    int32_t net_tile_stride;     // floats between networks in tile_loss
    int32_t* status;
    int32_t path;                // VnetPath chosen for this launch (never PATH_AUTO)
    // layered tensor-core path
    uint8_t* act[3];             // h1, dz2, dz1 images [n_nets][act_tiles][planes][128 x H]
    float* tvec;                 // [n_nets][act_tiles][tvec_stride]: dW3 and db2 column sums, db3
    int32_t tvec_stride;
    int32_t act_tiles;
    int32_t n_ranges;            // K-ranges of the weight-gradient kernel (its partials per network)
    const WideMaps* maps;        // the context's tensor maps (host memory)
    // forward-only launches (launch_vnet_forward): the IQL target inputs
    const float* rewards;        // [B] or null
    const float* dones;          // [B] or null
    float gamma;
    float* target_out;           // [n_nets, B] or null
};
int vnet_tile_rows(int hidden);
cudaError_t launch_vnet_fwd_bwd(const VnetLaunch& a, cudaStream_t st);
// V forward only (CUDA cores, every hidden size): v_out and, with target_out,
// rewards + gamma (1 - dones) V.
cudaError_t launch_vnet_forward(const VnetLaunch& a, cudaStream_t st);
// V forward only on the tensor cores (hidden 64 or 128, S <= 64; one
// network): packs the weight images into img, then one launch; v_out and,
// with target_out, rewards + gamma (1 - dones) V.
cudaError_t launch_vnet_tc_forward(const VnetLaunch& a, uint8_t* img, cudaStream_t st);
// tensor-core kernel (hidden 128): packed weight images per network
int64_t vnet_tc_image_bytes();
bool vnet_tc_supported(const VnetLaunch& a);
cudaError_t launch_vnet_tc_pack(const VnetLaunch& a, uint8_t* img, cudaStream_t st);
cudaError_t launch_vnet_tc(const VnetLaunch& a, const uint8_t* img, cudaStream_t st);
// Layered tensor-core path (hidden 128 or 256, state_dim < 64): workspace
// sizes, tensor maps over the context's buffers, weight and state-image
// packing for standalone calls, and the two kernels.
bool vnet_wide_supported(const VnetLaunch& a);
int64_t vnet_wide_act_bytes(int hidden, int planes);     // one 128-row tile of one activation image
int32_t vnet_wide_tvec_stride(int hidden);
cudaError_t vnet_wide_maps(WideMaps* m, int hidden, int planes, int n_nets, int act_tiles, uint8_t* const act[3],
                           uint8_t* ximg, int x_tiles, uint8_t* wimg);
int vnet_wide_ranges(const VnetLaunch& a, int num_sms);  // partials per network the weight-gradient kernel writes
cudaError_t launch_vnet_wide_pack(const VnetLaunch& a, uint8_t* wimg, uint8_t* ximg, cudaStream_t st);
cudaError_t launch_vnet_wide(const VnetLaunch& a, const uint8_t* wimg, cudaStream_t st);
// CTAs per network of the fused tensor-core kernel (its gradient partials
// per network): one wave of one CTA per SM, each CTA running an equal share
// of the n_tiles tiles back to back.
int vnet_tc_ctas(int n_tiles, int n_nets);

struct ReduceLaunch {
    int n_nets;
    int64_t P;
    int n_tiles;                 // tiles: entries of tile_loss per network
    int n_parts;                 // gradient partials per network (0: n_tiles)
    const float* partials;       // [n_nets][n_parts][part_stride]; null: g0 is given in src[.][0]
    int64_t part_stride;
    int64_t net_partial_stride;
    const float* tile_loss;      // [n_nets][n_tiles] or null
    int32_t net_tile_stride;
    float inv_batch;
    float* g0_out[kMaxNets];     // where the reduced primary is written (if partials)
    const float* src[kMaxNets][kMaxSrc];  // sources; src[n][0] ignored when partials != null
    int n_src;
    float budget[kMaxSrc];
    float alpha[kMaxSrc];
    float max_grad_norm;
    float* gram_part;            // [n_nets][grid][kGramStride]
    float* scalars;              // [n_nets][kScalars]
    unsigned int* counter;       // [n_nets]
    float* norms_out;            // [n_nets][5] or null: n_0..n_3, combined
    float* loss_out;             // [n_nets] or null
    int sanitize;                // 1: non-finite source elements count as 0
    int32_t* status;             // counts them (OFRL_STAT_SANITIZED) when sanitize
};
int reduce_grid(int64_t P, int elem_lanes);
cudaError_t launch_reduce_gram(const ReduceLaunch& a, cudaStream_t st);

struct AdamLaunch {
    int n_nets;
    int64_t n;
    float* p[kMaxNets];
    float* m[kMaxNets];
    float* v[kMaxNets];
    const float* src[kMaxNets][kMaxSrc];
    int n_src;
    const float* scalars;        // [n_nets][kScalars]: coefficients and the combined norm
    const float* grad_norm;      // standalone: device scalar or null (then scalars[SC_COMBINED])
    float lr[kMaxNets], bc1[kMaxNets], bc2[kMaxNets];
    float beta1, beta2, eps, weight_decay, max_grad_norm;
    int32_t* status;
    int sanitize;                // 1: non-finite source elements count as 0
    float clamp;                 // > 0: |p| <= clamp after the update
    float* target[kMaxNets];     // Polyak target per network, or null
    float polyak[kMaxNets];
    uint64_t wait_ns;            // fused reduce + Adam: how long a CTA waits at the grid barrier
};
cudaError_t launch_target_ema(const float* p, float* target, int64_t n, float polyak, cudaStream_t st);
cudaError_t launch_adam(const AdamLaunch& a, cudaStream_t st);
// Adam bias corrections 1 - beta^t, computed in double and rounded to float.
void bias_corrections(float beta1, float beta2, int32_t t, float* bc1, float* bc2);
// Reduce + Gram + norms and Adam in one cooperative launch (a grid barrier
// between them): possible when one pass of the reduce grid covers P and the
// grid fits on the device at once.  barrier_base: arrivals before this launch.
bool reduce_adam_fusable(const ReduceLaunch& r);
int reduce_adam_blocks(const ReduceLaunch& r);   // CTAs of that launch
cudaError_t launch_reduce_adam(const ReduceLaunch& r, const AdamLaunch& a, unsigned long long* barrier,
                               unsigned long long barrier_base, cudaStream_t st);

struct CombineLaunch {
    int64_t n;
    const float* src[kMaxSrc];
    int n_src;
    const float* scalars;
    float* out;
    float* norms_out;            // [n_src + 1] or null
};
cudaError_t launch_combine(const CombineLaunch& a, cudaStream_t st);

cudaError_t launch_expectile(const float* q_taken, const float* v, int batch, float tau,
                             float* loss_out, float* dv_out, cudaStream_t st);
cudaError_t launch_policy(const float* q, const float* v, int batch, int num_actions, float beta,
                          float* pi_out, int32_t* argmax_out, int64_t net_stride_v,
                          int n_nets, cudaStream_t st);

}  // namespace ofrl
