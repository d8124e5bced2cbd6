// V forward + expectile loss + V backward without a context: the variant of
// ofrl_iql_value_fwd_bwd for callers that may not allocate device memory.
//
// Who needs it: code whose device memory is owned by someone else (a host
// application or framework that hands out all GPU memory from its own pool
// and forbids direct cudaMalloc), code recorded into a CUDA graph under the
// global capture mode (where cudaMalloc is refused), and latency-critical
// loops that cannot afford cudaMalloc's implicit device synchronisation.
// Creating an ofrl_ctx allocates, so those callers use this entry point.
//
// Its scratch (per-tile gradient partials, loss partials, reduction scratch)
// is one file-scope __device__ array of kScratchBytes, reserved in every GPU
// that loads this library for as long as the library stays loaded.  Host
// code cannot use the array's name as a device address, so the address is
// looked up once per device with cudaGetSymbolAddress, on the first call
// made with that device current.

#include <cstring>
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;   // OFRL_NOALLOC_SCRATCH_BYTES
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

inline size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct ScratchLayout {
    size_t partials, tile_loss, gram, scalars, counter, status, total;
};

ScratchLayout scratch_layout(int64_t part_stride, int n_tiles) {
    ScratchLayout L;
    size_t o = 0;
    L.partials = o; o = up256(o + (size_t)n_tiles * part_stride * sizeof(float));
    L.tile_loss = o; o = up256(o + (size_t)n_tiles * sizeof(float));
    L.gram = o; o = up256(o + (size_t)ofrl::kMaxGramBlocks * ofrl::kGramStride * sizeof(float));
    L.scalars = o; o = up256(o + (size_t)ofrl::kScalars * sizeof(float));
    L.counter = o; o = up256(o + sizeof(unsigned int));
    L.status = o; o = up256(o + OFRL_STAT_WORDS * sizeof(int32_t));
    L.total = o;
    return L;
}

// Device address of the scratch array on the current device (looked up once).
ofrl_status scratch_for_current_device(unsigned char** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OFRL_ECUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return OFRL_ECUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    return OFRL_OK;
}

}  // namespace

extern "C" {

int64_t ofrl_noalloc_max_batch(const ofrl_vshape* shape) {
    if (shape == nullptr || shape->state_dim < 1 || shape->state_dim > ofrl::kMaxStateDim) return -1;
    if (shape->hidden != 64 && shape->hidden != 128 && shape->hidden != 256) return -1;
    const int tm = ofrl::vnet_tile_rows(shape->hidden);
    const int64_t stride = ofrl::part_stride_of(ofrl::n_params_of(shape->state_dim, shape->hidden));
    int n = 0;
    while (scratch_layout(stride, n + 1).total <= kScratchBytes) ++n;
    return (int64_t)n * tm;
}

ofrl_status ofrl_iql_value_fwd_bwd_noalloc(const ofrl_vshape* shape, const float* params, const float* states,
                                           int32_t state_stride, int32_t batch, const float* q_taken, float tau,
                                           float* v_out, float* loss_out, float* grad_out, void* stream) {
    if (shape == nullptr || !params || !states || !q_taken || !v_out || !loss_out || !grad_out) return OFRL_EINVAL;
    if (shape->state_dim < 1 || shape->state_dim > ofrl::kMaxStateDim || state_stride < shape->state_dim)
        return OFRL_EINVAL;
    if (shape->prec != OFRL_PREC_FP32 && shape->prec != OFRL_PREC_BF16) return OFRL_EINVAL;
    if (shape->hidden != 64 && shape->hidden != 128 && shape->hidden != 256) return OFRL_EUNSUPPORTED;
    if (batch < 1 || !(tau >= 0.0f && tau <= 1.0f)) return OFRL_EINVAL;
    const int tm = ofrl::vnet_tile_rows(shape->hidden);
    const int n_tiles = (batch + tm - 1) / tm;
    const int64_t P = ofrl::n_params_of(shape->state_dim, shape->hidden);
    const int64_t stride = ofrl::part_stride_of(P);
    const ScratchLayout L = scratch_layout(stride, n_tiles);
    if (L.total > kScratchBytes) return OFRL_EINVAL;   // batch above ofrl_noalloc_max_batch(shape)

    unsigned char* base = nullptr;
    const ofrl_status s = scratch_for_current_device(&base);
    if (s != OFRL_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* partials = reinterpret_cast<float*>(base + L.partials);
    float* tile_loss = reinterpret_cast<float*>(base + L.tile_loss);
    unsigned int* counter = reinterpret_cast<unsigned int*>(base + L.counter);
    int32_t* status = reinterpret_cast<int32_t*>(base + L.status);
    // the reduction's block ticket must start at zero; the rest is overwritten
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), st) != cudaSuccess) return OFRL_ECUDA;

    ofrl::VnetLaunch v;
    std::memset(&v, 0, sizeof(v));
    v.params[0] = params;
    v.tau[0] = tau;
    v.n_nets = 1;
    v.state_dim = shape->state_dim;
    v.hidden = shape->hidden;
    v.num_actions = shape->num_actions;
    v.prec = shape->prec;
    v.states = states;
    v.stride = state_stride;
    v.batch = batch;
    v.q_taken = q_taken;
    v.v_out = v_out;
    v.partials = partials;
    v.tile_loss = tile_loss;
    v.part_stride = stride;
    v.net_partial_stride = (int64_t)n_tiles * stride;
    v.net_tile_stride = n_tiles;
    v.status = status;
    if (ofrl::launch_vnet_fwd_bwd(v, st) != cudaSuccess) return OFRL_ECUDA;

    ofrl::ReduceLaunch r;
    std::memset(&r, 0, sizeof(r));
    r.n_nets = 1;
    r.P = P;
    r.n_tiles = n_tiles;
    r.partials = partials;
    r.part_stride = stride;
    r.net_partial_stride = v.net_partial_stride;
    r.tile_loss = tile_loss;
    r.net_tile_stride = n_tiles;
    r.inv_batch = 1.0f / (float)batch;
    r.g0_out[0] = grad_out;
    r.n_src = 0;
    r.max_grad_norm = INFINITY;
    r.gram_part = reinterpret_cast<float*>(base + L.gram);
    r.scalars = reinterpret_cast<float*>(base + L.scalars);
    r.counter = counter;
    r.loss_out = loss_out;
    return ofrl::launch_reduce_gram(r, st) == cudaSuccess ? OFRL_OK : OFRL_ECUDA;
}

}  // extern "C"
