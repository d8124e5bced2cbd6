// IQL value network V(s) forward, expectile loss, policy and backward on the
// 5th-generation tensor cores, in layers, for hidden widths whose operands do
// not fit one CTA's shared memory together (H = 256; H = 128 can take this
// path too).
//
// Method: "GPU IQL + HER Porting Plan", "IQL (CPU)" items 1-3 and "CUDA
// Kernel: iql_value_kernel.cu"; the same results as the fused tensor-core
// kernel (vnet_tc.cu) and the CUDA-core kernel (vnet_simt.cu) to fp32
// rounding.
//
// Kernel A, one CTA per 128-row batch tile (TMEM: z1 / dh1, z2):
//   G1  z1  = X . W1^T          X and W1 whole in shared memory
//       h1  = relu(z1 + b1)     -> global image; ReLU mask kept in registers
//   G2  z2  = h1 . W2^T         h1 and W2 streamed in K-chunks of 16 (TMA)
//       V, loss, dV, dz2 = dV w3 1[z2 > 0] -> global image; the tile's
//       column sums for dW3 and db2 and its db3
//   G4  dh1 = dz2 . W2          dz2 and W2 (MN-major) streamed (TMA); the
//       policy meanwhile
//       dz1 = dh1 1[z1 > 0]     -> global image
// Kernel B, split-K over the batch: CTA (range r, half h of the hidden units)
//   accumulates in TMEM over the 16-row K-steps of its range
//       dW2[h] = dz2[:, h]^T . h1      dW1[h] = dz1[:, h]^T . X
//   (the state image's ones column makes dW1's last column db1), adds the
//   tile vectors of its range and writes gradient partial row r.
//
// Images in global memory have the core-matrix layout of the shared-memory
// operands (tc_image.cuh), one 128-row tile after another.  5-D tensor maps
// (core matrix, chunk, row group, plane, tile) cut from one image either
// K-major chunks (all 128 rows x 16 columns) or MN-major chunks (16 rows x
// some or all columns), so the image written once serves both kinds of GEMM.
// fp32 precision as in the fused kernel: three bf16 planes per operand and
// six products per K-step; the weight-gradient kernel, whose K is the batch,
// issues the three leading ones, so it loads the two planes they read, and
// the dz1 image, which only that kernel reads, is written in two; the bf16
// workload has one plane and one product.

#include <cuda.h>

#include "common.cuh"
#include "tc_image.cuh"
#include "umma.cuh"

namespace ofrl {
namespace {

using tc::KX;
using tc::TM;

constexpr int kThreads = 544;     // warp 0: TMA and MMA issue, TMEM; warps 1..16: epilogues
constexpr int kEpiWarps = 16;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_Z1 = 0, TM_Z2 = 256;   // kernel A (TM_Z1 also holds dh1)
constexpr uint32_t TM_D2 = 0, TM_D1 = 256;   // kernel B
constexpr int kStagesA = 4;                  // K-chunks in flight, kernel A
constexpr int kStagesB = 3;                  // K-steps in flight, kernel B
constexpr int kWaysPerTile = TM / 16;        // K-steps per tile (kernel B)
constexpr uint64_t kWaitNs = 1000000000ull;  // bounded waits: 1 s

template <int H, int NP>
struct Geo {
    static_assert(H == 128 || H == 256, "layered path: hidden 128 or 256");
    static constexpr int kChunks = H / 16;                   // K-chunks of G2 and G4
    static constexpr int kCols = H / 4;                      // columns per epilogue warp
    static constexpr int kPieces = kCols / 16;
    static constexpr int kHalves = H / 128;
    // kernel A
    static constexpr uint32_t kPlaneA = TM * 16 * 2;         // activation K-chunk, one plane
    static constexpr uint32_t kPlaneB = H * 16 * 2;          // W2 chunk (either major), one plane
    static constexpr uint32_t kBytesA = NP * kPlaneA, kBytesB = NP * kPlaneB;
    static constexpr uint32_t kStageA = kBytesA + kBytesB;
    static constexpr uint32_t kPlaneX = TM * KX * 2, kPlaneW1 = H * KX * 2;
    static constexpr uint32_t kXBytes = NP * kPlaneX, kW1Bytes = NP * kPlaneW1;
    // kernel B: dz2 half, h1, dz1 half, X (16 rows each), the planes its
    // three leading products read (two of three)
    static constexpr int kNPB = NP == 3 ? 2 : 1;
    static constexpr uint32_t kPlaneHalf = 16 * 128 * 2, kPlaneN = 16 * H * 2, kPlaneXK = 16 * KX * 2;
    static constexpr uint32_t kOffB2 = kNPB * kPlaneHalf, kOffA1 = kOffB2 + kNPB * kPlaneN,
                              kOffB1 = kOffA1 + kNPB * kPlaneHalf;
    static constexpr uint32_t kStageB = kOffB1 + kNPB * kPlaneXK;
    static constexpr uint32_t kActPlane = TM * H * 2;        // one plane of a tile image
    static constexpr int kStride2 = H + 4;                   // staged dW2 rows (floats)
    // the stage rings, also holding kernel A's X and W1 images at the start
    // and kernel B's staged dW2 and dW1 rows (S <= 63) at the end
    static constexpr uint32_t kStaged = (uint32_t)(128 * kStride2 + 128 * 63) * 4;
    static constexpr uint32_t kRingA =
        kStagesA * kStageA > kXBytes + kW1Bytes ? kStagesA * kStageA : kXBytes + kW1Bytes;
    static constexpr uint32_t kRingB = kStagesB * kStageB > kStaged ? kStagesB * kStageB : kStaged;
};

template <int H, int NP>
struct SmemA {
    uint8_t ring[Geo<H, NP>::kRingA];   // stage s at s * kStageA; first the X image then the W1 image
    float b1[H], b2[H], w3[H];
    float vsum[4][TM];
    float red[2][kEpiWarps][H / 4];   // per epilogue warp column sums: dW3, db2
    float lred[2][4];
    float qt[TM * kMaxActions];
    int32_t act[TM];
    float vrow[TM];
    uint64_t full[kStagesA], empty[kStagesA], bar_mma, bar_load;
    uint64_t piece[2][4];   // round p of the h1 / dz2 pieces written (one arrival per epilogue warp)
    uint32_t tmem_slot;
};

template <int H, int NP>
struct SmemB {
    uint8_t ring[Geo<H, NP>::kRingB];   // stage s at s * kStageB; at the end the staged dW2 / dW1 rows
    __align__(16) float vec[3][128];                // the range's dW3, db2, db1 entries of the half
    float b3;
    uint64_t full[kStagesB], empty[kStagesB], bar_mma;
    uint32_t tmem_slot;
};

// The shared-memory budget and the chunk shapes, checked at compile time:
// each box of the tensor maps lands exactly in its slot.
template <int H, int NP>
struct Checks {
    using G = Geo<H, NP>;
    static_assert(sizeof(SmemA<H, NP>) <= 227 * 1024, "layered kernel A shared memory");
    static_assert(sizeof(SmemB<H, NP>) <= 227 * 1024, "layered kernel B shared memory");
    static_assert(G::kChunks >= kStagesA, "ring shorter than a GEMM");
    static_assert(G::kStageA % 1024 == 0 && G::kStageB % 1024 == 0, "stages stay 1 KB aligned");
    static constexpr bool ok = true;
};

__device__ __forceinline__ uint64_t desc(const uint8_t* p, uint32_t lbo, uint32_t sbo) {
    return umma::smem_desc(umma::smem_u32(p), lbo, sbo);
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, bool ok) {
    return ok && umma::mbar_wait(bar, parity, kWaitNs);
}

// Named barrier of the 16 epilogue warps (warp 0 keeps issuing).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Products of one K-step, smallest first: (A term, B term) = (2,0), (1,1),
// (0,2), (1,0), (0,1), (0,0); NP == 1: the one product (0,0).
__host__ __device__ constexpr int term_a(int t) { return t == 0 ? 2 : (t == 1 || t == 3) ? 1 : 0; }
__host__ __device__ constexpr int term_b(int t) { return t == 2 ? 2 : (t == 1 || t == 4) ? 1 : 0; }

// Store 16 fp32 values of row r, columns c0..c0+15 into a global tile image
// with C columns (NP planes of `plane` bytes).
template <int NP, bool LEADING = false>
__device__ __forceinline__ void store16_global(uint8_t* img, uint32_t plane, int C, int r, int c0,
                                               const float (&v)[16], uint64_t pol) {
    constexpr int NW = NP == 3 && LEADING ? 2 : NP;
    uint32_t t[NP][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if constexpr (NP == 3 && LEADING) tc::split2x2(v[2 * j], v[2 * j + 1], t[0][j], t[1][j]);
        else if constexpr (NP == 3) tc::split3x2(v[2 * j], v[2 * j + 1], t[0][j], t[1][j], t[2][j]);
        else t[0][j] = tc::pack_bf16x2(v[2 * j], v[2 * j + 1]);
    }
    const uint32_t o0 = tc::img_off(r, c0, C), o1 = tc::img_off(r, c0 + 8, C);
#pragma unroll
    for (int p = 0; p < NW; ++p) {
        umma::st16_hint(img + (uint32_t)p * plane + o0, make_uint4(t[p][0], t[p][1], t[p][2], t[p][3]), pol);
        umma::st16_hint(img + (uint32_t)p * plane + o1, make_uint4(t[p][4], t[p][5], t[p][6], t[p][7]), pol);
    }
}

// Kernel A's loads of chunk j of G2 (h1 and W2 K-chunks) or G4 (dz2 K-chunk,
// W2 MN-chunk) into stage s: the W2 part (`w`) and the activation part
// (`x`) can go separately; the first of them announces the stage's bytes.
template <int H, int NP, bool G4>
__device__ __forceinline__ void load_w(SmemA<H, NP>& sm, const WideMaps& mp, int s, int j, int net) {
    using G = Geo<H, NP>;
    umma::mbar_expect_tx(&sm.full[s], G::kStageA);
    if constexpr (G4) umma::tma_load5(sm.ring + s * G::kStageA + G::kBytesA, &mp.w2n, 0, 0, 2 * j, 0, net, &sm.full[s]);
    else umma::tma_load5(sm.ring + s * G::kStageA + G::kBytesA, &mp.w2k, 0, 2 * j, 0, 0, net, &sm.full[s]);
}
template <int H, int NP, bool G4>
__device__ __forceinline__ void load_x(SmemA<H, NP>& sm, const WideMaps& mp, int s, int j, int nt) {
    using G = Geo<H, NP>;
    umma::tma_load5_hint(sm.ring + s * G::kStageA, G4 ? &mp.dz2k : &mp.h1k, 0, 2 * j, 0, 0, nt, &sm.full[s],
                         umma::l2_evict_last());
}

// The i-th K-chunk a streamed GEMM consumes: the epilogue writes the
// activation in rounds, round p holding piece p (16 columns) of every column
// group (H / 4 columns each), so chunk order follows the rounds and a GEMM
// starts on the first round while the epilogue writes the next.
template <int H>
__device__ __forceinline__ int chunk_of(int i) { return (i % 4) * (H / 64) + i / 4; }

// Thread 0 of kernel A: the activation part of the i-th chunk once its
// round of pieces is written.
template <int H, int NP, bool G4>
__device__ __forceinline__ bool load_x_when_written(SmemA<H, NP>& sm, const WideMaps& mp, int s, int i, int nt,
                                                    bool ok) {
    ok = wait_bar(&sm.piece[G4 ? 1 : 0][i / 4], 0u, ok);
    load_x<H, NP, G4>(sm, mp, s, chunk_of<H>(i), nt);
    return ok;
}

// Thread 0 of kernel A: one streamed GEMM (G2 or G4) over the chunks
// n0 .. n0 + kChunks - 1 of the stage ring (chunk n uses stage n % S for the
// (n / S)-th time), K-chunks in chunk_of order.  Chunks n0 .. n0 + S - 1
// were loaded before; every later chunk goes into the stage of the chunk
// before it as soon as that chunk's MMAs are done, so one issued chunk
// always waits in the queue.
template <int H, int NP, bool G4>
__device__ __forceinline__ bool run_gemm(SmemA<H, NP>& sm, const WideMaps& mp, int n0, uint32_t d_tmem, int net,
                                         int nt, bool ok) {
    using G = Geo<H, NP>;
    constexpr int S = kStagesA;
    constexpr int nt_ = NP == 3 ? 6 : 1;
    const uint32_t idesc = umma::instr_desc(umma::kTypeBF16, false, G4, TM, H);
    for (int j = 0; j < G::kChunks; ++j) {
        const int n = n0 + j, s = n % S;
        ok = wait_bar(&sm.full[s], (uint32_t)(n / S) & 1u, ok);
        umma::fence_after_sync();
        const uint8_t* st = sm.ring + s * G::kStageA;
#pragma unroll
        for (int t = 0; t < nt_; ++t) {
            const int ta = NP == 3 ? term_a(t) : 0, tb = NP == 3 ? term_b(t) : 0;
            // activation K-chunk: [plane][16 row groups][2 chunks]: LBO 128, SBO 256
            const uint64_t ad = desc(st + (uint32_t)ta * G::kPlaneA, 128u, 256u);
            // W2 K-chunk: [plane][H/8 row groups][2 chunks]; MN-chunk: [plane][2 row groups][H/8 chunks]
            const uint64_t bd = G4 ? desc(st + G::kBytesA + (uint32_t)tb * G::kPlaneB, (uint32_t)(16 * H), 128u)
                                   : desc(st + G::kBytesA + (uint32_t)tb * G::kPlaneB, 128u, 256u);
            umma::mma_f16(d_tmem, ad, bd, idesc, (j > 0 || t > 0) ? 1u : 0u);
        }
        umma::commit(&sm.empty[s]);
        if (j >= 1 && j - 1 + S < G::kChunks) {
            const int p = n - 1, sp = p % S;
            ok = wait_bar(&sm.empty[sp], (uint32_t)(p / S) & 1u, ok);
            load_w<H, NP, G4>(sm, mp, sp, chunk_of<H>(j - 1 + S), net);
            ok = load_x_when_written<H, NP, G4>(sm, mp, sp, j - 1 + S, nt, ok);
        }
    }
    return ok;
}

template <int H, int NP>
__global__ void __launch_bounds__(kThreads, 1)
    vnet_wide_fwd_kernel(const VnetLaunch a, const uint8_t* __restrict__ wimg, const __grid_constant__ WideMaps mp) {
    using G = Geo<H, NP>;
    static_assert(Checks<H, NP>::ok, "");
    constexpr int S = kStagesA, K = G::kChunks, kCols = G::kCols;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SmemA<H, NP>& sm = *reinterpret_cast<SmemA<H, NP>*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp != 0;
    const int ew = warp - 1, et = tid - 32;
    const int q = warp & 3, cg = (warp - 1) >> 2;
    const int row = 32 * q + lane;
    const int tile = blockIdx.x, net = blockIdx.y;
    const int S_ = a.state_dim, B = a.batch, NA = a.num_actions;
    const int row0 = tile * TM;
    const int nt = net * a.act_tiles + tile;
    const Offsets off = offsets_of(S_, H);
    const float* __restrict__ prm = a.params[net];
    const float tau = a.tau[net];
    const uint8_t* w1i = wimg + (int64_t)net * tc::weight_image_bytes(H);
    const uint8_t* xi = a.ximg + (int64_t)tile * NP * G::kPlaneX;
    uint8_t* h1g = a.act[0] + (int64_t)nt * NP * G::kActPlane;
    uint8_t* dz2g = a.act[1] + (int64_t)nt * NP * G::kActPlane;
    uint8_t* dz1g = a.act[2] + (int64_t)nt * NP * G::kActPlane;
    // the images stay in L2 for this kernel's streamed GEMMs and kernel B
    const uint64_t keep = umma::l2_evict_last();
    uint8_t* ring = sm.ring;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            umma::mbar_init(&sm.full[s], 1);
            umma::mbar_init(&sm.empty[s], 1);
        }
        umma::mbar_init(&sm.bar_mma, 1);
        umma::mbar_init(&sm.bar_load, 1);
        for (int r = 0; r < 4; ++r) {
            umma::mbar_init(&sm.piece[0][r], kEpiWarps);
            umma::mbar_init(&sm.piece[1][r], kEpiWarps);
        }
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(&sm.tmem_slot, kTmemCols);
    pdl_trigger();
    pdl_wait();
    // ---- stage 1: X image and W1 image across the ring ----
    if (tid == 0) {
        umma::mbar_expect_tx(&sm.bar_load, G::kXBytes + G::kW1Bytes);
        umma::bulk_g2s(ring, xi, G::kXBytes, &sm.bar_load);
        umma::bulk_g2s(ring + G::kXBytes, w1i, G::kW1Bytes, &sm.bar_load);
    }
    for (int i = tid; i < H; i += kThreads) {
        sm.b1[i] = __ldg(prm + off.b1 + i);
        sm.b2[i] = __ldg(prm + off.b2 + i);
        sm.w3[i] = __ldg(prm + off.w3 + i);
    }
    const float b3 = __ldg(prm + off.b3);
    {
        const int nrow = B - row0 < TM ? B - row0 : TM;
        if (a.q != nullptr) {
            for (int e = tid; e < nrow * NA; e += kThreads) sm.qt[e] = __ldg(a.q + (int64_t)row0 * NA + e);
            for (int e = tid; e < nrow; e += kThreads) sm.act[e] = __ldg(a.actions + row0 + e);
        } else {
            for (int e = tid; e < nrow; e += kThreads) sm.qt[e] = __ldg(a.q_taken + row0 + e);
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    uint32_t ph_mma = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        ok = wait_bar(&sm.bar_mma, ph_mma, ok);
        ph_mma ^= 1u;
        umma::fence_after_sync();
    };

    // ---- G1: z1 = X . W1^T; then the first W2 K-chunks of G2 ----
    if (tid == 0) {
        ok = wait_bar(&sm.bar_load, 0u, ok);
        umma::fence_after_sync();
        const uint32_t idesc = umma::instr_desc(umma::kTypeBF16, false, false, TM, H);
        constexpr int nt_ = NP == 3 ? 6 : 1;
        for (int ks = 0; ks < KX / 16; ++ks) {
#pragma unroll
            for (int t = 0; t < nt_; ++t) {
                const int ta = NP == 3 ? term_a(t) : 0, tb = NP == 3 ? term_b(t) : 0;
                const uint64_t ad = desc(ring + (uint32_t)ta * G::kPlaneX + (uint32_t)ks * 256u, 128u, (KX / 8) * 128u);
                const uint64_t bd =
                    desc(ring + G::kXBytes + (uint32_t)tb * G::kPlaneW1 + (uint32_t)ks * 256u, 128u, (KX / 8) * 128u);
                umma::mma_f16(tmem + TM_Z1, ad, bd, idesc, (ks > 0 || t > 0) ? 1u : 0u);
            }
        }
        umma::commit(&sm.bar_mma);
    }
    wait_mma();
    // ---- G2: z2 = h1 . W2^T, streamed; each K-chunk as soon as its round of
    // h1 pieces is written; then the first W2 MN-chunks of G4 ----
    if (tid == 0) {
        for (int j = 0; j < S; ++j) load_w<H, NP, false>(sm, mp, j, chunk_of<H>(j), net);
        for (int j = 0; j < S; ++j) ok = load_x_when_written<H, NP, false>(sm, mp, j, j, nt, ok);
        ok = run_gemm<H, NP, false>(sm, mp, 0, tmem + TM_Z2, net, nt, ok);
        umma::commit(&sm.bar_mma);
        for (int j = 0; j < S; ++j) {
            const int n = K + j, s = n % S;
            ok = wait_bar(&sm.empty[s], (uint32_t)((n - S) / S) & 1u, ok);
            load_w<H, NP, true>(sm, mp, s, chunk_of<H>(j), net);
        }
        // ---- G4: dh1 = dz2 . W2, streamed the same way behind the dz2 pieces ----
        for (int j = 0; j < S; ++j) ok = load_x_when_written<H, NP, true>(sm, mp, (K + j) % S, j, nt, ok);
        ok = run_gemm<H, NP, true>(sm, mp, K, tmem + TM_Z1, net, nt, ok);
        umma::commit(&sm.bar_mma);
    }

    // ---- epilogue 1: h1 = relu(z1 + b1) -> global image; ReLU mask kept ----
    uint64_t mask1 = 0;
    if (epi) {
#pragma unroll
        for (int p = 0; p < G::kPieces; ++p) {
            const int c0 = cg * kCols + 16 * p;
            float v[16];
            umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float z = v[j] + sm.b1[c0 + j];
                v[j] = z < 0.0f ? 0.0f : z;
                if (v[j] > 0.0f) mask1 |= 1ull << (16 * p + j);
            }
            store16_global<NP>(h1g, G::kActPlane, H, row, c0, v, keep);
            // round p written by this warp: visible to the tensor copies,
            // this warp's TMEM reads of z1 ordered before G4 overwrites it
            umma::fence_global_to_async();
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(&sm.piece[0][p]);
        }
    }

    // ---- epilogue 2: V, loss, dV, dz2 -> global image, tile column sums ----
    float dv = 0.0f, lossp = 0.0f;
    if (epi) {
        wait_mma();
        float vp = 0.0f;
#pragma unroll
        for (int p = 0; p < G::kPieces; ++p) {
            const int c0 = cg * kCols + 16 * p;
            float v[16];
            umma::tmem_ld16(tq + TM_Z2 + (uint32_t)c0, v);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float z = v[j] + sm.b2[c0 + j];
                vp = fmaf(z < 0.0f ? 0.0f : z, sm.w3[c0 + j], vp);
            }
        }
        sm.vsum[cg][row] = vp;
        epi_sync();
        const float V = ((sm.vsum[0][row] + sm.vsum[1][row]) + (sm.vsum[2][row] + sm.vsum[3][row])) + b3;
        const int b = row0 + row;
        if (b < B) {
            float qv;
            if (a.q != nullptr) {
                int act = sm.act[row];
                if (act < 0 || act >= NA) {
                    if (cg == 0) atomicAdd(a.status + OFRL_STAT_BAD_ACTION, 1);
                    act = 0;
                }
                qv = sm.qt[row * NA + act];
            } else {
                qv = sm.qt[row];
            }
            const float d = qv - V;
            const float w = d >= 0.0f ? tau : 1.0f - tau;
            lossp = w * d * d;
            dv = (-2.0f * w * d) / (float)B;
            if (cg == 0 && a.v_out != nullptr) a.v_out[(int64_t)net * B + b] = V;
        }
        if (cg == 0) sm.vrow[row] = V;
#pragma unroll
        for (int p = 0; p < G::kPieces; ++p) {
            const int c0 = cg * kCols + 16 * p;
            float g[16], hw[16];
            umma::tmem_ld16(tq + TM_Z2 + (uint32_t)c0, g);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float z = g[j] + sm.b2[c0 + j];
                g[j] = z > 0.0f ? dv * sm.w3[c0 + j] : 0.0f;
                hw[j] = dv * (z < 0.0f ? 0.0f : z);
            }
            store16_global<NP>(dz2g, G::kActPlane, H, row, c0, g, keep);
            umma::fence_global_to_async();
            __syncwarp();
            if (lane == 0) umma::mbar_arrive(&sm.piece[1][p]);   // round p of dz2 written by this warp
            const float s3 = colsum16(hw);
            const float s2 = colsum16(g);
            if ((lane & 1) == 0) {
                sm.red[0][ew][16 * p + ((lane >> 1) & 15)] = s3;
                sm.red[1][ew][16 * p + ((lane >> 1) & 15)] = s2;
            }
        }
        if (cg == 0) {
            const float ls = warp_sum(lossp), ds = warp_sum(dv);
            if (lane == 0) { sm.lred[0][q] = ls; sm.lred[1][q] = ds; }
        }
        epi_sync();
    }
    if (epi) {
        // the tile's vectors (fixed order over the four lane-quarter warps)
        float* tv = a.tvec + (int64_t)nt * a.tvec_stride;
        for (int c = et; c < H; c += kThreads - 32) {
            const int g = c / kCols, cl = c % kCols;
            float s3 = 0.0f, s2 = 0.0f;
            for (int qq = 0; qq < 4; ++qq) { s3 += sm.red[0][g * 4 + qq][cl]; s2 += sm.red[1][g * 4 + qq][cl]; }
            tv[c] = s3;
            tv[H + c] = s2;
        }
        if (et == 0) {
            const float l = (sm.lred[0][0] + sm.lred[0][1]) + (sm.lred[0][2] + sm.lred[0][3]);
            const float d3 = (sm.lred[1][0] + sm.lred[1][1]) + (sm.lred[1][2] + sm.lred[1][3]);
            a.tile_loss[(int64_t)net * a.net_tile_stride + tile] = l;
            tv[2 * H] = d3;
        }
        // the policy while G4 runs: four threads per row (lanes 4r .. 4r + 3),
        // each over actions j, j + 4, ...; max / argmax (lowest index on
        // ties) and the sum of exponentials combined over the four lanes
        if (a.pi_out != nullptr) {
            const int pr = et >> 2, j = et & 3;
            const int pb = row0 + pr;
            const bool prow = pb < B;
            const float Vp = sm.vrow[pr];
            const float* qr = sm.qt + pr * NA;
            float zmax = -INFINITY, amax = -INFINITY;
            int best = NA;
            if (prow)
                for (int k = j; k < NA; k += 4) {
                    const float adv = fminf(fmaxf(qr[k] - Vp, -10.0f), 10.0f);
                    if (adv > amax) { amax = adv; best = k; }
                    zmax = fmaxf(zmax, a.beta * adv);
                }
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                const float oa = __shfl_xor_sync(0xffffffffu, amax, o);
                const int ob = __shfl_xor_sync(0xffffffffu, best, o);
                if (oa > amax || (oa == amax && ob < best)) { amax = oa; best = ob; }
                zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
            }
            float sum = 0.0f;
            if (prow)
                for (int k = j; k < NA; k += 4) sum += expf(a.beta * fminf(fmaxf(qr[k] - Vp, -10.0f), 10.0f) - zmax);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (prow) {
                float* po = a.pi_out + ((int64_t)net * B + pb) * NA;
                for (int k = j; k < NA; k += 4)
                    po[k] = expf(a.beta * fminf(fmaxf(qr[k] - Vp, -10.0f), 10.0f) - zmax) / sum;
                if (j == 0 && a.argmax_out != nullptr) a.argmax_out[(int64_t)net * B + pb] = best < NA ? best : 0;
            }
        }
        // ---- epilogue 4: dz1 = dh1 * 1[z1 > 0] -> global image ----
        wait_mma();
#pragma unroll
        for (int p = 0; p < G::kPieces; ++p) {
            const int c0 = cg * kCols + 16 * p;
            float v[16];
            umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = ((mask1 >> (16 * p + j)) & 1ull) ? v[j] : 0.0f;
            store16_global<NP, true>(dz1g, G::kActPlane, H, row, c0, v, keep);
        }
        umma::fence_global_to_async();
    }
    if (!ok && (tid == 0 || tid == 32)) atomicAdd(a.status + OFRL_STAT_TIMEOUT, 1);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

// Kernel B's loads of K-step g (tile g / 8, rows 16 (g % 8) ..) into stage s.
template <int H, int NP>
__device__ __forceinline__ void load_step(SmemB<H, NP>& sm, const WideMaps& mp, int s, int g, int h, int nt0) {
    using G = Geo<H, NP>;
    const int tile = g / kWaysPerTile, rg = 2 * (g % kWaysPerTile), nt = nt0 + tile;
    uint8_t* st = sm.ring + s * G::kStageB;
    umma::mbar_expect_tx(&sm.full[s], G::kStageB);
    const uint64_t last = umma::l2_evict_first();
    umma::tma_load5_hint(st, &mp.dz2h, 0, 16 * h, rg, 0, nt, &sm.full[s], last);
    umma::tma_load5(st + G::kOffB2, &mp.h1n, 0, 0, rg, 0, nt, &sm.full[s]);
    umma::tma_load5_hint(st + G::kOffA1, &mp.dz1h, 0, 16 * h, rg, 0, nt, &sm.full[s], last);
    umma::tma_load5(st + G::kOffB1, &mp.xk, 0, 0, rg, 0, tile, &sm.full[s]);
}

template <int H, int NP>
__global__ void __launch_bounds__(kThreads, 1)
    vnet_wide_wgrad_kernel(const VnetLaunch a, const __grid_constant__ WideMaps mp) {
    using G = Geo<H, NP>;
    static_assert(Checks<H, NP>::ok, "");
    constexpr int S = kStagesB, kCols = G::kCols;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SmemB<H, NP>& sm = *reinterpret_cast<SmemB<H, NP>*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp != 0;
    const int et = tid - 32;
    const int q = warp & 3, cg = (warp - 1) >> 2;
    const int row = 32 * q + lane;          // accumulator lane: hidden unit 128 h + row
    const int kr = blockIdx.x, h = blockIdx.y, net = blockIdx.z;
    const int S_ = a.state_dim, B = a.batch;
    const int n_tiles = (B + TM - 1) / TM;
    const int KS = kWaysPerTile * n_tiles;
    const int ks0 = (int)((int64_t)kr * KS / a.n_ranges), ks1 = (int)((int64_t)(kr + 1) * KS / a.n_ranges);
    const int nk = ks1 - ks0;
    const int nt0 = net * a.act_tiles;
    const Offsets off = offsets_of(S_, H);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            umma::mbar_init(&sm.full[s], 1);
            umma::mbar_init(&sm.empty[s], 1);
        }
        umma::mbar_init(&sm.bar_mma, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(&sm.tmem_slot, kTmemCols);
    pdl_trigger();
    pdl_wait();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;

    if (tid == 0) {
        // weight gradients (K = batch rows): the three leading products of
        // the split (terms 3..5; the fused kernel's G3 / G5 note has why)
        constexpr int t0_ = NP == 3 ? 3 : 0;
        constexpr int nt_ = NP == 3 ? 6 : 1;
        const uint32_t id2 = umma::instr_desc(umma::kTypeBF16, true, true, TM, H);
        const uint32_t id1 = umma::instr_desc(umma::kTypeBF16, true, true, TM, KX);
        for (int i = 0; i < S && i < nk; ++i) load_step<H, NP>(sm, mp, i, ks0 + i, h, nt0);
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            ok = wait_bar(&sm.full[s], (uint32_t)(i / S) & 1u, ok);
            umma::fence_after_sync();
            const uint8_t* st = sm.ring + s * G::kStageB;
#pragma unroll
            for (int t = t0_; t < nt_; ++t) {
                const int ta = NP == 3 ? term_a(t) : 0, tb = NP == 3 ? term_b(t) : 0;
                const uint32_t acc = (i > 0 || t > t0_) ? 1u : 0u;
                // MN-major chunks: [plane][2 row groups][chunks]: LBO = one row group, SBO = 128
                const uint64_t a2 = desc(st + (uint32_t)ta * G::kPlaneHalf, 16u * 128u, 128u);
                const uint64_t b2 = desc(st + G::kOffB2 + (uint32_t)tb * G::kPlaneN, (uint32_t)(H / 8) * 128u, 128u);
                umma::mma_f16(tmem + TM_D2, a2, b2, id2, acc);
                const uint64_t a1 = desc(st + G::kOffA1 + (uint32_t)ta * G::kPlaneHalf, 16u * 128u, 128u);
                const uint64_t b1 = desc(st + G::kOffB1 + (uint32_t)tb * G::kPlaneXK, (uint32_t)(KX / 8) * 128u, 128u);
                umma::mma_f16(tmem + TM_D1, a1, b1, id1, acc);
            }
            umma::commit(&sm.empty[s]);
            if (i >= 1 && i - 1 + S < nk) {
                const int sp = (i - 1) % S;
                ok = wait_bar(&sm.empty[sp], (uint32_t)((i - 1) / S) & 1u, ok);
                load_step<H, NP>(sm, mp, sp, ks0 + i - 1 + S, h, nt0);
            }
        }
        umma::commit(&sm.bar_mma);
    }
    if (epi) {
        // the tile vectors of the range (tiles whose first K-step lies in it)
        const int t0 = (ks0 + kWaysPerTile - 1) / kWaysPerTile, t1 = (ks1 + kWaysPerTile - 1) / kWaysPerTile;
        for (int e = et; e < 2 * 128; e += kThreads - 32) {
            const int k = e >> 7, i = 128 * h + (e & 127);
            float s = 0.0f;
            for (int t = t0; t < t1; ++t) s += a.tvec[(int64_t)(nt0 + t) * a.tvec_stride + k * H + i];
            sm.vec[k][e & 127] = s;
        }
        if (et == 2 * 128 && h == 0) {
            float s = 0.0f;
            for (int t = t0; t < t1; ++t) s += a.tvec[(int64_t)(nt0 + t) * a.tvec_stride + 2 * H];
            sm.b3 = s;
        }
        ok = wait_bar(&sm.bar_mma, 0u, ok);
        umma::fence_after_sync();
        // stage dW2 rows (padded stride, float4 stores) and the dW1 rows of the half
        float* st2 = reinterpret_cast<float*>(sm.ring);
        float* st1 = st2 + 128 * G::kStride2;
#pragma unroll
        for (int p = 0; p < G::kPieces; ++p) {
            const int c0 = cg * kCols + 16 * p;
            float v[16];
            umma::tmem_ld16(tq + TM_D2 + (uint32_t)c0, v);
            umma::tmem_ld_wait();
            float4* dst = reinterpret_cast<float4*>(st2 + row * G::kStride2 + c0);
#pragma unroll
            for (int f = 0; f < 4; ++f) dst[f] = make_float4(v[4 * f], v[4 * f + 1], v[4 * f + 2], v[4 * f + 3]);
        }
        {
            const int c0 = cg * 16;
            float v[16];
            umma::tmem_ld16(tq + TM_D1 + (uint32_t)c0, v);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < S_) st1[row * S_ + c0 + j] = v[j];
            if (c0 + 15 == KX - 1) sm.vec[2][row] = v[15];   // the ones column: db1
        }
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();
    // partial row kr: the half's rows of dW2 and dW1 and entries of db1, db2,
    // dW3 (and db3 from half 0), all 16-byte aligned bulk copies
    float* dst = a.partials + (int64_t)net * a.net_partial_stride + (int64_t)kr * a.part_stride;
    if (tid < 128 + 5) {
        const float* st2 = reinterpret_cast<const float*>(sm.ring);
        const float* st1 = st2 + 128 * G::kStride2;
        const uint64_t keep = umma::l2_evict_last();
        if (tid < 128)
            umma::bulk_s2g_hint(dst + off.w2 + (int64_t)(128 * h + tid) * H, st2 + tid * G::kStride2, H * 4, keep);
        if (tid == 128) umma::bulk_s2g_hint(dst + off.w1 + (int64_t)128 * h * S_, st1, (uint32_t)(128 * S_ * 4), keep);
        if (tid == 129) umma::bulk_s2g(dst + off.w3 + 128 * h, sm.vec[0], 512);
        if (tid == 130) umma::bulk_s2g(dst + off.b2 + 128 * h, sm.vec[1], 512);
        if (tid == 131) umma::bulk_s2g(dst + off.b1 + 128 * h, sm.vec[2], 512);
        if (tid == 132 && h == 0) dst[off.b3] = sm.b3;
        umma::bulk_commit();
        umma::bulk_wait_read();
    }
    if (!ok && (tid == 0 || tid == 32)) atomicAdd(a.status + OFRL_STAT_TIMEOUT, 1);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

// Standalone calls: W1 ([H][S] -> [H x 64]) and W2 ([H][H] -> [H x H])
// images of every network and the state-tile images of the batch (the ones
// column when S < 64; rows past the batch zero), np planes.
__global__ void wide_pack_kernel(const VnetLaunch a, uint8_t* __restrict__ wimg, uint8_t* __restrict__ ximg, int np) {
    const int S = a.state_dim, H = a.hidden;
    const Offsets off = offsets_of(S, H);
    const int n1 = H * (KX / 4), n2 = H * (H / 4), nw = a.n_nets * (n1 + n2);
    const int rows = (a.batch + TM - 1) / TM * TM;
    const int64_t total = (int64_t)nw + (int64_t)rows * (KX / 4);
    const uint32_t plane1 = (uint32_t)(H * KX * 2), plane2 = (uint32_t)(H * H * 2);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        float x[4];
        if (e < nw) {
            const int net = (int)(e / (n1 + n2)), f = (int)(e % (n1 + n2));
            const float* __restrict__ prm = a.params[net];
            uint8_t* w1i = wimg + (int64_t)net * tc::weight_image_bytes(H);
            if (f < n1) {
                const int r = f / (KX / 4), c = 4 * (f % (KX / 4));
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = c + j < S ? __ldg(prm + off.w1 + (int64_t)r * S + c + j) : 0.0f;
                tc::put4(w1i, plane1, np, KX, r, c, x);
            } else {
                const int g = f - n1, r = g / (H / 4), c = 4 * (g % (H / 4));
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = __ldg(prm + off.w2 + (int64_t)r * H + c + j);
                tc::put4(w1i + tc::w2_image_offset(H), plane2, np, H, r, c, x);
            }
        } else {
            const int64_t f = e - nw;
            const int r = (int)(f / (KX / 4)), c = 4 * (int)(f % (KX / 4));
            const bool live = r < a.batch;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int cc = c + j;
                x[j] = !live ? 0.0f
                             : cc < S ? __ldg(a.states + (int64_t)r * a.stride + cc)
                                      : (tc::ones_column(cc, S) ? 1.0f : 0.0f);
            }
            tc::put4(ximg + (int64_t)(r / TM) * np * tc::kPlaneX, tc::kPlaneX, np, KX, r % TM, c, x);
        }
    }
}

template <int H, int NP>
cudaError_t configure() {
    static cudaError_t state = cudaErrorNotReady;
    if (state == cudaErrorNotReady) {
        auto ka = vnet_wide_fwd_kernel<H, NP>;
        auto kb = vnet_wide_wgrad_kernel<H, NP>;
        state = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SmemA<H, NP>));
        if (state == cudaSuccess)
            state = cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SmemB<H, NP>));
        if (state == cudaSuccess) state = set_max_shared_carveout(ka);
        if (state == cudaSuccess) state = set_max_shared_carveout(kb);
    }
    return state;
}

template <int H, int NP>
cudaError_t launch_hn(const VnetLaunch& a, const uint8_t* wimg, cudaStream_t st) {
    const cudaError_t e = configure<H, NP>();
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.batch + TM - 1) / TM;
    const WideMaps& m = *a.maps;
    cudaError_t r = launch_ex(vnet_wide_fwd_kernel<H, NP>, dim3((unsigned)n_tiles, (unsigned)a.n_nets),
                              dim3(kThreads), sizeof(SmemA<H, NP>), st, 1u, false, a, wimg, m);
    if (r != cudaSuccess) return r;
    return launch_ex(vnet_wide_wgrad_kernel<H, NP>,
                     dim3((unsigned)a.n_ranges, (unsigned)Geo<H, NP>::kHalves, (unsigned)a.n_nets), dim3(kThreads),
                     sizeof(SmemB<H, NP>), st, 1u, false, a, m);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static EncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
        cudaGetLastError();
    }
    return fn;
}

// A 5-D bf16 tensor map: dims innermost first, strides (bytes) of dims 1..4.
cudaError_t encode5(CUtensorMap* m, const void* base, const cuuint64_t (&dim)[5], const cuuint64_t (&stride)[4],
                    const cuuint32_t (&box)[5]) {
    const EncodeFn fn = encoder();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dim, stride, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool vnet_wide_supported(const VnetLaunch& a) {
    return (a.hidden == 128 || a.hidden == 256) && a.state_dim < KX && a.maps != nullptr && a.act[0] != nullptr;
}

int64_t vnet_wide_act_bytes(int hidden, int planes) { return (int64_t)planes * TM * hidden * 2; }

int32_t vnet_wide_tvec_stride(int hidden) { return 2 * hidden + 32; }

int vnet_wide_ranges(const VnetLaunch& a, int num_sms) {
    const int n_tiles = (a.batch + TM - 1) / TM;
    const int ks = kWaysPerTile * n_tiles;
    const int halves = a.hidden / 128;
    int r = num_sms / (halves * (a.n_nets > 0 ? a.n_nets : 1));
    if (r < 1) r = 1;
    return r < ks ? r : ks;
}

cudaError_t vnet_wide_maps(WideMaps* m, int hidden, int planes, int n_nets, int act_tiles, uint8_t* const act[3],
                           uint8_t* ximg, int x_tiles, uint8_t* wimg) {
    const cuuint64_t H = (cuuint64_t)hidden, NP = (cuuint64_t)planes;
    const cuuint64_t plane = (cuuint64_t)TM * H * 2;
    // activation images: (core matrix, chunk, row group, plane, tile)
    const cuuint64_t adim[5] = {64, H / 8, TM / 8, NP, (cuuint64_t)n_nets * act_tiles};
    const cuuint64_t astr[4] = {128, 16 * H, plane, NP * plane};
    const cuuint32_t kbox[5] = {64, 2, TM / 8, (cuuint32_t)NP, 1};
    // kernel B's boxes take the planes its three leading products read
    const cuuint32_t npb = NP == 3 ? 2 : (cuuint32_t)NP;
    const cuuint32_t hbox[5] = {64, 16, 2, npb, 1};
    const cuuint32_t nbox[5] = {64, (cuuint32_t)(H / 8), 2, npb, 1};
    cudaError_t e = encode5(&m->h1k, act[0], adim, astr, kbox);
    if (e == cudaSuccess) e = encode5(&m->dz2k, act[1], adim, astr, kbox);
    if (e == cudaSuccess) e = encode5(&m->dz2h, act[1], adim, astr, hbox);
    if (e == cudaSuccess) e = encode5(&m->dz1h, act[2], adim, astr, hbox);
    if (e == cudaSuccess) e = encode5(&m->h1n, act[0], adim, astr, nbox);
    // state-tile images: [tile][plane][128 x 64]
    const cuuint64_t xdim[5] = {64, KX / 8, TM / 8, NP, (cuuint64_t)x_tiles};
    const cuuint64_t xstr[4] = {128, (KX / 8) * 128, tc::kPlaneX, NP * tc::kPlaneX};
    const cuuint32_t xbox[5] = {64, KX / 8, 2, npb, 1};
    if (e == cudaSuccess) e = encode5(&m->xk, ximg, xdim, xstr, xbox);
    // W2 images: (core matrix, chunk, row group, plane, network)
    const cuuint64_t wdim[5] = {64, H / 8, H / 8, NP, (cuuint64_t)n_nets};
    const cuuint64_t wstr[4] = {128, 16 * H, H * H * 2, (cuuint64_t)tc::weight_image_bytes(hidden)};
    const cuuint32_t wkbox[5] = {64, 2, (cuuint32_t)(H / 8), (cuuint32_t)NP, 1};
    const cuuint32_t wnbox[5] = {64, (cuuint32_t)(H / 8), 2, (cuuint32_t)NP, 1};
    uint8_t* w2 = wimg + tc::w2_image_offset(hidden);
    if (e == cudaSuccess) e = encode5(&m->w2k, w2, wdim, wstr, wkbox);
    if (e == cudaSuccess) e = encode5(&m->w2n, w2, wdim, wstr, wnbox);
    return e;
}

cudaError_t launch_vnet_wide_pack(const VnetLaunch& a, uint8_t* wimg, uint8_t* ximg, cudaStream_t st) {
    wide_pack_kernel<<<dim3(128), 256, 0, st>>>(a, wimg, ximg, a.prec == OFRL_PREC_BF16 ? 1 : 3);
    return cudaGetLastError();
}

cudaError_t launch_vnet_wide(const VnetLaunch& a, const uint8_t* wimg, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    if (!vnet_wide_supported(a) || a.n_ranges < 1) return cudaErrorInvalidValue;
    const bool bf = a.prec == OFRL_PREC_BF16;
    if (a.hidden == 256) return bf ? launch_hn<256, 1>(a, wimg, st) : launch_hn<256, 3>(a, wimg, st);
    return bf ? launch_hn<128, 1>(a, wimg, st) : launch_hn<128, 3>(a, wimg, st);
}

}  // namespace ofrl
