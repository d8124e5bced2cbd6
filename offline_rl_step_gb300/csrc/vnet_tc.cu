// IQL value network V(s) forward, expectile loss, policy and backward for one
// 128-row batch tile per CTA on the 5th-generation tensor cores (tcgen05),
// hidden width 128 (64 runs in the same images zero-padded to 128 units, the
// GEMMs over the units cut to 64 and the padded columns' epilogue work
// skipped; only the H x H, H x S and H entries are written out).
//
// Method: "GPU IQL + HER Porting Plan", "IQL (CPU)" items 1-3 and "CUDA
// Kernel: iql_value_kernel.cu"; same results as the CUDA-core kernel
// (vnet_simt.cu) to fp32 rounding.
//
// Five GEMMs per tile, accumulated in tensor memory (TMEM, fp32):
//   G1  z1  [rows x H]  = X  . W1^T      (A: X   K-major,  B: W1 K-major)
//   G2  z2  [rows x H]  = h1 . W2^T      (A: h1  K-major,  B: W2 K-major)
//   G3  dW2 [H x H]     = dz2^T . h1     (A: dz2 MN-major, B: h1 MN-major)
//   G4  dh1 [rows x H]  = dz2 . W2       (A: dz2 K-major,  B: W2 MN-major)
//   G5  dW1 [H x 64]    = dz1^T . X      (A: dz1 MN-major, B: X  MN-major)
// Operands are bf16 images in shared memory (tc_image.cuh): core matrices of
// 8 rows x 8 elements, so an activation tile written once is the K-major
// operand of one GEMM and the MN-major operand of another.
//
// Precision: for fp32 results every operand is split into three bf16 terms
// x = x0 + x1 + x2 (24 significand bits).  The forward GEMMs (G1, G2) issue
// per K-step the six products down to 2^-16 of the leading one (x2 y0,
// x1 y1, x0 y2, x1 y0, x0 y1, x0 y0); the rest lie below fp32 rounding.  The
// backward GEMMs issue the three leading ones (x1 y0, x0 y1, x0 y0): with
// |x2| <= 2^-18 |x| each product is then off by at most 3.1 * 2^-18 of
// itself, at random.  In the weight-gradient GEMMs (G3, G5), whose K runs
// over the batch rows, that adds about sqrt(n) 3.1 2^-18 rms(terms) to a sum
// of n rows, against an fp32 summation error of order sqrt(n) 2^-24 times
// the sum of |terms|, about n / 200 times larger (comparable within one
// 128-row tile, 80 times larger over a 16,384-row batch).  G4's dh1 feeds
// only those sums (its ReLU mask comes from the forward z1, which keeps full
// precision, so no mask decision moves).  The bf16 workload has one term and
// one product.
//
// Shared memory: two 96 KB regions of three 32 KB plane slots, reused
// through the step:
//   R0: X image -> h1 (planes 0-2; G2, then planes 0-1 for G3)
//       + dz2 plane 0 in slot 2 -> X planes 0-1 (for G5, 32 KB) in slot 0
//   R1: W1 image -> W2 (planes 0-2; G2, then planes 0-1 for G4)
//       + dz2 plane 1 in slot 2 -> dz1 (planes 0-1, for G5)
// so W2 is loaded once per tile and G3, G4 run back to back.
// Images arrive by bulk asynchronous copies (cp.async.bulk) on an mbarrier:
// the weights from the per-step pack, the state tiles from the relabel
// kernel (or, without those, are built here from the fp32 batch).
// 17 warps: warp 0 issues the MMAs and bulk copies; epilogue warp w = 1..16
// reads TMEM lane quarter w % 4 (tile rows, or hidden units for the weight
// gradients) and column group (w - 1) / 4 (32 columns).

#include <cstddef>

#include "common.cuh"
#include "tc_image.cuh"
#include "umma.cuh"

namespace ofrl {
namespace {

using tc::HH;
using tc::KX;
using tc::kPlaneH;
using tc::kPlaneX;
using tc::TM;

// Warp 0 issues the MMAs and the bulk copies and owns TMEM; warps 1..16 run
// the epilogues (warp w reads TMEM lane quarter w % 4; column group
// (w - 1) / 4), so the MMA issue never waits behind epilogue work.
constexpr int kThreads = 544;
constexpr int kEpiWarps = 16;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_Z1 = 0, TM_Z2 = 128, TM_DW2 = 256, TM_DW1 = 384;   // TM_Z1 also holds dh1
constexpr uint32_t kRegion = 3 * kPlaneH;    // 96 KB
constexpr uint64_t kWaitNs = 1000000000ull;  // bounded waits: 1 s

// Descriptor of K-step ks (16 elements of K) of an image with C columns:
// K-major (rows = M/N, columns = K): LBO = 128 (next chunk along K),
//   SBO = next 8-row group;
// MN-major (rows = K, columns = M/N): LBO = next 8-row group (along K),
//   SBO = 128 (next chunk along M/N).
__device__ __forceinline__ uint64_t desc_k(const uint8_t* plane, int C, int ks) {
    return umma::smem_desc(umma::smem_u32(plane) + (uint32_t)ks * 256u, 128u, (uint32_t)(C >> 3) * 128u);
}
__device__ __forceinline__ uint64_t desc_mn(const uint8_t* plane, int C, int ks) {
    const uint32_t group = (uint32_t)(C >> 3) * 128u;
    return umma::smem_desc(umma::smem_u32(plane) + (uint32_t)ks * 2u * group, group, 128u);
}

// Issue one GEMM (all K-steps, all split terms) from one thread.
// accumulate: add to what D holds (else the first product overwrites it).
// LEADING: only the three leading products of the split (the batch-row
// weight-gradient GEMMs; see the precision note above).
template <int NP, bool LEADING = false>
__device__ __forceinline__ void gemm(uint32_t d_tmem, const uint8_t* a, uint32_t a_plane, int a_cols, bool a_mn,
                                     const uint8_t* b, uint32_t b_plane, int b_cols, bool b_mn, int ksteps, int n,
                                     bool accumulate = false) {
    const uint32_t idesc = umma::instr_desc(umma::kTypeBF16, a_mn, b_mn, TM, n);
    constexpr int t0 = NP == 3 && LEADING ? 3 : 0;
    constexpr int nt = NP == 3 ? 6 : 1;
    constexpr int ta[6] = {2, 1, 0, 1, 0, 0};   // smallest products first
    constexpr int tb[6] = {0, 1, 2, 0, 1, 0};
    uint32_t acc = accumulate ? 1u : 0u;
    for (int ks = 0; ks < ksteps; ++ks) {
#pragma unroll
        for (int t = t0; t < nt; ++t) {
            const uint8_t* ap = a + (uint32_t)(NP == 3 ? ta[t] : 0) * a_plane;
            const uint8_t* bp = b + (uint32_t)(NP == 3 ? tb[t] : 0) * b_plane;
            const uint64_t ad = a_mn ? desc_mn(ap, a_cols, ks) : desc_k(ap, a_cols, ks);
            const uint64_t bd = b_mn ? desc_mn(bp, b_cols, ks) : desc_k(bp, b_cols, ks);
            umma::mma_f16(d_tmem, ad, bd, idesc, acc);
            acc = 1;
        }
    }
}

// Store 16 fp32 values of row r, columns c0..c0+15 into a [128 x 128] image
// whose planes lie `plane` bytes apart.
// LEADING: only the two planes the three leading products read (dz2, dz1:
// operands of the backward GEMMs alone); plane 2 is left as it was.
template <int NP, bool LEADING = false>
__device__ __forceinline__ void store16(uint8_t* img, int r, int c0, const float (&v)[16],
                                        uint32_t plane = kPlaneH) {
    constexpr int NW = NP == 3 && LEADING ? 2 : NP;   // planes written
    uint32_t t[NP][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if constexpr (NP == 3 && LEADING) tc::split2x2(v[2 * j], v[2 * j + 1], t[0][j], t[1][j]);
        else if constexpr (NP == 3) tc::split3x2(v[2 * j], v[2 * j + 1], t[0][j], t[1][j], t[2][j]);
        else t[0][j] = tc::pack_bf16x2(v[2 * j], v[2 * j + 1]);
    }
    const uint32_t o0 = tc::img_off(r, c0, HH), o1 = tc::img_off(r, c0 + 8, HH);
#pragma unroll
    for (int p = 0; p < NW; ++p) {
        *reinterpret_cast<uint4*>(img + (uint32_t)p * plane + o0) = make_uint4(t[p][0], t[p][1], t[p][2], t[p][3]);
        *reinterpret_cast<uint4*>(img + (uint32_t)p * plane + o1) = make_uint4(t[p][4], t[p][5], t[p][6], t[p][7]);
    }
}

// Build the X image ([128 x 64]) of a tile from the fp32 batch (used when the
// relabel kernel did not write images): rows past the batch, columns past S
// are zero.  PREFETCH: every thread's loads are issued before any of them is
// split and stored, so the tile costs one round of memory latency (the
// forward-only kernel; the training kernel keeps the loop, whose registers
// it cannot spare).
template <bool PREFETCH = false>
__device__ __forceinline__ void build_x(uint8_t* img, int np, const float* __restrict__ states, int stride, int row0,
                                        int B, int S) {
    constexpr int kChunks = TM * (KX / 4);                      // float4 chunks of the tile
    constexpr int kPer = PREFETCH ? (kChunks + kThreads - 1) / kThreads : 1;
    for (int e0 = threadIdx.x; e0 < kChunks; e0 += kPer * kThreads) {
        float4 v[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = e0 + i * kThreads;
            const int r = e / (KX / 4), c = 4 * (e % (KX / 4));
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < kChunks && row0 + r < B && c < S)
                v[i] = __ldg(reinterpret_cast<const float4*>(states + (int64_t)(row0 + r) * stride + c));
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = e0 + i * kThreads;
            if (e >= kChunks) break;
            const int r = e / (KX / 4), c = 4 * (e % (KX / 4));
            float x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (c + j >= S) x[j] = row0 + r < B && tc::ones_column(c + j, S) ? 1.0f : 0.0f;
            tc::put4(img, kPlaneX, np, KX, r, c, x);
        }
    }
}

struct TcSmem {
    uint8_t r0[kRegion];
    uint8_t r1[kRegion];
    __align__(16) float b1[HH];
    __align__(16) float b2[HH];
    float w3[HH];                     // right after b2: one copy brings both
    float vsum[4][TM];
    float red[3][kEpiWarps][32];   // per epilogue warp column sums: dW3, db2, db1
    float lred[2][4];           // per lane-quarter warp of column group 0: loss, db3
    __align__(16) float vec[3][HH];   // this CTA's dW3, db2, db1 over its tiles
    __align__(16) float qt[TM * kMaxActions];   // the tile's Q rows [row][action] (or q_taken [row])
    __align__(16) int32_t act[TM];              // the tile's actions
    float vrow[TM];                   // V of each row
    float vb3;                  // this CTA's db3 over its tiles
    uint64_t bar_mma, bar_load, bar_g3;   // bar_g3: dW2's GEMM done (the training kernel)
    uint32_t tmem_slot;
};
static_assert(sizeof(TcSmem) <= 227 * 1024, "tensor-core kernel shared memory above the per-CTA limit");
static_assert(offsetof(TcSmem, w3) == offsetof(TcSmem, b2) + HH * sizeof(float), "w3 follows b2");
static_assert(kMaxActions % 4 == 0, "the policy gives each of a row's four lanes kMaxActions / 4 actions");

// 16 consecutive floats of shared memory (16-byte aligned) by four 16-byte loads
__device__ __forceinline__ void lds16(const float* p, float (&o)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 t = reinterpret_cast<const float4*>(p)[i];
        o[4 * i] = t.x; o[4 * i + 1] = t.y; o[4 * i + 2] = t.z; o[4 * i + 3] = t.w;
    }
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) vnet_tc_kernel(const VnetLaunch a, const uint8_t* __restrict__ wimg) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp != 0;                 // an epilogue warp
    const int ew = warp - 1, et = tid - 32;     // epilogue warp / thread index
    const int q = warp & 3, cg = (warp - 1) >> 2;   // TMEM lane quarter, column group (32 columns)
    const int row = 32 * q + lane;              // tile row / accumulator lane of this thread
    const int net = blockIdx.y;
    const int S = a.state_dim, B = a.batch, NA = a.num_actions;
    const int n_tiles = (B + TM - 1) / TM;
    const int Hn = a.hidden;   // 64 or 128: the weights are zero-padded to 128 units
    // the units computed: at H = 64 the GEMMs take K and N = 64 where they
    // run over units, and the epilogue warps of columns 64-127 skip their
    // work (what lies there is never read, or lands only in the padded rows
    // of dW2 and dW1, which are not written out)
    const int HN = Hn <= 64 ? 64 : HH;
    const bool live = cg * 32 < HN;   // this epilogue warp's columns are units
    const Offsets off = offsets_of(S, Hn);
    const float* __restrict__ prm = a.params[net];
    const float tau = a.tau[net];
    const uint8_t* w1i = wimg + (int64_t)net * tc::weight_image_bytes();
    const uint8_t* w2i = w1i + tc::w2_image_offset();
    constexpr uint32_t kXBytes = (uint32_t)NP * kPlaneX, kW2Bytes = (uint32_t)NP * kPlaneH;
    constexpr uint32_t kX2Bytes = (uint32_t)(NP < 2 ? NP : 2) * kPlaneX;   // the planes G5 reads

    if (tid == 0) {
        umma::mbar_init(&sm.bar_mma, 1);
        umma::mbar_init(&sm.bar_load, 1);
        umma::mbar_init(&sm.bar_g3, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(&sm.tmem_slot, kTmemCols);
    pdl_trigger();
    pdl_wait();
    // b1, b2 and w3 arrive by bulk copies with the first tile's images (one
    // round of latency for everything the tile needs) when H = 128 and the
    // parameters are 16-byte aligned; else (zero-padded units) loaded here
    const bool bulk_bias = Hn == HH && (reinterpret_cast<uintptr_t>(prm) & 15) == 0;
    for (int i = tid; i < HH; i += kThreads) {
        if (!bulk_bias) {
            const bool u = i < Hn;   // padded units: zero bias and output weight, so they stay zero
            sm.b1[i] = u ? __ldg(prm + off.b1 + i) : 0.0f;
            sm.b2[i] = u ? __ldg(prm + off.b2 + i) : 0.0f;
            sm.w3[i] = u ? __ldg(prm + off.w3 + i) : 0.0f;
        }
        sm.vec[0][i] = sm.vec[1][i] = sm.vec[2][i] = 0.0f;
    }
    if (tid == 0) sm.vb3 = 0.0f;
    const float b3 = __ldg(prm + off.b3);
    uint32_t tmem = 0, tq = 0;
    uint32_t ph_mma = 0, ph_load = 0, ph_g3 = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        ok &= umma::mbar_wait(&sm.bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1u;
        umma::fence_after_sync();
    };
    auto wait_load = [&]() {
        ok &= umma::mbar_wait(&sm.bar_load, ph_load, kWaitNs);
        ph_load ^= 1u;
    };

    // Tiles blockIdx.x, blockIdx.x + gridDim.x, ...: the weight-gradient
    // accumulators (dW2, dW1 in TMEM; dW3, db2, db1, db3 in shared memory)
    // run over all of them; one partial per CTA at the end.
    for (int tile = blockIdx.x, it = 0; tile < n_tiles; tile += gridDim.x, ++it) {
        const int row0 = tile * TM;
        const uint8_t* xi = a.ximg != nullptr ? a.ximg + (int64_t)tile * NP * kPlaneX : nullptr;
        // ---- stage 1: X image -> R0, W1 image -> R1, and the tile's Q rows
        // and actions (one contiguous block each) for the loss and the policy,
        // all by bulk copies on one barrier (the previous tile's G5 has
        // finished reading R0 and R1); Q and the actions by loads where a
        // copy's address or size is not a multiple of 16 bytes ----
        const int nrow = B - row0 < TM ? B - row0 : TM;
        const float* qsrc = a.q != nullptr ? a.q + (int64_t)row0 * NA : a.q_taken + row0;
        const uint32_t qbytes = (uint32_t)(nrow * (a.q != nullptr ? NA : 1)) * 4u;
        const bool bulk_q = (nrow & 3) == 0 && (reinterpret_cast<uintptr_t>(qsrc) & 15) == 0 &&
                            (a.q == nullptr || (reinterpret_cast<uintptr_t>(a.actions + row0) & 15) == 0);
        if (tid == 0) {
            uint32_t bytes = (xi ? kXBytes : 0u) + kXBytes;
            if (it == 0 && bulk_bias) bytes += 3u * HH * 4u;
            if (bulk_q) bytes += qbytes + (a.q != nullptr ? (uint32_t)nrow * 4u : 0u);
            umma::mbar_expect_tx(&sm.bar_load, bytes);
            if (xi) umma::bulk_g2s(sm.r0, xi, kXBytes, &sm.bar_load);
            umma::bulk_g2s(sm.r1, w1i, kXBytes, &sm.bar_load);
            if (it == 0 && bulk_bias) {
                umma::bulk_g2s(sm.b1, prm + off.b1, HH * 4u, &sm.bar_load);
                umma::bulk_g2s(sm.b2, prm + off.b2, 2u * HH * 4u, &sm.bar_load);   // b2, then w3
            }
            if (bulk_q) {
                umma::bulk_g2s(sm.qt, qsrc, qbytes, &sm.bar_load);
                if (a.q != nullptr) umma::bulk_g2s(sm.act, a.actions + row0, (uint32_t)nrow * 4u, &sm.bar_load);
            }
        }
        if (!bulk_q) {
            if (a.q != nullptr) {
                for (int e = tid; e < nrow * NA; e += kThreads) sm.qt[e] = __ldg(qsrc + e);
                for (int e = tid; e < nrow; e += kThreads) sm.act[e] = __ldg(a.actions + row0 + e);
            } else {
                for (int e = tid; e < nrow; e += kThreads) sm.qt[e] = __ldg(qsrc + e);
            }
        }
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        tmem = sm.tmem_slot;
        tq = tmem + ((uint32_t)(32 * q) << 16);   // this warp's lane quarter

        if (!xi) build_x(sm.r0, NP, a.states, a.stride, row0, B, S);
        umma::fence_smem_to_async();
        __syncthreads();
        wait_load();
        // ---- G1: z1 = X . W1^T ----
        if (tid == 0) {
            umma::fence_after_sync();
            gemm<NP>(tmem + TM_Z1, sm.r0, kPlaneX, KX, false, sm.r1, kPlaneX, KX, false, KX / 16, HN);
            umma::commit(&sm.bar_mma);
        }
        wait_mma();
        // W1 is no longer read: the W2 image streams into R1 during epilogue 1
        if (tid == 0) {
            umma::mbar_expect_tx(&sm.bar_load, kW2Bytes);
            umma::bulk_g2s(sm.r1, w2i, kW2Bytes, &sm.bar_load);
        }

        // ---- epilogue 1: h1 = relu(z1 + b1) -> R0; ReLU mask bits kept ----
        uint32_t mask1 = 0;
        if (epi && live) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float v[16];
                umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
                umma::tmem_ld_wait();
                float bb[16];
                lds16(sm.b1 + c0, bb);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float z = v[j] + bb[j];
                    v[j] = z < 0.0f ? 0.0f : z;
                    if (v[j] > 0.0f) mask1 |= 1u << (cc * 16 + j);
                }
                store16<NP>(sm.r0, row, c0, v);
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        wait_load();
        // ---- G2: z2 = h1 . W2^T ----
        if (tid == 0) {
            umma::fence_after_sync();
            gemm<NP>(tmem + TM_Z2, sm.r0, kPlaneH, HH, false, sm.r1, kPlaneH, HH, false, HN / 16, HN);
            umma::commit(&sm.bar_mma);
        }
        wait_mma();

        // ---- epilogue 2: V, loss, dV, dz2; then dW3 / db2 / db3 beside G3, G4 ----
        // z2 is read from TMEM twice (for V, then for dz2) instead of being kept
        // in registers across the row reduction.
        if (epi) {
            float vp = 0.0f;
#pragma unroll
            for (int cc = 0; cc < 2 && live; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float v[16];
                umma::tmem_ld16(tq + TM_Z2 + (uint32_t)c0, v);
                umma::tmem_ld_wait();
                float bb[16], ww[16];
                lds16(sm.b2 + c0, bb);
                lds16(sm.w3 + c0, ww);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float z = v[j] + bb[j];
                    vp = fmaf(z < 0.0f ? 0.0f : z, ww[j], vp);
                }
            }
            sm.vsum[cg][row] = vp;
        }
        __syncthreads();
        const float V = ((sm.vsum[0][row] + sm.vsum[1][row]) + (sm.vsum[2][row] + sm.vsum[3][row])) + b3;
        const int b = row0 + row;
        float dv = 0.0f, lossp = 0.0f;
        if (epi && b < B) {
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
        if (epi && cg == 0) sm.vrow[row] = V;
        // dz2 in its two planes -> the plane-2 slots of R0 and R1, which G2 was
        // the last to read (the backward GEMMs read planes 0 and 1 of h1 and
        // W2), so W2 stays in R1 for G4 and G3, G4 run back to back
        uint8_t* const dz2 = sm.r0 + 2u * kPlaneH;   // plane 1 at dz2 + kRegion
        if (epi && live) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float g[16];
                umma::tmem_ld16(tq + TM_Z2 + (uint32_t)c0, g);
                umma::tmem_ld_wait();
                float bb[16], ww[16];
                lds16(sm.b2 + c0, bb);
                lds16(sm.w3 + c0, ww);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float z = g[j] + bb[j];
                    g[j] = z > 0.0f ? dv * ww[j] : 0.0f;
                }
                store16<NP, true>(dz2, row, c0, g, kRegion);
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        // ---- G3: dW2 = dz2^T . h1, then G4: dh1 = dz2 . W2 (into z1's
        // columns: the ReLU mask of z1 is in registers) ----
        if (tid == 0) {
            umma::fence_after_sync();
            gemm<NP, true>(tmem + TM_DW2, dz2, kRegion, HH, true, sm.r0, kPlaneH, HH, true, TM / 16, HN, it > 0);
            umma::commit(&sm.bar_g3);
            gemm<NP, true>(tmem + TM_Z1, dz2, kRegion, HH, false, sm.r1, kPlaneH, HH, true, HN / 16, HN);
            umma::commit(&sm.bar_mma);
            // h1 is no longer read once G3 is done: the planes of the X image
            // that G5 reads stream into R0 while G4 runs
            ok &= umma::mbar_wait(&sm.bar_g3, ph_g3, kWaitNs);
            ph_g3 ^= 1u;
            umma::fence_after_sync();
            if (xi) {
                umma::mbar_expect_tx(&sm.bar_load, kX2Bytes);
                umma::bulk_g2s(sm.r0, xi, kX2Bytes, &sm.bar_load);
            }
        }
        if (epi && cg == 0) {
            const float ls = warp_sum(lossp), ds = warp_sum(dv);
            if (lane == 0) { sm.lred[0][q] = ls; sm.lred[1][q] = ds; }
        }
        // column sums for dW3 and db2 beside the two GEMMs
        if (epi && live) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float g[16], hw[16];
                umma::tmem_ld16(tq + TM_Z2 + (uint32_t)c0, g);
                umma::tmem_ld_wait();
                float bb[16], ww[16];
                lds16(sm.b2 + c0, bb);
                lds16(sm.w3 + c0, ww);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float z = g[j] + bb[j];
                    g[j] = z > 0.0f ? dv * ww[j] : 0.0f;
                    hw[j] = dv * (z < 0.0f ? 0.0f : z);
                }
                const float s3 = colsum16(hw);
                const float s2 = colsum16(g);
                if ((lane & 1) == 0) {
                    sm.red[0][ew][cc * 16 + ((lane >> 1) & 15)] = s3;
                    sm.red[1][ew][cc * 16 + ((lane >> 1) & 15)] = s2;
                }
            }
        }
        __syncthreads();
        // dW3, db2, db3 and the loss partial of the tile (fixed order over warps)
        for (int c = et; c >= 0 && c < HH; c += kThreads) {
            const int g = c >> 5, cl = c & 31;
            float s3 = 0.0f, s2 = 0.0f;
            for (int qq = 0; qq < 4; ++qq) { s3 += sm.red[0][g * 4 + qq][cl]; s2 += sm.red[1][g * 4 + qq][cl]; }
            sm.vec[0][c] += s3;
            sm.vec[1][c] += s2;
        }
        if (et == 0) {
            const float l = (sm.lred[0][0] + sm.lred[0][1]) + (sm.lred[0][2] + sm.lred[0][3]);
            const float d3 = (sm.lred[1][0] + sm.lred[1][1]) + (sm.lred[1][2] + sm.lred[1][3]);
            a.tile_loss[(int64_t)net * a.net_tile_stride + tile] = l;
            sm.vb3 += d3;
        }
        wait_mma();

        // ---- epilogue 4: dz1 = dh1 * 1[z1 > 0] -> R1 (W2 is no longer read);
        // without relabel images the X image is built in R0 here ----
        if (epi && live) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float v[16];
                umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
                umma::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = ((mask1 >> (cc * 16 + j)) & 1u) ? v[j] : 0.0f;
                store16<NP, true>(sm.r1, row, c0, v);
            }
        }
        if (!xi) build_x(sm.r0, NP, a.states, a.stride, row0, B, S);
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        if (xi) wait_load();
        // ---- G5: dW1 = dz1^T . X ----
        if (tid == 0) {
            umma::fence_after_sync();
            gemm<NP, true>(tmem + TM_DW1, sm.r1, kPlaneH, HH, true, sm.r0, kPlaneX, KX, true, TM / 16, KX, it > 0);
            umma::commit(&sm.bar_mma);
        }
        // the policy while G5 runs (beside G3 and G4 it would share their
        // window with the column sums): four threads per row (lanes 4r .. 4r + 3
        // of a warp), each over actions j, j + 4, ... (its exponentials kept in
        // registers); max / argmax (lowest index on ties) and the sum of
        // exponentials combined over the four lanes
        if (epi && a.pi_out != nullptr) {
            constexpr int kPer = kMaxActions / 4;
            const int pr = et >> 2, j = et & 3;
            const int pb = row0 + pr;
            const bool prow = pb < B;
            const float Vp = sm.vrow[pr];
            const float* qr = sm.qt + pr * NA;
            float adv[kPer];
            float zmax = -INFINITY, amax = -INFINITY;
            int best = NA;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int k = j + 4 * i;
                adv[i] = prow && k < NA ? fminf(fmaxf(qr[k] - Vp, -10.0f), 10.0f) : -INFINITY;
                if (adv[i] > amax) { amax = adv[i]; best = k; }
                if (prow && k < NA) zmax = fmaxf(zmax, a.beta * adv[i]);
            }
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                const float oa = __shfl_xor_sync(0xffffffffu, amax, o);
                const int ob = __shfl_xor_sync(0xffffffffu, best, o);
                if (oa > amax || (oa == amax && ob < best)) { amax = oa; best = ob; }
                zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
            }
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                adv[i] = j + 4 * i < NA ? expf(a.beta * adv[i] - zmax) : 0.0f;
                sum += adv[i];
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            if (prow) {
                float* po = a.pi_out + ((int64_t)net * B + pb) * NA;
#pragma unroll
                for (int i = 0; i < kPer; ++i)
                    if (j + 4 * i < NA) po[j + 4 * i] = adv[i] / sum;
                if (j == 0 && a.argmax_out != nullptr) a.argmax_out[(int64_t)net * B + pb] = best < NA ? best : 0;
            }
        }
        // db1: with S < 64 G5 yields it in its last column (the ones column of
        // the state-tile image); else column sums while G5 runs
        if (epi && live && !tc::ones_column(KX - 1, S)) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float v[16];
                umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
                umma::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = ((mask1 >> (cc * 16 + j)) & 1u) ? v[j] : 0.0f;
                const float s1 = colsum16(v);
                if ((lane & 1) == 0) sm.red[2][ew][cc * 16 + ((lane >> 1) & 15)] = s1;
            }
        }
        __syncthreads();
        for (int c = et; c >= 0 && c < HH; c += kThreads) {
            const int g = c >> 5, cl = c & 31;
            float s1 = 0.0f;
            for (int qq = 0; qq < 4; ++qq) s1 += sm.red[2][g * 4 + qq][cl];
            if (!tc::ones_column(KX - 1, S)) sm.vec[2][c] += s1;
        }
        wait_mma();
    }   // tiles

    // ---- dW2 (lane = output unit, 128 columns) and dW1 (lane = unit, 64 columns) ----
    // Staged in shared memory (R0, R1 are free now): dW2 rows at a padded
    // stride of 132 floats, so the float4 stores of 8 consecutive lanes
    // (8 rows) fall on distinct banks; dW1 unpadded.
    constexpr int kStride2 = HH + 4;
    float* st2 = reinterpret_cast<float*>(sm.r0);            // [HH][kStride2]
    float* st1 = reinterpret_cast<float*>(sm.r1);            // [HH][S]
    if (epi) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            float v[16];
            umma::tmem_ld16(tq + TM_DW2 + (uint32_t)(cg * 32 + cc * 16), v);
            umma::tmem_ld_wait();
            float4* dst = reinterpret_cast<float4*>(st2 + row * kStride2 + cg * 32 + cc * 16);
#pragma unroll
            for (int f = 0; f < 4; ++f) dst[f] = make_float4(v[4 * f], v[4 * f + 1], v[4 * f + 2], v[4 * f + 3]);
        }
    }
    if (epi) {
        const int c0 = cg * 16;
        float v[16];
        umma::tmem_ld16(tq + TM_DW1 + (uint32_t)c0, v);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (c0 + j < S) st1[row * S + c0 + j] = v[j];
        if (c0 + 15 == KX - 1 && tc::ones_column(KX - 1, S)) sm.vec[2][row] = v[15];
    }

    // this CTA's partial: one bulk copy per dW2 row (H floats), one for dW1,
    // one per vector (all offsets and sizes multiples of 16 bytes)
    float* dst = a.partials + (int64_t)net * a.net_partial_stride + (int64_t)blockIdx.x * a.part_stride;
    umma::fence_smem_to_async();
    __syncthreads();
    if (tid < Hn) {
        umma::bulk_s2g(dst + off.w2 + tid * Hn, st2 + tid * kStride2, (uint32_t)(Hn * 4));
        if (tid == 0) umma::bulk_s2g(dst + off.w1, st1, (uint32_t)(Hn * S * 4));
        if (tid == 1) umma::bulk_s2g(dst + off.w3, sm.vec[0], (uint32_t)(Hn * 4));
        if (tid == 2) umma::bulk_s2g(dst + off.b2, sm.vec[1], (uint32_t)(Hn * 4));
        if (tid == 3) umma::bulk_s2g(dst + off.b1, sm.vec[2], (uint32_t)(Hn * 4));
        if (tid == 4) dst[off.b3] = sm.vb3;
        umma::bulk_commit();
        umma::bulk_wait_read();
    }
    if (!ok && tid == 0) atomicAdd(a.status + OFRL_STAT_TIMEOUT, 1);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

// V forward only on the tensor cores ("GPU IQL + HER Porting Plan", "Rust
// Integration: gpu_iql_trainer.rs", forward_values, and "IQL modifies the
// target computation"): per 128-row tile G1 z1 = X W1^T, h1 = relu(z1 + b1)
// as the image G2 reads, G2 z2 = h1 W2^T, V = relu(z2 + b2) . w3 + b3; with
// target_out also r + gamma (1 - done) V.  The state tile is built here from
// the caller's fp32 states (the fused step's relabel is not involved), the
// weight images come from pack_weights_kernel.  Same warp roles, regions and
// bounded waits as vnet_tc_kernel; 256 TMEM columns (z1, z2).
template <int NP>
__global__ void __launch_bounds__(kThreads, 1) vnet_tc_forward_kernel(const VnetLaunch a,
                                                                      const uint8_t* __restrict__ wimg) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp != 0;
    const int q = warp & 3, cg = (warp - 1) >> 2;
    const int row = 32 * q + lane;
    const int S = a.state_dim, B = a.batch;
    const int n_tiles = (B + TM - 1) / TM;
    const int Hn = a.hidden;
    const Offsets off = offsets_of(S, Hn);
    const int HN = Hn <= 64 ? 64 : HH;   // the units computed (as in the training kernel)
    const bool live = cg * 32 < HN;
    const float* __restrict__ prm = a.params[0];
    const uint8_t* w1i = wimg;
    const uint8_t* w2i = w1i + tc::w2_image_offset();
    constexpr uint32_t kXBytes = (uint32_t)NP * kPlaneX, kW2Bytes = (uint32_t)NP * kPlaneH;
    constexpr uint32_t kCols = 256;

    if (tid == 0) {
        umma::mbar_init(&sm.bar_mma, 1);
        umma::mbar_init(&sm.bar_load, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(&sm.tmem_slot, kCols);
    pdl_trigger();
    pdl_wait();
    for (int i = tid; i < HH; i += kThreads) {
        const bool u = i < Hn;
        sm.b1[i] = u ? __ldg(prm + off.b1 + i) : 0.0f;
        sm.b2[i] = u ? __ldg(prm + off.b2 + i) : 0.0f;
        sm.w3[i] = u ? __ldg(prm + off.w3 + i) : 0.0f;
    }
    const float b3 = __ldg(prm + off.b3);
    uint32_t ph_mma = 0, ph_load = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        ok &= umma::mbar_wait(&sm.bar_mma, ph_mma, kWaitNs);
        ph_mma ^= 1u;
        umma::fence_after_sync();
    };
    auto wait_load = [&]() {
        ok &= umma::mbar_wait(&sm.bar_load, ph_load, kWaitNs);
        ph_load ^= 1u;
    };

    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int row0 = tile * TM;
        // W1 image -> R1 (the previous tile's G2 has finished reading R1)
        if (tid == 0) {
            umma::mbar_expect_tx(&sm.bar_load, kXBytes);
            umma::bulk_g2s(sm.r1, w1i, kXBytes, &sm.bar_load);
        }
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        const uint32_t tmem = sm.tmem_slot;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        build_x<true>(sm.r0, NP, a.states, a.stride, row0, B, S);
        umma::fence_smem_to_async();
        __syncthreads();
        wait_load();
        // ---- G1: z1 = X . W1^T ----
        if (tid == 0) {
            umma::fence_after_sync();
            gemm<NP>(tmem + TM_Z1, sm.r0, kPlaneX, KX, false, sm.r1, kPlaneX, KX, false, KX / 16, HN);
            umma::commit(&sm.bar_mma);
        }
        wait_mma();
        if (tid == 0) {
            umma::mbar_expect_tx(&sm.bar_load, kW2Bytes);
            umma::bulk_g2s(sm.r1, w2i, kW2Bytes, &sm.bar_load);
        }
        // ---- epilogue 1: h1 = relu(z1 + b1) -> R0 ----
        if (epi && live) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float v[16];
                umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
                umma::tmem_ld_wait();
                float bb[16];
                lds16(sm.b1 + c0, bb);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float z = v[j] + bb[j];
                    v[j] = z < 0.0f ? 0.0f : z;
                }
                store16<NP>(sm.r0, row, c0, v);
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        wait_load();
        // ---- G2: z2 = h1 . W2^T ----
        if (tid == 0) {
            umma::fence_after_sync();
            gemm<NP>(tmem + TM_Z2, sm.r0, kPlaneH, HH, false, sm.r1, kPlaneH, HH, false, HN / 16, HN);
            umma::commit(&sm.bar_mma);
        }
        wait_mma();
        // ---- epilogue 2: V (and the target) ----
        if (epi) {
            float vp = 0.0f;
#pragma unroll
            for (int cc = 0; cc < 2 && live; ++cc) {
                const int c0 = cg * 32 + cc * 16;
                float v[16];
                umma::tmem_ld16(tq + TM_Z2 + (uint32_t)c0, v);
                umma::tmem_ld_wait();
                float bb[16], ww[16];
                lds16(sm.b2 + c0, bb);
                lds16(sm.w3 + c0, ww);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float z = v[j] + bb[j];
                    vp = fmaf(z < 0.0f ? 0.0f : z, ww[j], vp);
                }
            }
            sm.vsum[cg][row] = vp;
        }
        __syncthreads();
        const int b = row0 + row;
        if (epi && cg == 0 && b < B) {
            const float V = ((sm.vsum[0][row] + sm.vsum[1][row]) + (sm.vsum[2][row] + sm.vsum[3][row])) + b3;
            if (a.v_out != nullptr) a.v_out[b] = V;
            if (a.target_out != nullptr)
                a.target_out[b] = __ldg(a.rewards + b) + a.gamma * (1.0f - __ldg(a.dones + b)) * V;
        }
    }
    if (!ok && tid == 0) atomicAdd(a.status + OFRL_STAT_TIMEOUT, 1);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_slot, kCols);
}

// Pack W1 ([H][S] -> [128 x 64] image) and W2 ([H][H] -> [128 x 128] image)
// of every network into NP bf16 planes each, units past H zero (standalone V
// forward/backward; the fused step packs inside the relabel launch).
__global__ void pack_weights_kernel(const VnetLaunch a, uint8_t* __restrict__ img, int np) {
    const int net = blockIdx.y;
    const int S = a.state_dim, Hn = a.hidden;
    const Offsets off = offsets_of(S, Hn);
    const float* __restrict__ prm = a.params[net];
    uint8_t* w1i = img + (int64_t)net * tc::weight_image_bytes();
    uint8_t* w2i = w1i + tc::w2_image_offset();
    const int n1 = HH * (KX / 4), n2 = HH * (HH / 4);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n1 + n2; e += gridDim.x * blockDim.x) {
        float x[4];
        if (e < n1) {
            const int r = e / (KX / 4), c = 4 * (e % (KX / 4));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                x[j] = r < Hn && c + j < S ? __ldg(prm + off.w1 + (int64_t)r * S + c + j) : 0.0f;
            tc::put4(w1i, kPlaneX, np, KX, r, c, x);
        } else {
            const int f = e - n1, r = f / (HH / 4), c = 4 * (f % (HH / 4));
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = r < Hn && c + j < Hn ? __ldg(prm + off.w2 + (int64_t)r * Hn + c + j) : 0.0f;
            tc::put4(w2i, kPlaneH, np, HH, r, c, x);
        }
    }
}

template <int NP>
cudaError_t configure_np() {
    static cudaError_t state = cudaErrorNotReady;
    if (state == cudaErrorNotReady) {
        auto kern = vnet_tc_kernel<NP>;
        state = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(TcSmem));
        if (state == cudaSuccess) state = set_max_shared_carveout(kern);
    }
    return state;
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                       cudaSuccess)
            n = 1;
        cudaGetLastError();
    }
    return n;
}

template <int NP>
cudaError_t launch_np(const VnetLaunch& a, const uint8_t* wimg, cudaStream_t st) {
    const cudaError_t e = configure_np<NP>();
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.batch + TM - 1) / TM;
    const dim3 grid((unsigned)vnet_tc_ctas(n_tiles, a.n_nets), a.n_nets);
    return launch_pdl(vnet_tc_kernel<NP>, grid, dim3(kThreads), sizeof(TcSmem), st, a, wimg);
}

template <int NP>
cudaError_t launch_forward_np(const VnetLaunch& a, const uint8_t* wimg, cudaStream_t st) {
    static cudaError_t state = cudaErrorNotReady;
    if (state == cudaErrorNotReady) {
        auto kern = vnet_tc_forward_kernel<NP>;
        state = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(TcSmem));
        if (state == cudaSuccess) state = set_max_shared_carveout(kern);
    }
    if (state != cudaSuccess) return state;
    const int n_tiles = (a.batch + TM - 1) / TM;
    const dim3 grid((unsigned)vnet_tc_ctas(n_tiles, 1));
    return launch_pdl(vnet_tc_forward_kernel<NP>, grid, dim3(kThreads), sizeof(TcSmem), st, a, wimg);
}

}  // namespace

int64_t vnet_tc_image_bytes() { return tc::weight_image_bytes(); }

int vnet_tc_ctas(int n_tiles, int n_nets) {
    // one wave of one CTA per SM, the tiles spread evenly: with more tiles
    // than that, each CTA runs ceil(tiles / CTAs) of them back to back and
    // writes one partial (512 tiles: 128 CTAs of 4 tiles)
    const int per_net = num_sms() / (n_nets > 0 ? n_nets : 1) > 0 ? num_sms() / (n_nets > 0 ? n_nets : 1) : 1;
    const int per_cta = (n_tiles + per_net - 1) / per_net;
    return (n_tiles + per_cta - 1) / per_cta;
}

bool vnet_tc_supported(const VnetLaunch& a) {
    return (a.hidden == HH || a.hidden == HH / 2) && a.state_dim <= KX && (a.stride & 3) == 0 &&
           (reinterpret_cast<uintptr_t>(a.states) & 15) == 0;
}

cudaError_t launch_vnet_tc_pack(const VnetLaunch& a, uint8_t* img, cudaStream_t st) {
    pack_weights_kernel<<<dim3(32, a.n_nets), 256, 0, st>>>(a, img, a.prec == OFRL_PREC_BF16 ? 1 : 3);
    return cudaGetLastError();
}

cudaError_t launch_vnet_tc(const VnetLaunch& a, const uint8_t* img, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    return a.prec == OFRL_PREC_BF16 ? launch_np<1>(a, img, st) : launch_np<3>(a, img, st);
}

cudaError_t launch_vnet_tc_forward(const VnetLaunch& a, uint8_t* img, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    VnetLaunch one = a;
    one.n_nets = 1;
    cudaError_t e = launch_vnet_tc_pack(one, img, st);
    if (e != cudaSuccess) return e;
    return a.prec == OFRL_PREC_BF16 ? launch_forward_np<1>(one, img, st) : launch_forward_np<3>(one, img, st);
}

}  // namespace ofrl
