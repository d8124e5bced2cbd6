// IQL value network V(s) forward, expectile loss, policy and backward for one
// 128-row batch tile per CTA on the 5th-generation tensor cores (tcgen05),
// hidden width 128.
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
// Every operand lives in shared memory as an "image": bf16 core matrices of
// 8 rows x 8 elements (16 bytes), chunk-major inside 8-row groups.  The same
// image of an activation tile is the K-major operand of one GEMM and the
// MN-major operand of another, so nothing is transposed.
//
// Precision: for fp32 results each fp32 operand is split into three bf16
// terms x = x0 + x1 + x2 (24 significand bits) and each K-step issues the six
// products whose size reaches 2^-16 of the leading one (x2 y0, x1 y1, x0 y2,
// x1 y0, x0 y1, x0 y0); the dropped ones are below fp32 rounding.  For the
// bf16 workload the operands are bf16 and one product is issued.
//
// Shared memory: two 96 KB regions reused through the step:
//   R0: X image -> h1 -> W2 image (for G4) -> dz1
//   R1: W1 image -> W2 image (for G2) -> dz2 -> X image (for G5)
// Weight images come from the pack kernel in global memory (one bulk async
// copy each); X images are built by the CTA's threads from the fp32 batch.

#include "common.cuh"
#include "umma.cuh"

namespace ofrl {
namespace {

constexpr int kThreads = 256;
constexpr int TM = 128;     // batch rows per tile (MMA M)
constexpr int HH = 128;     // hidden width of this kernel
constexpr int KX = 64;      // state columns, padded (K of G1, N of G5)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_Z1 = 0, TM_Z2 = 128, TM_DW2 = 256, TM_DW1 = 384;   // TM_Z1 also holds dh1
constexpr uint32_t kPlaneH = TM * HH * 2;    // one bf16 plane of a [128 x 128] image
constexpr uint32_t kPlaneX = TM * KX * 2;    // one bf16 plane of a [128 x 64] image
constexpr uint32_t kRegion = 3 * kPlaneH;    // 96 KB
constexpr uint64_t kWaitNs = 1000000000ull;  // bounded waits: 1 s

// Byte offset of element (r, c) inside one plane of an image with C columns.
__device__ __forceinline__ uint32_t img_off(int r, int c, int C) {
    return (uint32_t)((r >> 3) * (C >> 3) * 128 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

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
template <int NP>
__device__ __forceinline__ void gemm(uint32_t d_tmem, const uint8_t* a, uint32_t a_plane, int a_cols, bool a_mn,
                                     const uint8_t* b, uint32_t b_plane, int b_cols, bool b_mn, int ksteps, int n) {
    const uint32_t idesc = umma::instr_desc(umma::kTypeBF16, a_mn, b_mn, TM, n);
    // (a term, b term): smallest products first
    constexpr int na = NP == 3 ? 6 : 1;
    const int ta[6] = {2, 1, 0, 1, 0, 0};
    const int tb[6] = {0, 1, 2, 0, 1, 0};
    uint32_t acc = 0;
    for (int ks = 0; ks < ksteps; ++ks) {
#pragma unroll
        for (int t = 0; t < na; ++t) {
            const int pa = NP == 3 ? ta[t] : 0, pb = NP == 3 ? tb[t] : 0;
            const uint8_t* ap = a + (uint32_t)pa * a_plane;
            const uint8_t* bp = b + (uint32_t)pb * b_plane;
            const uint64_t ad = a_mn ? desc_mn(ap, a_cols, ks) : desc_k(ap, a_cols, ks);
            const uint64_t bd = b_mn ? desc_mn(bp, b_cols, ks) : desc_k(bp, b_cols, ks);
            umma::mma_f16(d_tmem, ad, bd, idesc, acc);
            acc = 1;
        }
    }
}

// Store 16 fp32 values of row r, columns c0..c0+15 (c0 a multiple of 16) into
// an image with C columns, as NP bf16 planes.
template <int NP>
__device__ __forceinline__ void store16(uint8_t* img, uint32_t plane, int C, int r, int c0, const float (&v)[16]) {
    __nv_bfloat16 t[3][16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (NP == 3) umma::split_bf16x3(v[j], t[0][j], t[1][j], t[2][j]);
        else t[0][j] = __float2bfloat16_rn(v[j]);
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        uint8_t* base = img + (uint32_t)p * plane;
        *reinterpret_cast<uint4*>(base + img_off(r, c0, C)) = *reinterpret_cast<const uint4*>(&t[p][0]);
        *reinterpret_cast<uint4*>(base + img_off(r, c0 + 8, C)) = *reinterpret_cast<const uint4*>(&t[p][8]);
    }
}

// Build the X image ([128 x 64], NP planes) of this tile from the fp32 batch:
// rows past the batch and columns past S are zero.
template <int NP>
__device__ __forceinline__ void build_x(uint8_t* img, const float* __restrict__ states, int stride, int row0, int B,
                                        int S) {
    for (int e = threadIdx.x; e < TM * (KX / 4); e += kThreads) {
        const int r = e / (KX / 4), c = 4 * (e % (KX / 4));
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + r < B && c < S) v = __ldg(reinterpret_cast<const float4*>(states + (int64_t)(row0 + r) * stride + c));
        float x[4] = {v.x, v.y, v.z, v.w};
        __nv_bfloat16 t[3][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (c + j >= S) x[j] = 0.0f;
            if (NP == 3) umma::split_bf16x3(x[j], t[0][j], t[1][j], t[2][j]);
            else t[0][j] = __float2bfloat16_rn(x[j]);
        }
#pragma unroll
        for (int p = 0; p < NP; ++p)
            *reinterpret_cast<uint2*>(img + (uint32_t)p * kPlaneX + img_off(r, c, KX)) =
                *reinterpret_cast<const uint2*>(&t[p][0]);
    }
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

struct TcSmem {
    uint8_t r0[kRegion];
    uint8_t r1[kRegion];
    float b1[HH], b2[HH], w3[HH];
    float vsum[2][TM];
    float red[3][8][64];    // per warp column sums: dW3, db2, db1
    float lred[2][8];       // per warp: loss, db3
    uint64_t bar_mma, bar_load;
    uint32_t tmem_slot;
};

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) vnet_tc_kernel(const VnetLaunch a, const uint8_t* __restrict__ w1img,
                                                              const uint8_t* __restrict__ w2img, int64_t img_stride) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hh = warp >> 2;      // TMEM lane quarter, column half
    const int row = 32 * q + lane;               // this thread's tile row (accumulator lane)
    const int tile = blockIdx.x, net = blockIdx.y;
    const int S = a.state_dim, B = a.batch, NA = a.num_actions;
    const int row0 = tile * TM;
    const Offsets off = offsets_of(S, HH);
    const float* __restrict__ prm = a.params[net];
    const float tau = a.tau[net];
    float* part = a.partials + (int64_t)net * a.net_partial_stride + (int64_t)tile * a.part_stride;
    const uint8_t* w1i = w1img + (int64_t)net * img_stride;
    const uint8_t* w2i = w1i + (uint32_t)NP * kPlaneX;
    (void)w2img;
    constexpr uint32_t kW1Bytes = (uint32_t)NP * kPlaneX, kW2Bytes = (uint32_t)NP * kPlaneH;

    if (tid == 0) {
        umma::mbar_init(&sm.bar_mma, 1);
        umma::mbar_init(&sm.bar_load, 1);
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(&sm.tmem_slot, kTmemCols);
    for (int i = tid; i < HH; i += kThreads) {
        sm.b1[i] = __ldg(prm + off.b1 + i);
        sm.b2[i] = __ldg(prm + off.b2 + i);
        sm.w3[i] = __ldg(prm + off.w3 + i);
    }
    const float b3 = __ldg(prm + off.b3);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_slot;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);   // this warp's lane quarter
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

    // ---- stage 1: W1 image -> R1 (bulk copy), X image -> R0 (threads) ----
    if (tid == 0) {
        umma::mbar_expect_tx(&sm.bar_load, kW1Bytes);
        umma::bulk_g2s(sm.r1, w1i, kW1Bytes, &sm.bar_load);
    }
    build_x<NP>(sm.r0, a.states, a.stride, row0, B, S);
    umma::fence_smem_to_async();
    __syncthreads();
    wait_load();
    // ---- G1: z1 = X . W1^T ----
    if (tid == 0) {
        umma::fence_after_sync();
        gemm<NP>(tmem + TM_Z1, sm.r0, kPlaneX, KX, false, sm.r1, kPlaneX, KX, false, KX / 16, HH);
        umma::commit(&sm.bar_mma);
    }
    wait_mma();

    // ---- epilogue 1: h1 = relu(z1 + b1) -> R0; ReLU mask bits kept ----
    uint64_t mask1 = 0;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int c0 = hh * 64 + cc * 16;
        float v[16];
        umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float z = v[j] + sm.b1[c0 + j];
            v[j] = z < 0.0f ? 0.0f : z;
            if (v[j] > 0.0f) mask1 |= 1ull << (cc * 16 + j);
        }
        store16<NP>(sm.r0, kPlaneH, HH, row, c0, v);
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();
    // ---- stage 2: W2 image -> R1 ----
    if (tid == 0) {
        umma::mbar_expect_tx(&sm.bar_load, kW2Bytes);
        umma::bulk_g2s(sm.r1, w2i, kW2Bytes, &sm.bar_load);
    }
    wait_load();
    // ---- G2: z2 = h1 . W2^T ----
    if (tid == 0) {
        umma::fence_after_sync();
        gemm<NP>(tmem + TM_Z2, sm.r0, kPlaneH, HH, false, sm.r1, kPlaneH, HH, false, HH / 16, HH);
        umma::commit(&sm.bar_mma);
    }
    wait_mma();

    // ---- epilogue 2: V, loss, dV, policy, dz2 -> R1, dW3 / db2 / db3 ----
    float z2[64];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        float v[16];
        umma::tmem_ld16(tq + TM_Z2 + (uint32_t)(hh * 64 + cc * 16), v);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) z2[cc * 16 + j] = v[j] + sm.b2[hh * 64 + cc * 16 + j];
    }
    {
        float vp = 0.0f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            const float h = z2[j] < 0.0f ? 0.0f : z2[j];
            vp = fmaf(h, sm.w3[hh * 64 + j], vp);
        }
        sm.vsum[hh][row] = vp;
    }
    __syncthreads();
    const float V = (sm.vsum[0][row] + sm.vsum[1][row]) + b3;
    const int b = row0 + row;
    float dv = 0.0f, lossp = 0.0f;
    if (b < B) {
        float qv;
        if (a.q != nullptr) {
            int act = __ldg(a.actions + b);
            if (act < 0 || act >= NA) {
                if (hh == 0) atomicAdd(a.status + OFRL_STAT_BAD_ACTION, 1);
                act = 0;
            }
            qv = __ldg(a.q + (int64_t)b * NA + act);
        } else {
            qv = __ldg(a.q_taken + b);
        }
        const float d = qv - V;
        const float w = d >= 0.0f ? tau : 1.0f - tau;
        lossp = w * d * d;
        dv = (-2.0f * w * d) / (float)B;
        if (hh == 0 && a.v_out != nullptr) a.v_out[(int64_t)net * B + b] = V;
        if (hh == 1 && a.pi_out != nullptr) {
            const float* qr = a.q + (int64_t)b * NA;
            float zz[kMaxActions];
            float zmax = -INFINITY, amax = -INFINITY;
            int best = 0;
            for (int k = 0; k < NA; ++k) {
                const float adv = fminf(fmaxf(__ldg(qr + k) - V, -10.0f), 10.0f);
                if (adv > amax) { amax = adv; best = k; }
                zz[k] = a.beta * adv;
                zmax = fmaxf(zmax, zz[k]);
            }
            float sum = 0.0f;
            for (int k = 0; k < NA; ++k) { zz[k] = expf(zz[k] - zmax); sum += zz[k]; }
            float* po = a.pi_out + ((int64_t)net * B + b) * NA;
            for (int k = 0; k < NA; ++k) po[k] = zz[k] / sum;
            if (a.argmax_out != nullptr) a.argmax_out[(int64_t)net * B + b] = best;
        }
    }
    {
        const float ls = warp_sum(hh == 0 ? lossp : 0.0f);
        const float ds = warp_sum(hh == 0 ? dv : 0.0f);
        if (lane == 0) { sm.lred[0][warp] = ls; sm.lred[1][warp] = ds; }
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int c0 = hh * 64 + cc * 16;
        float g[16], hw[16], gs[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float z = z2[cc * 16 + j];
            g[j] = z > 0.0f ? dv * sm.w3[c0 + j] : 0.0f;
            hw[j] = dv * (z < 0.0f ? 0.0f : z);
            gs[j] = g[j];
        }
        store16<NP>(sm.r1, kPlaneH, HH, row, c0, g);
        const float s3 = colsum16(hw);
        const float s2 = colsum16(gs);
        if ((lane & 1) == 0) {
            sm.red[0][warp][cc * 16 + ((lane >> 1) & 15)] = s3;
            sm.red[1][warp][cc * 16 + ((lane >> 1) & 15)] = s2;
        }
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();
    // ---- G3: dW2 = dz2^T . h1 ----
    if (tid == 0) {
        umma::fence_after_sync();
        gemm<NP>(tmem + TM_DW2, sm.r1, kPlaneH, HH, true, sm.r0, kPlaneH, HH, true, TM / 16, HH);
        umma::commit(&sm.bar_mma);
    }
    // dW3, db2, db3 and the loss partial of the tile (fixed order over warps)
    for (int c = tid; c < HH; c += kThreads) {
        const int h2 = c >> 6, cl = c & 63;
        float s3 = 0.0f, s2 = 0.0f;
        for (int qq = 0; qq < 4; ++qq) { s3 += sm.red[0][h2 * 4 + qq][cl]; s2 += sm.red[1][h2 * 4 + qq][cl]; }
        part[off.w3 + c] = s3;
        part[off.b2 + c] = s2;
    }
    if (tid == 0) {
        float l = 0.0f, d3 = 0.0f;
        for (int w = 0; w < 4; ++w) { l += sm.lred[0][w]; d3 += sm.lred[1][w]; }
        a.tile_loss[(int64_t)net * a.net_tile_stride + tile] = l;
        part[off.b3] = d3;
    }
    wait_mma();
    // ---- stage 3: W2 image -> R0 (h1 is no longer read) ----
    if (tid == 0) {
        umma::mbar_expect_tx(&sm.bar_load, kW2Bytes);
        umma::bulk_g2s(sm.r0, w2i, kW2Bytes, &sm.bar_load);
    }
    wait_load();
    // ---- G4: dh1 = dz2 . W2 ----
    if (tid == 0) {
        umma::fence_after_sync();
        gemm<NP>(tmem + TM_Z1, sm.r1, kPlaneH, HH, false, sm.r0, kPlaneH, HH, true, HH / 16, HH);
        umma::commit(&sm.bar_mma);
    }
    wait_mma();

    // ---- epilogue 4: dz1 = dh1 * 1[z1 > 0] -> R0; db1 ----
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int c0 = hh * 64 + cc * 16;
        float v[16];
        umma::tmem_ld16(tq + TM_Z1 + (uint32_t)c0, v);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = ((mask1 >> (cc * 16 + j)) & 1ull) ? v[j] : 0.0f;
        store16<NP>(sm.r0, kPlaneH, HH, row, c0, v);
        float vs[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) vs[j] = v[j];
        const float s1 = colsum16(vs);
        if ((lane & 1) == 0) sm.red[2][warp][cc * 16 + ((lane >> 1) & 15)] = s1;
    }
    // ---- stage 4: X image -> R1 (dz2 is no longer read) ----
    build_x<NP>(sm.r1, a.states, a.stride, row0, B, S);
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();
    // ---- G5: dW1 = dz1^T . X ----
    if (tid == 0) {
        umma::fence_after_sync();
        gemm<NP>(tmem + TM_DW1, sm.r0, kPlaneH, HH, true, sm.r1, kPlaneX, KX, true, TM / 16, KX);
        umma::commit(&sm.bar_mma);
    }
    for (int c = tid; c < HH; c += kThreads) {
        const int h2 = c >> 6, cl = c & 63;
        float s1 = 0.0f;
        for (int qq = 0; qq < 4; ++qq) s1 += sm.red[2][h2 * 4 + qq][cl];
        part[off.b1 + c] = s1;
    }
    wait_mma();

    // ---- dW2 (lane = output unit, 128 columns) and dW1 (lane = unit, 64 columns) ----
    {
        float* dst = part + off.w2 + (int64_t)row * HH + hh * 64;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            float v[16];
            umma::tmem_ld16(tq + TM_DW2 + (uint32_t)(hh * 64 + cc * 16), v);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(dst + cc * 16 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        float* d1 = part + off.w1 + (int64_t)row * S;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int c0 = hh * 32 + cc * 16;
            float v[16];
            umma::tmem_ld16(tq + TM_DW1 + (uint32_t)c0, v);
            umma::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < S) d1[c0 + j] = v[j];
        }
    }
    if (!ok && tid == 0) atomicAdd(a.status + OFRL_STAT_TIMEOUT, 1);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

// Pack W1 ([H][S] -> [128 x 64] image) and W2 ([H][H] -> [128 x 128] image)
// of every network into NP bf16 planes each, for the tensor-core kernel.
template <int NP>
__global__ void pack_weights_kernel(const VnetLaunch a, uint8_t* __restrict__ img, int64_t img_stride) {
    const int net = blockIdx.y;
    const int S = a.state_dim;
    const Offsets off = offsets_of(S, HH);
    const float* __restrict__ prm = a.params[net];
    uint8_t* w1i = img + (int64_t)net * img_stride;
    uint8_t* w2i = w1i + (uint32_t)NP * kPlaneX;
    const int n1 = HH * KX, n2 = HH * HH;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n1 + n2; e += gridDim.x * blockDim.x) {
        float x;
        uint8_t* base;
        uint32_t plane, o;
        if (e < n1) {
            const int r = e / KX, c = e % KX;
            x = c < S ? __ldg(prm + off.w1 + (int64_t)r * S + c) : 0.0f;
            base = w1i; plane = kPlaneX; o = img_off(r, c, KX);
        } else {
            const int f = e - n1, r = f / HH, c = f % HH;
            x = __ldg(prm + off.w2 + (int64_t)r * HH + c);
            base = w2i; plane = kPlaneH; o = img_off(r, c, HH);
        }
        __nv_bfloat16 t0, t1, t2;
        if (NP == 3) umma::split_bf16x3(x, t0, t1, t2);
        else t0 = __float2bfloat16_rn(x);
        *reinterpret_cast<__nv_bfloat16*>(base + o) = t0;
        if (NP == 3) {
            *reinterpret_cast<__nv_bfloat16*>(base + plane + o) = t1;
            *reinterpret_cast<__nv_bfloat16*>(base + 2 * plane + o) = t2;
        }
    }
}

template <int NP>
cudaError_t launch_np(const VnetLaunch& a, uint8_t* img, int64_t img_stride, cudaStream_t st) {
    pack_weights_kernel<NP><<<dim3(48, a.n_nets), 256, 0, st>>>(a, img, img_stride);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kern = vnet_tc_kernel<NP>;
    const size_t smem = sizeof(TcSmem) + 1024;
    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid((a.batch + TM - 1) / TM, a.n_nets);
    kern<<<grid, kThreads, smem, st>>>(a, img, img, img_stride);
    return cudaGetLastError();
}

}  // namespace

int64_t vnet_tc_image_bytes() { return 3 * (int64_t)(kPlaneX + kPlaneH); }

bool vnet_tc_supported(const VnetLaunch& a) {
    return a.hidden == HH && a.state_dim <= KX && (a.stride & 3) == 0 &&
           (reinterpret_cast<uintptr_t>(a.states) & 15) == 0;
}

cudaError_t launch_vnet_tc(const VnetLaunch& a, uint8_t* img, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    const int64_t stride = vnet_tc_image_bytes();
    return a.prec == OFRL_PREC_BF16 ? launch_np<1>(a, img, stride, st) : launch_np<3>(a, img, stride, st);
}

}  // namespace ofrl
