// IQL value network V(s): forward, expectile loss, advantage-weighted
// policy and backward for one tile of batch rows per CTA, on CUDA cores.
//
// Method: "GPU IQL + HER Porting Plan", "IQL (CPU)" items 1-3 and "CUDA
// Kernel: iql_value_kernel.cu" (V forward, Q(s, a_taken) target, expectile
// loss, backward into a flat gradient).  The pages run one warp per sample
// and accumulate the loss and the gradient with float atomics; here a CTA
// owns TM rows, keeps every activation of its tile in shared memory, stages
// the weights through shared memory in 32-row chunks, and writes one
// gradient partial per tile (no atomics) that a separate pass reduces in a
// fixed order.  Loss partials are likewise per tile.
//
// Thread layout (256 threads = 8 warps): thread (ty, tx) owns rows
// ty + 8 i (i < TM / 8) and columns tx + 32 j (j < H / 32) of every
// [TM, H] activation, so a warp holds whole columns for eight-row strides and
// each row's V is a warp sum.

#include "common.cuh"

namespace ofrl {
namespace {

constexpr int kThreads = 256;
constexpr int kXStride = 64;      // shared-memory row stride of the state tile (S <= 64)
constexpr int kKChunk = 32;       // weight rows staged per chunk

template <int H>
struct TileRows { static constexpr int value = H <= 128 ? 128 : 64; };

template <int H, int TM>
constexpr size_t smem_floats() {
    return (size_t)TM * kXStride + 2 * (size_t)TM * H + 2 * 8 * (size_t)H + (size_t)kKChunk * (H + 1);
}

template <bool BF16>
__device__ __forceinline__ float op(float x) { return BF16 ? to_bf16_rn(x) : x; }

// Stage kKChunk rows k0.. of the GEMM's right operand into wt[kk][c]
// (row stride H + 1).  TRANS: W is [H][K] row-major and we need W[c][k0+kk];
// otherwise W is [K][H] row-major and we need W[k0+kk][c].  Rows at or past
// K are zero.
template <int H, bool TRANS, bool BF16>
__device__ __forceinline__ void stage_weights(float* wt, const float* __restrict__ w, int K, int k0) {
    for (int e = threadIdx.x; e < kKChunk * H; e += kThreads) {
        int kk, c;
        if (TRANS) { c = e / kKChunk; kk = e % kKChunk; } else { kk = e / H; c = e % H; }
        const int k = k0 + kk;
        float x = 0.0f;
        if (k < K) x = TRANS ? __ldg(w + (int64_t)c * K + k) : __ldg(w + (int64_t)k * H + c);
        wt[kk * (H + 1) + c] = op<BF16>(x);
    }
}

// acc[i][j] += sum_k As[(ty + 8 i) * lda + k] * W(k, tx + 32 j) for k < K
// (K rounded up to 4; As must hold zeros there).
template <int H, int TM, bool TRANS, bool BF16>
__device__ __forceinline__ void gemm_rows(float (&acc)[TM / 8][H / 32], const float* As, int lda,
                                          const float* __restrict__ w, int K, float* wt) {
    constexpr int RPT = TM / 8, CPT = H / 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int k0 = 0; k0 < K; k0 += kKChunk) {
        __syncthreads();
        stage_weights<H, TRANS, BF16>(wt, w, K, k0);
        __syncthreads();
        const int kn = min(kKChunk, (K - k0 + 3) & ~3);
#pragma unroll 1
        for (int kk = 0; kk < kn; kk += 4) {
            float wv[4][CPT];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < CPT; ++j) wv[u][j] = wt[(kk + u) * (H + 1) + tx + 32 * j];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const float4 x = *reinterpret_cast<const float4*>(As + (ty + 8 * i) * lda + k0 + kk);
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    acc[i][j] = fmaf(x.x, wv[0][j], acc[i][j]);
                    acc[i][j] = fmaf(x.y, wv[1][j], acc[i][j]);
                    acc[i][j] = fmaf(x.z, wv[2][j], acc[i][j]);
                    acc[i][j] = fmaf(x.w, wv[3][j], acc[i][j]);
                }
            }
        }
    }
}

// out[i][j] = sum_r A[r][i] * Bm[r][j] over the TM tile rows, i < NI, j < NJ,
// written to dst[i * ldd + j].  A has row stride lda, Bm row stride ldb.
template <int TM>
__device__ __forceinline__ void gemm_tn_store(const float* A, int lda, int NI, const float* Bm, int ldb,
                                              int NJ, float* __restrict__ dst, int ldd) {
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int ib = 0; ib < NI; ib += 64) {
        for (int jb = 0; jb < NJ; jb += 64) {
            float acc[8][2];
#pragma unroll
            for (int a = 0; a < 8; ++a) { acc[a][0] = 0.0f; acc[a][1] = 0.0f; }
            const int i0 = ib + ty * 8;
            const int j0 = jb + tx, j1 = jb + tx + 32;
            const bool ok0 = j0 < NJ, ok1 = j1 < NJ;
#pragma unroll 2
            for (int r = 0; r < TM; ++r) {
                const float4 a0 = *reinterpret_cast<const float4*>(A + r * lda + i0);
                const float4 a1 = *reinterpret_cast<const float4*>(A + r * lda + i0 + 4);
                const float b0 = ok0 ? Bm[r * ldb + j0] : 0.0f;
                const float b1 = ok1 ? Bm[r * ldb + j1] : 0.0f;
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    acc[a][0] = fmaf(av[a], b0, acc[a][0]);
                    acc[a][1] = fmaf(av[a], b1, acc[a][1]);
                }
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                if (i0 + a < NI) {
                    if (ok0) dst[(int64_t)(i0 + a) * ldd + j0] = acc[a][0];
                    if (ok1) dst[(int64_t)(i0 + a) * ldd + j1] = acc[a][1];
                }
            }
        }
    }
}

// The forward part shared by the training and the forward-only kernels: the
// state tile into Xs (zero rows past the batch, zero columns past S), h1 =
// relu(X W1^T + b1) into h1s, and z2 = h1 W2^T + b2 left in acc.
template <int H, bool BF16>
__device__ __forceinline__ void forward_tile(const VnetLaunch& a, float* Xs, float* h1s, float* wt,
                                             float (&acc)[TileRows<H>::value / 8][H / 32]) {
    constexpr int TM = TileRows<H>::value;
    constexpr int RPT = TM / 8, CPT = H / 32;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int tile = blockIdx.x, net = blockIdx.y;
    const int S = a.state_dim, B = a.batch;
    const Offsets off = offsets_of(S, H);
    const float* __restrict__ prm = a.params[net];
    const int row0 = tile * TM;

    for (int e = tid; e < TM * kXStride; e += kThreads) {
        const int r = e / kXStride, k = e % kXStride;
        float x = 0.0f;
        if (k < S && row0 + r < B) x = __ldg(a.states + (int64_t)(row0 + r) * a.stride + k);
        Xs[e] = op<BF16>(x);
    }
    // ---- layer 1: z1 = X W1^T + b1, h1 = relu(z1) ----
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const float bj = __ldg(prm + off.b1 + tx + 32 * j);
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[i][j] = bj;
    }
    gemm_rows<H, TM, true, BF16>(acc, Xs, kXStride, prm + off.w1, S, wt);
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const float z = acc[i][j];
            h1s[(ty + 8 * i) * H + tx + 32 * j] = op<BF16>(z < 0.0f ? 0.0f : z);
        }
    // ---- layer 2: z2 = h1 W2^T + b2 ----
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const float bj = __ldg(prm + off.b2 + tx + 32 * j);
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[i][j] = bj;
    }
    gemm_rows<H, TM, true, BF16>(acc, h1s, H, prm + off.w2, H, wt);
}

// V forward only ("GPU IQL + HER Porting Plan", forward_values, and "IQL
// modifies the target computation"): V of every row into v_out and, with
// target_out, the IQL bootstrap target r + gamma (1 - done) V.
template <int H, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) vnet_forward_kernel(const VnetLaunch a) {
    constexpr int TM = TileRows<H>::value;
    constexpr int RPT = TM / 8, CPT = H / 32;
    extern __shared__ float4 smem4[];
    float* Xs = reinterpret_cast<float*>(smem4);   // [TM][kXStride]
    float* h1s = Xs + TM * kXStride;               // [TM][H]
    float* wt = h1s + 2 * TM * H + 2 * 8 * H;      // [kKChunk][H + 1] (same layout as the training kernel)
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int net = blockIdx.y, B = a.batch;
    const Offsets off = offsets_of(a.state_dim, H);
    const float* __restrict__ prm = a.params[net];
    const int row0 = blockIdx.x * TM;
    pdl_trigger();
    pdl_wait();
    float acc[RPT][CPT];
    forward_tile<H, BF16>(a, Xs, h1s, wt, acc);
    float w3[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) w3[j] = __ldg(prm + off.w3 + tx + 32 * j);
    const float b3 = __ldg(prm + off.b3);
    float vrow[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const float h = acc[i][j] < 0.0f ? 0.0f : acc[i][j];
            s = fmaf(h, w3[j], s);
        }
        vrow[i] = warp_sum(s) + b3;
    }
    if (tx < RPT) {
        float myv = 0.0f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) if (tx == i) myv = vrow[i];
        const int b = row0 + ty + 8 * tx;
        if (b < B) {
            if (a.v_out != nullptr) a.v_out[(int64_t)net * B + b] = myv;
            if (a.target_out != nullptr)
                a.target_out[(int64_t)net * B + b] = __ldg(a.rewards + b) + a.gamma * (1.0f - __ldg(a.dones + b)) * myv;
        }
    }
}

template <int H, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) vnet_fwd_bwd_kernel(const VnetLaunch a) {
    constexpr int TM = TileRows<H>::value;
    constexpr int RPT = TM / 8, CPT = H / 32;
    extern __shared__ float4 smem4[];
    float* Xs = reinterpret_cast<float*>(smem4);   // [TM][kXStride]
    float* h1s = Xs + TM * kXStride;               // [TM][H]: h1, later dz1
    float* a2s = h1s + TM * H;                     // [TM][H]: dz2
    float* red = a2s + TM * H;                     // [2][8][H]
    float* wt = red + 2 * 8 * H;                   // [kKChunk][H + 1]
    __shared__ float lred[2][8];

    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int tile = blockIdx.x, net = blockIdx.y;
    const int S = a.state_dim, B = a.batch, NA = a.num_actions;
    const Offsets off = offsets_of(S, H);
    const float* __restrict__ prm = a.params[net];
    const float tau = a.tau[net];
    const int row0 = tile * TM;
    float* part = a.partials + (int64_t)net * a.net_partial_stride + (int64_t)tile * a.part_stride;
    pdl_trigger();
    pdl_wait();

    float acc[RPT][CPT];
    forward_tile<H, BF16>(a, Xs, h1s, wt, acc);

    // ---- head: V = h2 w3 + b3, loss, dV, policy, dz2, dW3, db2, db3 ----
    float w3[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) w3[j] = __ldg(prm + off.w3 + tx + 32 * j);
    const float b3 = __ldg(prm + off.b3);
    float vrow[RPT], dv[RPT];
    float loss_part = 0.0f, db3_part = 0.0f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const float h = acc[i][j] < 0.0f ? 0.0f : acc[i][j];
            s = fmaf(h, w3[j], s);
        }
        vrow[i] = warp_sum(s) + b3;
        const int b = row0 + ty + 8 * i;
        dv[i] = 0.0f;
        if (b < B) {
            float q;
            if (a.q != nullptr) {
                int act = __ldg(a.actions + b);
                if (act < 0 || act >= NA) {
                    if (tx == 0) atomicAdd(a.status + OFRL_STAT_BAD_ACTION, 1);
                    act = 0;
                }
                q = __ldg(a.q + (int64_t)b * NA + act);
            } else {
                q = __ldg(a.q_taken + b);
            }
            const float d = q - vrow[i];
            const float w = d >= 0.0f ? tau : 1.0f - tau;
            loss_part += w * d * d;
            dv[i] = (-2.0f * w * d) / (float)B;
            db3_part += dv[i];
        }
    }
    // outputs for the rows of this warp
    if (a.v_out != nullptr && tx < RPT) {
        float myv = 0.0f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) if (tx == i) myv = vrow[i];
        const int b = row0 + ty + 8 * tx;
        if (b < B) a.v_out[(int64_t)net * B + b] = myv;
    }
    if (a.pi_out != nullptr && tx < RPT) {
        float myv = 0.0f;
#pragma unroll
        for (int i = 0; i < RPT; ++i) if (tx == i) myv = vrow[i];
        const int b = row0 + ty + 8 * tx;
        if (b < B) {
            // three passes over the row of Q (no local array): max / argmax,
            // sum of exponentials, outputs
            const float* qr = a.q + (int64_t)b * NA;
            float zmax = -INFINITY;
            int best = 0;
            float amax = -INFINITY;
            for (int k = 0; k < NA; ++k) {
                const float adv = fminf(fmaxf(__ldg(qr + k) - myv, -10.0f), 10.0f);
                if (adv > amax) { amax = adv; best = k; }
                zmax = fmaxf(zmax, a.beta * adv);
            }
            float sum = 0.0f;
            for (int k = 0; k < NA; ++k) sum += expf(a.beta * fminf(fmaxf(__ldg(qr + k) - myv, -10.0f), 10.0f) - zmax);
            float* po = a.pi_out + ((int64_t)net * B + b) * NA;
            for (int k = 0; k < NA; ++k)
                po[k] = expf(a.beta * fminf(fmaxf(__ldg(qr + k) - myv, -10.0f), 10.0f) - zmax) / sum;
            if (a.argmax_out != nullptr) a.argmax_out[(int64_t)net * B + b] = best;
        }
    }
    // dz2 = dV w3 * 1[z2 > 0] into a2s; per-thread dW3 and db2 partials
    float dw3p[CPT], db2p[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) { dw3p[j] = 0.0f; db2p[j] = 0.0f; }
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const float z = acc[i][j];
            const float h = z < 0.0f ? 0.0f : z;
            const float g = z > 0.0f ? dv[i] * w3[j] : 0.0f;
            dw3p[j] = fmaf(dv[i], h, dw3p[j]);
            db2p[j] += g;
            a2s[(ty + 8 * i) * H + tx + 32 * j] = op<BF16>(g);
        }
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        red[(0 * 8 + ty) * H + tx + 32 * j] = dw3p[j];
        red[(1 * 8 + ty) * H + tx + 32 * j] = db2p[j];
    }
    if (tx == 0) { lred[0][ty] = loss_part; lred[1][ty] = db3_part; }
    __syncthreads();
    for (int c = tid; c < H; c += kThreads) {
        float s0 = 0.0f, s1 = 0.0f;
        for (int y = 0; y < 8; ++y) { s0 += red[(0 * 8 + y) * H + c]; s1 += red[(1 * 8 + y) * H + c]; }
        part[off.w3 + c] = s0;
        part[off.b2 + c] = s1;
    }
    if (tid == 0) {
        float s0 = 0.0f, s1 = 0.0f;
        for (int y = 0; y < 8; ++y) { s0 += lred[0][y]; s1 += lred[1][y]; }
        a.tile_loss[(int64_t)net * a.net_tile_stride + tile] = s0;
        part[off.b3] = s1;
    }

    // ---- dW2 = dz2^T h1 ----
    gemm_tn_store<TM>(a2s, H, H, h1s, H, H, part + off.w2, H);
    __syncthreads();

    // ---- dh1 = dz2 W2, dz1 = dh1 * 1[z1 > 0] (into h1s), db1 ----
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[i][j] = 0.0f;
    gemm_rows<H, TM, false, BF16>(acc, a2s, H, prm + off.w2, H, wt);
    float db1p[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) db1p[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < RPT; ++i)
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            float* hp = h1s + (ty + 8 * i) * H + tx + 32 * j;
            const float g = *hp > 0.0f ? acc[i][j] : 0.0f;
            db1p[j] += g;
            *hp = op<BF16>(g);
        }
#pragma unroll
    for (int j = 0; j < CPT; ++j) red[(0 * 8 + ty) * H + tx + 32 * j] = db1p[j];
    __syncthreads();
    for (int c = tid; c < H; c += kThreads) {
        float s0 = 0.0f;
        for (int y = 0; y < 8; ++y) s0 += red[(0 * 8 + y) * H + c];
        part[off.b1 + c] = s0;
    }

    // ---- dW1 = dz1^T X ----
    gemm_tn_store<TM>(h1s, H, H, Xs, kXStride, S, part + off.w1, S);
}

template <int H, bool BF16, bool FWD = false>
cudaError_t launch_h(const VnetLaunch& a, cudaStream_t st) {
    constexpr int TM = TileRows<H>::value;
    const size_t smem = smem_floats<H, TM>() * sizeof(float);
    auto kern = FWD ? vnet_forward_kernel<H, BF16> : vnet_fwd_bwd_kernel<H, BF16>;
    static bool configured = false;   // per instantiation; setting it twice is harmless
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid((a.batch + TM - 1) / TM, a.n_nets);
    return launch_pdl(kern, grid, dim3(kThreads), smem, st, a);
}

}  // namespace

int vnet_tile_rows(int hidden) { return hidden <= 128 ? 128 : 64; }

cudaError_t launch_vnet_fwd_bwd(const VnetLaunch& a, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    const bool bf = a.prec == OFRL_PREC_BF16;
    switch (a.hidden) {
        case 64: return bf ? launch_h<64, true>(a, st) : launch_h<64, false>(a, st);
        case 128: return bf ? launch_h<128, true>(a, st) : launch_h<128, false>(a, st);
        case 256: return bf ? launch_h<256, true>(a, st) : launch_h<256, false>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_vnet_forward(const VnetLaunch& a, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    const bool bf = a.prec == OFRL_PREC_BF16;
    switch (a.hidden) {
        case 64: return bf ? launch_h<64, true, true>(a, st) : launch_h<64, false, true>(a, st);
        case 128: return bf ? launch_h<128, true, true>(a, st) : launch_h<128, false, true>(a, st);
        case 256: return bf ? launch_h<256, true, true>(a, st) : launch_h<256, false, true>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ofrl
