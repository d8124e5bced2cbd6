// Gradient reduction, per-source norms, budgeted clipped SAXPY and Adam.
//
// Method: "Gradient Stability -- Multi-Task Gradient Isolation + Full
// Spectral Norm", "Proper design" (each source clipped to its budget
// fraction of max_grad_norm, then added; Adam's own clip at max_grad_norm)
// and Task 1 Step 5 (norm of the source first, then the clipped SAXPY);
// "DQN Backward-Path NaN Audit", Adam kernel findings (norm kept as a raw sum
// of squares and square-rooted where used, the (n > c && n > 0) ? c / n : 1
// clip, non-finite elements skipped, bias correction with t >= 1).
//
// The pages run one norm kernel and one SAXPY kernel per source and a
// separate Adam launch, each a full pass over the parameters.  Here one pass
// (reduce_gram) sums the per-tile gradient partials into the primary
// gradient and accumulates the Gram matrix <g_j, g_k> of all sources; its
// last block turns the Gram matrix into the source norms, the clip
// coefficients and the norm of the combined gradient
// ||sum_k c_k g_k||^2 = sum_jk c_j c_k <g_j, g_k>.  A second pass (adam)
// forms the combined gradient element by element and applies Adam, so the
// combined gradient is never stored.  Every reduction is in a fixed order.

#include <cstring>

#include "common.cuh"
#include "step_math.cuh"

namespace ofrl {
namespace {

// A reduce block is EL element lanes (a float4 each) x 256 / EL partial
// lanes, each with eight loads in flight: EL = 32 (8 partial lanes), or for
// many partials EL = 64 when only that grid covers P in one resident pass
// (the reduce and Adam then run as one launch), else EL = 8 (32 partial
// lanes, two launches).
constexpr int kRedThreads = 256;
constexpr int kManyParts = 64;     // more partials than this: EL = 32 or 64 (fused), else 8
constexpr int kRedUnroll = 8;      // partial loads in flight per thread

__device__ __forceinline__ void add4(float4& s, const float4& v) {
    s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
}

// 16-byte load of a gradient partial, read once: evict_first in L2.
__device__ __forceinline__ float4 ld_last(const float* p) {
    float4 v;
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

// Sum of the partials of element group i4..i4+3 over partials ty, ty + TL,
// ... in that order, U independent 16-byte loads in flight at a time.
template <int TL, int U>
__device__ __forceinline__ float4 sum_tiles(const float* __restrict__ pp, int64_t stride, int n_parts, int ty,
                                            int64_t i4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = ty; t < n_parts; t += U * TL) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = t + u * TL < n_parts ? ld_last(pp + (int64_t)(t + u * TL) * stride + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < U; ++u) add4(acc, v[u]);
    }
    return acc;
}

// (j, k) of Gram entry p (gram_index order)
__device__ __forceinline__ int pair_j(int p) { return p < 4 ? 0 : p < 7 ? 1 : p < 9 ? 2 : 3; }
__device__ __forceinline__ int pair_k(int p) {
    return p < 4 ? p : p < 7 ? p - 3 : p < 9 ? p - 5 : 3;
}

// The tail of the fused reduce + Adam launch (see below).
template <int EL>
__device__ __forceinline__ void fused_norms_adam(const ReduceLaunch& a, const AdamLaunch& d, unsigned long long* bar,
                                                 unsigned long long bar_target, const float (&gacc)[kGramPairs],
                                                 const float (&x)[kMaxSrc][4], float4* scratch) {
    constexpr int kRedElems = 4 * EL;
    const int tid = threadIdx.x, tx = tid % EL, ty = tid / EL, lane = tid & 31, wid = tid >> 5;
    const int net = blockIdx.y, G = gridDim.x, nsrc = a.n_src;
    const int64_t P = a.P;
    // Adam runs one element per thread (threads 0 .. 4 EL - 1): this
    // thread's weight, moments and target, read before the barrier (only
    // this block writes them)
    const int64_t ie = (int64_t)blockIdx.x * kRedElems + tid;
    const bool has_e = tid < kRedElems && ie < P;
    float pe = 0.0f, me = 0.0f, ve = 0.0f, te = 0.0f;
    if (has_e) {
        pe = d.p[net][ie];
        me = d.m[net][ie];
        ve = d.v[net][ie];
        if (d.target[net] != nullptr) te = d.target[net][ie];
    }
    float* gp = a.gram_part + ((int64_t)net * G + blockIdx.x) * kGramStride;
    if constexpr (EL <= 32) {
        // the element lanes are lanes 0..EL-1 of warp 0
        if (wid == 0) {
#pragma unroll
            for (int p = 0; p < kGramPairs; ++p) {
                if (pair_j(p) >= nsrc || pair_k(p) >= nsrc) continue;
                const float s = warp_sum(gacc[p]);
                if (lane == 0) gp[p] = s;
            }
        }
    } else {
        // the element lanes fill warps 0..EL/32-1: per-warp sums, then in warp order
        __shared__ float gw[EL / 32][kGramPairs];
        if (wid < EL / 32) {
#pragma unroll
            for (int p = 0; p < kGramPairs; ++p) {
                const float s = warp_sum(gacc[p]);
                if (lane == 0) gw[wid][p] = s;
            }
        }
        __syncthreads();
        if (tid < kGramPairs && pair_j(tid) < nsrc && pair_k(tid) < nsrc) {
            float s = gw[0][tid];
#pragma unroll
            for (int w = 1; w < EL / 32; ++w) s += gw[w][tid];
            gp[tid] = s;
        }
    }
    // A CTA that gave up waiting cannot know the other CTAs' Gram partials:
    // it writes nothing more (no norms, no p / m / v / target) and only
    // counts the timeout.  ok is the same for every thread of the CTA.
    if (!grid_barrier(bar, bar_target, d.wait_ns)) {
        if (tid == 0) atomicAdd(d.status + OFRL_STAT_TIMEOUT, 1);
        return;
    }

    // totals of the Gram entries present and of the loss, in the same fixed
    // order in every block.  Every block reads all G Gram partials.  With one
    // source: a warp per entry, lanes stride the blocks.  With several, the
    // entries are read with contiguous 16-byte loads instead (thread t takes
    // quad t % 4 of partials t / 4, t / 4 + 64, ...; strided 4-byte loads of
    // the same few lines by every block queue at their L2 slices), lanes of
    // equal quad combined by shuffles, the warps in order through `scratch`
    // (the reduce's staging, free by now; no shared memory is added, so a
    // block still fits beside a tensor-core V CTA).
    __shared__ float totals[kGramPairs + 1];
    if (nsrc <= 1) {
        const float* gall = a.gram_part + (int64_t)net * G * kGramStride;
        for (int item = wid; item <= kGramPairs; item += kRedThreads / 32) {
            const bool need = item == kGramPairs ? a.tile_loss != nullptr
                                                 : pair_j(item) < nsrc && pair_k(item) < nsrc;
            float v = 0.0f;
            if (need) {
                const int n = item == kGramPairs ? a.n_tiles : G;
                for (int b0 = lane; b0 < n; b0 += 8 * 32) {
                    float u[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int b = b0 + 32 * r;
                        u[r] = b >= n ? 0.0f
                                      : item == kGramPairs ? __ldcg(a.tile_loss + (int64_t)net * a.net_tile_stride + b)
                                                           : __ldcg(gall + (int64_t)b * kGramStride + item);
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) v += u[r];
                }
                v = warp_sum(v);
            }
            if (lane == 0) totals[item] = v;
        }
    } else {
        float4* wq = scratch;                                           // [warps][4]
        float* wl = reinterpret_cast<float*>(scratch + 4 * (kRedThreads / 32));   // [warps]
        const float4* g4 = reinterpret_cast<const float4*>(a.gram_part + (int64_t)net * G * kGramStride);
        const int quad = tid & 3;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (quad < (kGramPairs + 3) / 4) {
#pragma unroll 4
            for (int b = tid >> 2; b < G; b += kRedThreads / 4)
                add4(s, __ldcg(g4 + (int64_t)b * (kGramStride / 4) + quad));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
            s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
            s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
            s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
        }
        if (lane < 4) wq[wid * 4 + lane] = s;
        float l = 0.0f;
        if (a.tile_loss != nullptr)
            for (int t = tid; t < a.n_tiles; t += kRedThreads) l += __ldcg(a.tile_loss + (int64_t)net * a.net_tile_stride + t);
        l = warp_sum(l);
        if (lane == 0) wl[wid] = l;
        __syncthreads();
        if (tid <= kGramPairs) {
            float v = 0.0f;
            for (int w = 0; w < kRedThreads / 32; ++w) {
                if (tid == kGramPairs) {
                    v += wl[w];
                } else {
                    const float4 q4 = wq[w * 4 + (tid >> 2)];
                    const int c = tid & 3;
                    v += c == 0 ? q4.x : c == 1 ? q4.y : c == 2 ? q4.z : q4.w;
                }
            }
            totals[tid] = v;
        }
    }
    __syncthreads();
    float gram[kGramPairs];
#pragma unroll
    for (int p = 0; p < kGramPairs; ++p) gram[p] = totals[p];
    const NormResult r = finish_norms(gram, totals[kGramPairs], nsrc, a.budget, a.alpha, a.max_grad_norm, a.inv_batch);
    if (blockIdx.x == 0 && tid == 0) {
        float* sc = a.scalars + (int64_t)net * kScalars;
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k) {
            sc[SC_NORM0 + k] = r.nrm[k];
            sc[SC_COEF0 + k] = r.coef[k];
        }
        sc[SC_COMBINED] = r.combined;
        sc[SC_LOSS] = r.loss;
        if (a.norms_out != nullptr) {
#pragma unroll
            for (int k = 0; k < kMaxSrc; ++k) a.norms_out[net * 5 + k] = r.nrm[k];
            a.norms_out[net * 5 + 4] = r.combined;
        }
        if (a.loss_out != nullptr) a.loss_out[net] = r.loss;
    }

    // the clipped combination and Adam, one element per thread: the element
    // lanes hand their sources (already guarded when sanitize is on) over
    // through `scratch` (free since the totals; it holds kMaxSrc x 4 EL floats)
    float* xs = reinterpret_cast<float*>(scratch);
    if (ty == 0) {
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k)
            if (k < nsrc) {
#pragma unroll
                for (int e = 0; e < 4; ++e) xs[k * kRedElems + 4 * tx + e] = x[k][e];
            }
    }
    __syncthreads();
    int bad = 0;
    if (has_e) {
        const float s = clip_scale(r.combined, d.max_grad_norm);
        float gsum = 0.0f;
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k)
            if (k < nsrc) gsum = fmaf(r.coef[k], xs[k * kRedElems + tid], gsum);
        const float g = s * gsum;
        float p = pe, m = me, v = ve;
        if (adam_element(p, m, v, g, d.beta1, d.beta2, d.eps, d.weight_decay, d.lr[net], d.bc1[net], d.bc2[net])) {
            if (d.clamp > 0.0f) p = fminf(fmaxf(p, -d.clamp), d.clamp);
            d.m[net][ie] = m;
            d.v[net][ie] = v;
            d.p[net][ie] = p;
        } else {
            bad = 1;
        }
        if (d.target[net] != nullptr) {
            const float pk = d.polyak[net];
            d.target[net][ie] = (1.0f - pk) * te + pk * p;
        }
    }
    bad = __syncthreads_count(bad);
    if (bad && tid == 0) atomicAdd(d.status + OFRL_STAT_NONFINITE_GRAD, bad);
}

// ADAM: one cooperative launch does the reduce and Adam.  One pass of the
// grid covers P; after the block's Gram partial a grid barrier; then every
// block forms the totals, norms and coefficients in the same fixed order and
// applies the clipped combination and Adam to its own elements, which its
// element lanes still hold.
template <int EL, bool ADAM>
__global__ void __launch_bounds__(kRedThreads, ADAM ? 3 : 4)
    reduce_gram_kernel(const ReduceLaunch a, const AdamLaunch d, unsigned long long* bar,
                       unsigned long long bar_target) {
    constexpr int TL = kRedThreads / EL, kRedElems = 4 * EL;
    __shared__ float4 sh[TL][EL + 1];
    __shared__ unsigned int ticket;
    const int tid = threadIdx.x, tx = tid % EL, ty = tid / EL;
    const int n_parts = a.n_parts > 0 ? a.n_parts : a.n_tiles;
    const int lane = tid & 31, wid = tid >> 5;
    const int net = blockIdx.y;
    const int64_t P = a.P;
    const int nsrc = a.n_src;
    // dependents launch only once everything before this kernel (the V
    // kernel reading the batch) has completed: the next step's relabel rows
    // may then overwrite the batch without waiting for this kernel
    pdl_wait();
    pdl_trigger();

    float gacc[kGramPairs];
#pragma unroll
    for (int p = 0; p < kGramPairs; ++p) gacc[p] = 0.0f;
    float x[kMaxSrc][4];   // (after the loop: this lane's elements, for the fused Adam)

    for (int64_t base = (int64_t)blockIdx.x * kRedElems; base < P; base += (int64_t)gridDim.x * kRedElems) {
        const int64_t i4 = base + 4 * tx;
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[k][e] = 0.0f;
        if (a.partials != nullptr) {
            // partial rows are padded to a multiple of 32 floats: the float4 at
            // i4 < P stays inside the tile's slice
            const float* pp = a.partials + (int64_t)net * a.net_partial_stride;
            sh[ty][tx] = i4 < P ? sum_tiles<TL, kRedUnroll>(pp, a.part_stride, n_parts, ty, i4)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            __syncthreads();
            if (ty == 0) {
                float g[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int y = 0; y < TL; ++y) {
                    const float4 v = sh[y][tx];
                    g[0] += v.x; g[1] += v.y; g[2] += v.z; g[3] += v.w;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (i4 + e < P) {
                        a.g0_out[net][i4 + e] = g[e];
                        x[0][e] = g[e];
                    }
                }
            }
            __syncthreads();
        } else if (ty == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (i4 + e < P) x[0][e] = __ldg(a.src[net][0] + i4 + e);
        }
        if (ty == 0 && nsrc > 0) {
#pragma unroll
            for (int k = 1; k < kMaxSrc; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (k < nsrc && i4 + e < P) x[k][e] = __ldg(a.src[net][k] + i4 + e);
            if (a.sanitize) {
                int bad = 0;
#pragma unroll
                for (int k = 0; k < kMaxSrc; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (!isfinite(x[k][e])) { x[k][e] = 0.0f; ++bad; }
                if (bad) atomicAdd(a.status + OFRL_STAT_SANITIZED, bad);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int j = 0; j < kMaxSrc; ++j)
#pragma unroll
                    for (int k = j; k < kMaxSrc; ++k)
                        gacc[gram_index(j, k)] = fmaf(x[j][e], x[k][e], gacc[gram_index(j, k)]);
        }
    }
    if constexpr (ADAM) {
        fused_norms_adam<EL>(a, d, bar, bar_target, gacc, x, &sh[0][0]);
        return;
    }
    float* gp = a.gram_part + ((int64_t)net * gridDim.x + blockIdx.x) * kGramStride;
    // the element lanes (ty == 0) are threads 0..EL-1; the rest hold zeros.
    // Thread 0 writes the block's Gram partial and alone fences before taking
    // a ticket: the last block reads nothing else written in this launch.
    if constexpr (EL <= 32) {
        if (wid == 0) {
#pragma unroll
            for (int p = 0; p < kGramPairs; ++p) {
                const float s = warp_sum(gacc[p]);
                if (lane == 0) gp[p] = s;
            }
            if (lane == 0) {
                __threadfence();
                ticket = atomicAdd(a.counter + net, 1u);
            }
        }
    } else {
        // element lanes in warps 0..EL/32-1: per-warp sums, then in warp order
        __shared__ float gw[EL / 32][kGramPairs];
        if (wid < EL / 32) {
#pragma unroll
            for (int p = 0; p < kGramPairs; ++p) {
                const float s = warp_sum(gacc[p]);
                if (lane == 0) gw[wid][p] = s;
            }
        }
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int p = 0; p < kGramPairs; ++p) {
                float s = gw[0][p];
#pragma unroll
                for (int w = 1; w < EL / 32; ++w) s += gw[w][p];
                gp[p] = s;
            }
            __threadfence();
            ticket = atomicAdd(a.counter + net, 1u);
        }
    }
    __syncthreads();
    if (ticket != gridDim.x - 1) return;

    // ---- last block: fixed-order totals, norms, clip coefficients ----
    // Every thread loads all ten Gram partials (and the loss partials) of its
    // blocks at once, so the block pays one round of L2 latency, then one
    // fixed-order tree over the block.  fp32 throughout: FP64 on this part is
    // a small fraction of the fp32 rate and a chain of dependent FP64
    // operations on one thread costs microseconds.
    __threadfence();
    float acc[kGramPairs + 1];
#pragma unroll
    for (int p = 0; p <= kGramPairs; ++p) acc[p] = 0.0f;
    const float* gall = a.gram_part + (int64_t)net * gridDim.x * kGramStride;
    for (int b = tid; b < (int)gridDim.x; b += kRedThreads) {
        float v[kGramPairs];
#pragma unroll
        for (int p = 0; p < kGramPairs; ++p) v[p] = __ldcg(gall + (int64_t)b * kGramStride + p);
#pragma unroll
        for (int p = 0; p < kGramPairs; ++p) acc[p] += v[p];
    }
    if (a.tile_loss != nullptr) {
        const float* tl = a.tile_loss + (int64_t)net * a.net_tile_stride;
        for (int t = tid; t < a.n_tiles; t += kRedThreads) acc[kGramPairs] += __ldcg(tl + t);
    }
    __shared__ float tot[kGramPairs + 1][kRedThreads / 32];
#pragma unroll
    for (int p = 0; p <= kGramPairs; ++p) {
        const float s = warp_sum(acc[p]);
        if (lane == 0) tot[p][wid] = s;
    }
    __syncthreads();
    __shared__ float totals[kGramPairs + 1];
    if (tid <= kGramPairs) {
        float s = 0.0f;
        for (int y = 0; y < kRedThreads / 32; ++y) s += tot[tid][y];
        totals[tid] = s;
    }
    __syncthreads();
    if (tid == 0) {
        float gram[kGramPairs];
#pragma unroll
        for (int p = 0; p < kGramPairs; ++p) gram[p] = totals[p];
        const NormResult r = finish_norms(gram, totals[kGramPairs], nsrc, a.budget, a.alpha, a.max_grad_norm,
                                          a.inv_batch);
        float* sc = a.scalars + (int64_t)net * kScalars;
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k) {
            sc[SC_NORM0 + k] = r.nrm[k];
            sc[SC_COEF0 + k] = r.coef[k];
        }
        sc[SC_COMBINED] = r.combined;
        sc[SC_LOSS] = r.loss;
        const float lmean = r.loss;
        if (a.norms_out != nullptr) {
#pragma unroll
            for (int k = 0; k < kMaxSrc; ++k) a.norms_out[net * 5 + k] = r.nrm[k];
            a.norms_out[net * 5 + 4] = r.combined;
        }
        if (a.loss_out != nullptr) a.loss_out[net] = lmean;
        a.counter[net] = 0u;
    }
}

__global__ void __launch_bounds__(256) adam_kernel(const AdamLaunch a) {
    pdl_wait();      // then dependents (as in reduce_gram_kernel)
    pdl_trigger();
    const int net = blockIdx.y;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    float coef[kMaxSrc] = {1.0f, 0.0f, 0.0f, 0.0f};
    float gn;
    if (a.scalars != nullptr) {
        const float* sc = a.scalars + (int64_t)net * kScalars;
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k) coef[k] = sc[SC_COEF0 + k];
        gn = a.grad_norm != nullptr ? __ldg(a.grad_norm) : sc[SC_COMBINED];
    } else {
        gn = __ldg(a.grad_norm);
    }
    const float s = clip_scale(gn, a.max_grad_norm);
    bool bad = false;
    if (i < a.n) {
        float gsum = 0.0f;
        for (int k = 0; k < a.n_src; ++k) {
            float x = __ldg(a.src[net][k] + i);
            if (a.sanitize && !isfinite(x)) x = 0.0f;
            gsum = fmaf(coef[k], x, gsum);
        }
        const float g = s * gsum;
        float m = a.m[net][i], v = a.v[net][i], p = a.p[net][i];
        if (adam_element(p, m, v, g, a.beta1, a.beta2, a.eps, a.weight_decay, a.lr[net], a.bc1[net], a.bc2[net])) {
            if (a.clamp > 0.0f) p = fminf(fmaxf(p, -a.clamp), a.clamp);
            a.m[net][i] = m;
            a.v[net][i] = v;
            a.p[net][i] = p;
        } else {
            bad = true;
        }
        // the target network follows the (possibly unchanged) weights
        if (a.target[net] != nullptr) {
            const float pk = a.polyak[net];
            a.target[net][i] = (1.0f - pk) * a.target[net][i] + pk * p;
        }
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, bad);
    if ((threadIdx.x & 31) == 0 && ballot != 0u) atomicAdd(a.status + OFRL_STAT_NONFINITE_GRAD, __popc(ballot));
}

__global__ void __launch_bounds__(256) combine_kernel(const CombineLaunch a) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < a.n) {
        float g = 0.0f;
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k)   // unrolled: the source pointers stay in registers
            if (k < a.n_src) g = fmaf(a.scalars[SC_COEF0 + k], __ldg(a.src[k] + i), g);
        a.out[i] = g;
    }
    if (blockIdx.x == 0 && a.norms_out != nullptr) {
        if ((int)threadIdx.x < a.n_src) a.norms_out[threadIdx.x] = a.scalars[SC_NORM0 + threadIdx.x];
        if ((int)threadIdx.x == a.n_src) a.norms_out[threadIdx.x] = a.scalars[SC_COMBINED];
    }
}

constexpr int kLossThreads = 1024;

__global__ void __launch_bounds__(kLossThreads) expectile_kernel(const float* __restrict__ q,
                                                                 const float* __restrict__ v, int B,
                                                                 float tau, float* loss_out,
                                                                 float* dv_out) {
    __shared__ float sh[kLossThreads / 32];
    float s = 0.0f;
    for (int i = threadIdx.x; i < B; i += kLossThreads) {
        const float d = __ldg(q + i) - __ldg(v + i);
        const float w = d >= 0.0f ? tau : 1.0f - tau;
        s += w * d * d;
        if (dv_out != nullptr) dv_out[i] = (-2.0f * w * d) / (float)B;
    }
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int y = 0; y < kLossThreads / 32; ++y) t += sh[y];
        *loss_out = t / (float)B;
    }
}

__global__ void __launch_bounds__(256) policy_kernel(const float* __restrict__ q, const float* __restrict__ v,
                                                     int B, int NA, float beta, float* pi_out,
                                                     int32_t* argmax_out) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const float vb = __ldg(v + b);
    const float* qr = q + (int64_t)b * NA;
    // three passes over the row (no local array): max / argmax, sum of
    // exponentials, outputs
    float zmax = -INFINITY, amax = -INFINITY;
    int best = 0;
    for (int k = 0; k < NA; ++k) {
        const float adv = fminf(fmaxf(__ldg(qr + k) - vb, -10.0f), 10.0f);
        if (adv > amax) { amax = adv; best = k; }
        zmax = fmaxf(zmax, beta * adv);
    }
    float sum = 0.0f;
    for (int k = 0; k < NA; ++k) sum += expf(beta * fminf(fmaxf(__ldg(qr + k) - vb, -10.0f), 10.0f) - zmax);
    float* po = pi_out + (int64_t)b * NA;
    for (int k = 0; k < NA; ++k) po[k] = expf(beta * fminf(fmaxf(__ldg(qr + k) - vb, -10.0f), 10.0f) - zmax) / sum;
    if (argmax_out != nullptr) argmax_out[b] = best;
}

}  // namespace

int reduce_grid(int64_t P, int el) {
    const int64_t g = (P + 4 * el - 1) / (4 * el);
    return (int)(g < kMaxGramBlocks ? (g < 1 ? 1 : g) : kMaxGramBlocks);
}

template <int EL, bool ADAM>
cudaError_t configure_reduce() {
    static cudaError_t state = cudaErrorNotReady;
    if (state == cudaErrorNotReady) state = set_max_shared_carveout(reduce_gram_kernel<EL, ADAM>);
    return state;
}

template <int EL>
cudaError_t launch_reduce_el(const ReduceLaunch& a, cudaStream_t st) {
    const cudaError_t e = configure_reduce<EL, false>();
    if (e != cudaSuccess) return e;
    const dim3 grid(reduce_grid(a.P, EL), a.n_nets);
    AdamLaunch none;
    memset(&none, 0, sizeof(none));
    return launch_ex(reduce_gram_kernel<EL, false>, grid, dim3(kRedThreads), 0, st, 1u, false, a, none,
                     (unsigned long long*)nullptr, 0ull);
}

// CTAs of the fused kernel resident at once on the current device (0
// without cooperative launch support).
template <int EL>
int max_resident_reduce_adam() {
    static int n = -1;
    if (n < 0) {
        n = 0;
        int dev = 0, coop = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            configure_reduce<EL, true>() == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reduce_gram_kernel<EL, true>, kRedThreads, 0) ==
                cudaSuccess)
            n = per_sm * sms;
        cudaGetLastError();
    }
    return n;
}

// One pass of the EL-lane grid covers P and fits on the device at once.
template <int EL>
bool fits_one_pass(const ReduceLaunch& a) {
    const int g = reduce_grid(a.P, EL);
    return (int64_t)g * 4 * EL >= a.P && g * a.n_nets <= max_resident_reduce_adam<EL>();
}

int reduce_el(const ReduceLaunch& a) {
    const int parts = a.n_parts > 0 ? a.n_parts : a.n_tiles;
    if (a.partials == nullptr) return 8;
    if (parts <= kManyParts) return 32;
    // many partials: 32 element lanes (8 partial lanes), else 64, when that
    // grid fits one pass (measured with 128 partials: 33.9 us a step at 32
    // lanes, 34.9 at 64, 35.2 at 16, whose grid is twice as large)
    if (fits_one_pass<32>(a)) return 32;
    if (fits_one_pass<64>(a)) return 64;
    return 8;
}

cudaError_t launch_reduce_gram(const ReduceLaunch& a, cudaStream_t st) {
    switch (reduce_el(a)) {
        case 32: return launch_reduce_el<32>(a, st);
        case 64: return launch_reduce_el<64>(a, st);
        default: return launch_reduce_el<8>(a, st);
    }
}

int reduce_adam_blocks(const ReduceLaunch& r) { return reduce_grid(r.P, reduce_el(r)) * r.n_nets; }

bool reduce_adam_fusable(const ReduceLaunch& r) {
    if (r.partials == nullptr) return false;
    const int el = reduce_el(r);
    const int64_t per_pass = (int64_t)reduce_grid(r.P, el) * 4 * el;
    if (per_pass < r.P) return false;   // one pass of the grid must cover P
    const int resident = el == 32   ? max_resident_reduce_adam<32>()
                         : el == 64 ? max_resident_reduce_adam<64>()
                                    : max_resident_reduce_adam<8>();
    return reduce_adam_blocks(r) <= resident;
}

cudaError_t launch_reduce_adam(const ReduceLaunch& r, const AdamLaunch& a, unsigned long long* barrier,
                               unsigned long long barrier_base, cudaStream_t st) {
    const int el = reduce_el(r);
    const dim3 grid(reduce_grid(r.P, el), r.n_nets);
    const unsigned long long target = barrier_base + (unsigned long long)grid.x * grid.y;
    if (el == 32) {
        const cudaError_t e = configure_reduce<32, true>();
        if (e != cudaSuccess) return e;
        return launch_ex(reduce_gram_kernel<32, true>, grid, dim3(kRedThreads), 0, st, 1u, true, r, a, barrier,
                         target);
    }
    if (el == 64) {
        const cudaError_t e = configure_reduce<64, true>();
        if (e != cudaSuccess) return e;
        return launch_ex(reduce_gram_kernel<64, true>, grid, dim3(kRedThreads), 0, st, 1u, true, r, a, barrier,
                         target);
    }
    const cudaError_t e = configure_reduce<8, true>();
    if (e != cudaSuccess) return e;
    return launch_ex(reduce_gram_kernel<8, true>, grid, dim3(kRedThreads), 0, st, 1u, true, r, a, barrier, target);
}

cudaError_t launch_adam(const AdamLaunch& a, cudaStream_t st) {
    if (a.n <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((a.n + 255) / 256), a.n_nets);
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = set_max_shared_carveout(adam_kernel);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(adam_kernel, grid, dim3(256), 0, st, a);
}

__global__ void __launch_bounds__(256) target_ema_kernel(const float* __restrict__ p, float* __restrict__ target,
                                                         int64_t n, float polyak) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) target[i] = (1.0f - polyak) * target[i] + polyak * __ldg(p + i);
}

cudaError_t launch_target_ema(const float* p, float* target, int64_t n, float polyak, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    target_ema_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p, target, n, polyak);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineLaunch& a, cudaStream_t st) {
    const unsigned blocks = (unsigned)((a.n + 255) / 256);
    combine_kernel<<<blocks < 1 ? 1 : blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_expectile(const float* q_taken, const float* v, int batch, float tau,
                             float* loss_out, float* dv_out, cudaStream_t st) {
    expectile_kernel<<<1, kLossThreads, 0, st>>>(q_taken, v, batch, tau, loss_out, dv_out);
    return cudaGetLastError();
}

cudaError_t launch_policy(const float* q, const float* v, int batch, int num_actions, float beta,
                          float* pi_out, int32_t* argmax_out, int64_t, int, cudaStream_t st) {
    policy_kernel<<<(batch + 255) / 256, 256, 0, st>>>(q, v, batch, num_actions, beta, pi_out, argmax_out);
    return cudaGetLastError();
}

}  // namespace ofrl
