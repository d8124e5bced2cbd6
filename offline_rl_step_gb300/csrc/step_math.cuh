// Device arithmetic of the reduce and Adam kernels: turning the Gram matrix
// of the gradient sources into norms, clip coefficients and the combined
// norm; one Adam element; a bounded grid barrier for the cooperative launch
// that does both.
//
// Method: "Gradient Stability -- Multi-Task Gradient Isolation + Full
// Spectral Norm", "Proper design" (each source clipped to its budget
// fraction of max_grad_norm, then added) and "DQN Backward-Path NaN Audit",
// Adam kernel findings (the (n > c && n > 0) ? c / n : 1 clip, non-finite
// elements skipped, bias correction with t >= 1).
#pragma once

#include "common.cuh"

namespace ofrl {

struct NormResult {
    float nrm[kMaxSrc];    // pre-clip source norms (0 for absent sources)
    float coef[kMaxSrc];   // alpha_k * s_k (0 for absent sources)
    float combined;        // ||sum_k coef_k g_k|| from the Gram matrix
    float loss;            // mean expectile loss
};

// Norms, coefficients and the combined norm from the Gram matrix of the
// n_src sources (upper triangle, gram_index order) and the summed loss.
// Loops run over kMaxSrc with guards, so the arrays stay in registers.
// IEEE arithmetic throughout: a NaN source norm gives coefficient 1 and a
// NaN total; an infinite one gives coefficient 0 and 0 * inf = NaN, as the
// element-wise sum of the clipped sources would.
__device__ __forceinline__ NormResult finish_norms(const float (&gram)[kGramPairs], float loss_sum, int n_src,
                                                   const float* budget, const float* alpha, float max_grad_norm,
                                                   float inv_batch) {
    NormResult r;
#pragma unroll
    for (int k = 0; k < kMaxSrc; ++k) {
        r.nrm[k] = 0.0f;
        r.coef[k] = 0.0f;
        if (k < n_src) {
            r.nrm[k] = sqrtf(gram[gram_index(k, k)]);
            r.coef[k] = alpha[k] * clip_scale(r.nrm[k], budget[k] * max_grad_norm);
        }
    }
    float c2 = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxSrc; ++j)
#pragma unroll
        for (int k = 0; k < kMaxSrc; ++k) {
            const int lo = j < k ? j : k, hi = j < k ? k : j;
            if (j < n_src && k < n_src) c2 += r.coef[j] * r.coef[k] * gram[gram_index(lo, hi)];
        }
    r.combined = c2 < 0.0f ? 0.0f : sqrtf(c2);
    r.loss = loss_sum * inv_batch;
    return r;
}

// One Adam element with decoupled weight decay; false (and nothing written)
// when the clipped gradient g is not finite.
__device__ __forceinline__ bool adam_element(float& p, float& m, float& v, float g, float beta1, float beta2,
                                             float eps, float weight_decay, float lr, float bc1, float bc2) {
    if (!isfinite(g)) return false;
    m = beta1 * m + (1.0f - beta1) * g;
    v = beta2 * v + (1.0f - beta2) * g * g;
    const float mhat = m / bc1;
    const float vhat = v / bc2;
    p = p - lr * (mhat / (sqrtf(vhat) + eps) + weight_decay * p);
    return true;
}

// Grid-wide barrier of a cooperative launch (every CTA resident).  The
// arrival counter only grows: barrier k of the context's history completes
// when it reaches `target` = (k + 1) * CTAs, so a CTA that gave up waiting
// (after limit_ns; returns false) still arrives exactly once and later
// barriers stay consistent.  All threads of the CTA call it.
__device__ __forceinline__ bool grid_barrier(unsigned long long* count, unsigned long long target,
                                             uint64_t limit_ns) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(count, 1ull);
        const volatile unsigned long long* c = count;
        bool ok = true;
        if (*c < target) {
            uint64_t t0;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
            while (*c < target) {
                __nanosleep(32);
                uint64_t t;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
                if (t - t0 > limit_ns) {
                    ok = false;
                    break;
                }
            }
        }
        __threadfence();
        ok_s = ok ? 1 : 0;
    }
    __syncthreads();
    return ok_s != 0;
}

}  // namespace ofrl
