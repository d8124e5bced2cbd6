// HER index sampling + gather + relabel.
//
// Method: "GPU IQL + HER Porting Plan", "CUDA Kernel: her_relabel_kernel.cu"
// (copy the source transition, overwrite the goal slice of state and
// next_state with the donor's achieved goal next_states[donor, :g], copy
// action and done, recompute the reward from the fp32 goal distance) and
// "Donor Index Generation" (Final / Future / Random).  The pages launch one
// warp per relabelled row and a separate donor kernel; here the index draw,
// the donor search and the row copy are one pass, and a row is moved by 16
// lanes with 16-byte loads and stores, so one warp moves two rows.  Random
// numbers come from a counter-based SplitMix64 instead of cuRAND, so any
// row's indices depend only on (seed, step, row).
//
// Memory-bound: per row 2 * copy_cols * 4 bytes gathered and written, plus
// g * 4 donor bytes and the scalars.  Source rows are whole 32-byte sectors
// when the row stride is a multiple of 8 floats.

#include "common.cuh"

namespace ofrl {
namespace {

constexpr int kLanesPerRow = 16;
constexpr int kRelabelThreads = 256;
constexpr int kRowsPerBlock = kRelabelThreads / kLanesPerRow;

// First entry of `ends` above i (binary search); n if there is none.
__device__ __forceinline__ int upper_bound_i32(const int32_t* __restrict__ ends, int n, int i) {
    int lo = 0, hi = n;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (__ldg(ends + mid) > i) hi = mid; else lo = mid + 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kRelabelThreads) her_relabel_kernel(const HerLaunch a) {
    const int lane = threadIdx.x & (kLanesPerRow - 1);
    const int row = blockIdx.x * kRowsPerBlock + threadIdx.x / kLanesPerRow;
    const bool live = row < a.batch;

    int src = 0, donor = -1, bad = 0;
    if (lane == 0 && live) {
        const uint64_t ctr = (a.step << 32) | ((uint64_t)row << 1);
        src = (int)below(sm64_at(a.seed, ctr), (uint64_t)a.capacity);
        if (row >= a.first_her) {
            if (a.strategy == OFRL_HER_RANDOM) {
                donor = (int)below(sm64_at(a.seed, ctr | 1ull), (uint64_t)a.capacity);
            } else {
                const int k = upper_bound_i32(a.episode_ends, a.num_episodes, src);
                int end;
                if (k < a.num_episodes) {
                    end = __ldg(a.episode_ends + k);
                } else {
                    end = a.capacity;  // malformed boundaries: flagged, stay in the buffer
                    bad = 1;
                }
                if (a.strategy == OFRL_HER_FINAL) {
                    donor = end - 1;
                } else {
                    const int lo = src + 1;
                    donor = lo < end ? lo + (int)below(sm64_at(a.seed, ctr | 1ull), (uint64_t)(end - lo))
                                     : src;
                }
            }
        }
    }
    src = __shfl_sync(0xffffffffu, src, 0, kLanesPerRow);
    donor = __shfl_sync(0xffffffffu, donor, 0, kLanesPerRow);
    if (!live) return;

    const float4* s_in = reinterpret_cast<const float4*>(a.states + (int64_t)src * a.in_stride);
    const float4* n_in = reinterpret_cast<const float4*>(a.next_states + (int64_t)src * a.in_stride);
    const float4* d_in = reinterpret_cast<const float4*>(a.next_states + (int64_t)(donor < 0 ? 0 : donor) * a.in_stride);
    float4* s_out = reinterpret_cast<float4*>(a.out_states + (int64_t)row * a.out_stride);
    float4* n_out = reinterpret_cast<float4*>(a.out_next_states + (int64_t)row * a.out_stride);
    const int chunks = a.copy_cols >> 2;
    for (int c = lane; c < chunks; c += kLanesPerRow) {
        float4 sv = __ldg(s_in + c);
        float4 nv = __ldg(n_in + c);
        if (donor >= 0 && 4 * c < a.goal_dim) {
            const float4 gv = __ldg(d_in + c);
            const int base = 4 * c;
            if (base + 0 < a.goal_dim) { sv.x = gv.x; nv.x = gv.x; }
            if (base + 1 < a.goal_dim) { sv.y = gv.y; nv.y = gv.y; }
            if (base + 2 < a.goal_dim) { sv.z = gv.z; nv.z = gv.z; }
            if (base + 3 < a.goal_dim) { sv.w = gv.w; nv.w = gv.w; }
        }
        s_out[c] = sv;
        n_out[c] = nv;
    }
    if (lane == 0) {
        float r;
        if (donor >= 0) {
            // fp32 distance as the pages' kernel: float accumulator in order,
            // each product and sum rounded on its own (no FMA), IEEE sqrtf.
            const float* ns = a.next_states + (int64_t)src * a.in_stride;
            const float* nd = a.next_states + (int64_t)donor * a.in_stride;
            float dsq = 0.0f;
            for (int d = 0; d < a.goal_dim; ++d) {
                const float diff = __fsub_rn(__ldg(ns + d), __ldg(nd + d));
                dsq = __fadd_rn(dsq, __fmul_rn(diff, diff));
            }
            const float dist = __fsqrt_rn(dsq);
            r = dist < a.threshold ? 1.0f : -0.01f;
        } else {
            r = __ldg(a.rewards + src);
        }
        a.out_actions[row] = __ldg(a.actions + src);
        a.out_dones[row] = __ldg(a.dones + src);
        a.out_rewards[row] = r;
        a.out_src[row] = src;
        a.out_donor[row] = donor;
        if (bad) atomicAdd(a.status + OFRL_STAT_BAD_INDEX, 1);
    }
}

}  // namespace

cudaError_t launch_her_relabel(const HerLaunch& a, cudaStream_t st) {
    if (a.batch <= 0) return cudaSuccess;
    const int blocks = (a.batch + kRowsPerBlock - 1) / kRowsPerBlock;
    her_relabel_kernel<<<blocks, kRelabelThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ofrl
