// Self-test of the tensor-core building blocks: one 128 x N x K product on
// one CTA, operands staged into shared memory in the layout and major-ness
// the caller picks, D read back from tensor memory.  Used by the tests to
// check the descriptors, the MMA kinds and the tf32 split before the hot-path
// kernels rely on them.

#include "common.cuh"
#include "umma.cuh"
#include "../../include/ofrl_selftest.h"

namespace ofrl {
namespace {

constexpr int kSelfThreads = 128;

// Byte offset of element (r, c) of a tile with `rows` rows (r = batch-row-like
// index, grouped in 8s) and c along the 16-byte chunk dimension, core matrices
// of 8 rows x 16 bytes: chunk-major inside an 8-row group (LBO = 128 between
// chunks), groups SBO = chunks * 128 apart.
__device__ __forceinline__ uint32_t core_offset(int r, int c, int n_chunks, int esize) {
    const int per = 16 / esize;
    return (uint32_t)((r >> 3) * n_chunks * 128 + (c / per) * 128 + (r & 7) * 16 + (c % per) * esize);
}

__global__ void __launch_bounds__(kSelfThreads, 1) umma_selftest_kernel(const float* __restrict__ A,
                                                                        const float* __restrict__ B,
                                                                        float* __restrict__ D, int N, int K,
                                                                        int kind, int a_mn, int b_mn, int mn_swap,
                                                                        int* flag) {
    constexpr int M = 128;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    const bool tf32 = kind != OFRL_SELFTEST_BF16;
    const bool split = kind == OFRL_SELFTEST_TF32X3;
    const int esize = tf32 ? 4 : 2;
    const int per = 16 / esize;
    // A is [M][K] (M rows, K along chunks) when K-major; [K][M] (K rows,
    // M along chunks) when MN-major.  Same for B with N.
    const int a_rows = a_mn ? K : M, a_cols = a_mn ? M : K;
    const int b_rows = b_mn ? K : N, b_cols = b_mn ? N : K;
    const uint32_t a_bytes = (uint32_t)(a_rows * a_cols * esize);
    const uint32_t b_bytes = (uint32_t)(b_rows * b_cols * esize);
    uint8_t* a_hi = smem;
    uint8_t* b_hi = smem + a_bytes;
    uint8_t* a_lo = smem + a_bytes + b_bytes;
    uint8_t* b_lo = a_lo + a_bytes;

    for (int e = threadIdx.x; e < M * K; e += kSelfThreads) {
        const int m = e / K, k = e % K;
        const float x = A[e];
        const uint32_t off = a_mn ? core_offset(k, m, a_cols / per, esize) : core_offset(m, k, a_cols / per, esize);
        if (tf32) {
            float hi = x, lo = 0.0f;
            if (split) umma::split_tf32(x, hi, lo);
            *reinterpret_cast<float*>(a_hi + off) = hi;
            if (split) *reinterpret_cast<float*>(a_lo + off) = lo;
        } else {
            *reinterpret_cast<__nv_bfloat16*>(a_hi + off) = __float2bfloat16_rn(x);
        }
    }
    for (int e = threadIdx.x; e < N * K; e += kSelfThreads) {
        const int n = e / K, k = e % K;
        const float x = B[e];
        const uint32_t off = b_mn ? core_offset(k, n, b_cols / per, esize) : core_offset(n, k, b_cols / per, esize);
        if (tf32) {
            float hi = x, lo = 0.0f;
            if (split) umma::split_tf32(x, hi, lo);
            *reinterpret_cast<float*>(b_hi + off) = hi;
            if (split) *reinterpret_cast<float*>(b_lo + off) = lo;
        } else {
            *reinterpret_cast<__nv_bfloat16*>(b_hi + off) = __float2bfloat16_rn(x);
        }
    }
    umma::fence_smem_to_async();
    if (threadIdx.x == 0) {
        umma::mbar_init(&bar, 1);
        umma::fence_mbar_init();
    }
    uint32_t ncols = 32;
    while (ncols < (uint32_t)N) ncols <<= 1;
    if (threadIdx.x < 32) umma::tmem_alloc(&tmem_slot, ncols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (threadIdx.x == 0) {
        const uint32_t idesc = umma::instr_desc(tf32 ? umma::kTypeTF32 : umma::kTypeBF16, a_mn, b_mn, M, N);
        const int kstep = tf32 ? 8 : 16;   // 32 bytes of K per instruction
        const uint32_t a_sbo = (uint32_t)(a_cols / per) * 128, b_sbo = (uint32_t)(b_cols / per) * 128;
        int issued = 0;
        for (int k0 = 0; k0 < K; k0 += kstep) {
            // K-major: K runs along chunks (two 16-byte chunks per step);
            // MN-major: K runs along rows (kstep rows = kstep / 8 groups per step)
            const uint32_t a_off = a_mn ? (uint32_t)(k0 / 8) * a_sbo : (uint32_t)(k0 / per) * 128;
            const uint32_t b_off = b_mn ? (uint32_t)(k0 / 8) * b_sbo : (uint32_t)(k0 / per) * 128;
            const int terms = split ? 3 : 1;
            for (int t = 0; t < terms; ++t) {
                const uint8_t* ap = (t == 2) ? a_lo : a_hi;    // hi*hi, hi*lo, lo*hi
                const uint8_t* bp = (t == 1) ? b_lo : b_hi;
                // The leading byte offset is the stride between core matrices
                // along K, the stride byte offset the stride along M (or N):
                // K-major: LBO = next chunk (128), SBO = next 8-row group;
                // MN-major: LBO = next 8-row group, SBO = next chunk (128).
                // mn_swap exchanges the two for MN-major operands (a
                // deliberately wrong assignment, to show the test can tell).
                const bool sa = a_mn && !mn_swap, sb = b_mn && !mn_swap;
                const uint64_t ad = umma::smem_desc(umma::smem_u32(ap) + a_off, sa ? a_sbo : 128u, sa ? 128u : a_sbo);
                const uint64_t bd = umma::smem_desc(umma::smem_u32(bp) + b_off, sb ? b_sbo : 128u, sb ? 128u : b_sbo);
                if (tf32) umma::mma_tf32(tmem, ad, bd, idesc, issued > 0);
                else umma::mma_f16(tmem, ad, bd, idesc, issued > 0);
                ++issued;
            }
        }
        umma::commit(&bar);
    }
    __syncwarp();
    const bool done = umma::mbar_wait(&bar, 0, 1000000000ull);
    if (!done && (threadIdx.x & 31) == 0) atomicAdd(flag, 1);
    umma::fence_after_sync();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        umma::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        umma::tmem_ld_wait();
        for (int j = 0; j < 16; ++j)
            if (c0 + j < N) D[row * N + c0 + j] = done ? v[j] : 0.0f;
    }
    umma::fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) umma::tmem_dealloc(tmem, ncols);
}

}  // namespace
}  // namespace ofrl

extern "C" ofrl_status ofrl_selftest_umma(const float* a, const float* b, float* d, int32_t n, int32_t k,
                                          int32_t kind, int32_t a_mn, int32_t b_mn, int32_t mn_swap, int32_t* flag,
                                          void* stream) {
    if (!a || !b || !d || !flag) return OFRL_EINVAL;
    if (kind != OFRL_SELFTEST_TF32 && kind != OFRL_SELFTEST_TF32X3 && kind != OFRL_SELFTEST_BF16) return OFRL_EINVAL;
    // tf32 operands are K-major only (MN-major tf32 gives wrong products)
    if (kind != OFRL_SELFTEST_BF16 && (a_mn || b_mn)) return OFRL_EUNSUPPORTED;
    if (n < 16 || n > 256 || n % 16 != 0) return OFRL_EINVAL;
    const int kstep = kind == OFRL_SELFTEST_BF16 ? 16 : 8;
    if (k < kstep || k > 128 || k % kstep != 0 || (a_mn && k % 8) || (b_mn && k % 8)) return OFRL_EINVAL;
    const int esize = kind == OFRL_SELFTEST_BF16 ? 2 : 4;
    const size_t need = (size_t)(128 + n) * k * esize * (kind == OFRL_SELFTEST_TF32X3 ? 2 : 1);
    if (need > 96 * 1024) return OFRL_EINVAL;
    // an MN-major operand wider than 128 could, under a misread descriptor,
    // address past the shared-memory window: refuse it
    if ((b_mn && n > 128)) return OFRL_EINVAL;
    // reserve the whole window, so every address a descriptor of these
    // operands can form stays inside this CTA's shared memory
    const size_t smem = 226 * 1024;
    auto kern = ofrl::umma_selftest_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return OFRL_ECUDA;
    kern<<<1, ofrl::kSelfThreads, smem, static_cast<cudaStream_t>(stream)>>>(a, b, d, n, k, kind, a_mn, b_mn, mn_swap, flag);
    return cudaGetLastError() == cudaSuccess ? OFRL_OK : OFRL_ECUDA;
}

extern "C" ofrl_status ofrl_selftest_barrier(ofrl_ctx* ctx, uint64_t wait_ns, int32_t unreachable) {
    if (ctx == nullptr || (unreachable != 0 && unreachable != 1)) return OFRL_EINVAL;
    if (wait_ns != 0 && (wait_ns < 1000ull || wait_ns > 10000000000ull)) return OFRL_EINVAL;
    ctx->barrier_wait_ns = wait_ns != 0 ? wait_ns : 1000000000ull;
    ctx->barrier_unreachable = unreachable;
    return OFRL_OK;
}
