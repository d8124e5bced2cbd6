/*
 * ofrl_selftest.h -- self-test hook of the ofrl library's tensor-core
 * building blocks (not part of the method; the tests use it to check the
 * shared-memory descriptors and MMA kinds the hot-path kernels rely on).
 */
#ifndef OFRL_SELFTEST_H
#define OFRL_SELFTEST_H

#include <stdint.h>

#include "ofrl.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { OFRL_SELFTEST_TF32 = 0, OFRL_SELFTEST_TF32X3 = 1, OFRL_SELFTEST_BF16 = 2 };

/* D[128, n] = A[128, k] . B[n, k]^T on one CTA with tcgen05 MMAs.
 * a, b, d: device fp32, row-major as shown.  kind: TF32 (operands read as
 * tf32), TF32X3 (each operand split into a tf32 high part and the fp32
 * remainder; hi.hi + hi.lo + lo.hi), BF16 (operands rounded to bf16).
 * a_mn / b_mn: stage the operand MN-major (1) instead of K-major (0); BF16
 * only (TF32 / TF32X3 with an MN-major operand return OFRL_EUNSUPPORTED).
 * Descriptor rule checked here: the leading byte offset is the stride between
 * core matrices along K, the stride byte offset the stride along M or N, for
 * both majors.  mn_swap = 1 exchanges them for MN-major operands (a wrong
 * assignment, for the test to show it is detected).
 * n: 16..256, multiple of 16; k: multiple of the instruction's K (8 for tf32,
 * 16 for bf16), up to 128.  *flag (device int) is incremented if the MMA
 * completion wait gave up (then D is zero).  Asynchronous on `stream`. */
ofrl_status ofrl_selftest_umma(const float* a, const float* b, float* d, int32_t n, int32_t k, int32_t kind,
                               int32_t a_mn, int32_t b_mn, int32_t mn_swap, int32_t* flag, void* stream);

/* Self-test of the bounded grid barrier of the fused reduce + Adam launch
 * (the train step's optimizer kernel when its grid fits on the device at
 * once; "DQN Backward-Path NaN Audit", Phase E: device anomalies become
 * sticky status flags the host reads, never a fault or a hang).
 * For the train steps of ctx that follow:
 *   wait_ns      how long each CTA waits at the barrier before it gives up
 *                (1000 .. 1e10 ns; 0 restores the default, 1 s);
 *   unreachable  1: the launch's barrier target is one above the arrivals
 *                its grid can make, so every CTA waits wait_ns and gives up;
 *                0: the normal target.
 * A CTA that gives up writes no norms, loss, weights, moments or target and
 * adds 1 to the status word's timeout count (ofrl_poll_status); the reduced
 * primary gradient (written before the barrier) is complete.  The arrival
 * count stays consistent, so the next normal step runs as usual.  Returns
 * OFRL_EINVAL for a null ctx or values out of range; launches nothing. */
ofrl_status ofrl_selftest_barrier(ofrl_ctx* ctx, uint64_t wait_ns, int32_t unreachable);

#ifdef __cplusplus
}
#endif
#endif /* OFRL_SELFTEST_H */
