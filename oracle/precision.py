"""bf16 rounding of GEMM operands for the bf16-operand workload (oracle side).

TEST INFRASTRUCTURE ONLY (see the package header).

"Phase 2: Multi-Stream Graph Parallelism", "2C. Grouped GEMM for IQL": the
twin IQL networks run their GEMMs with bf16 inputs, fp32 accumulation and
fp32 master weights.  The oracle's reading of that mode: every operand of the
five matrix products of the step (z1 = X W1^T, z2 = h1 W2^T, dW2 = dz2^T h1,
dh1 = dz2 W2, dW1 = dz1^T X) is rounded to the nearest bf16 value, ties to
the even significand; the products are then summed exactly (fp64).  Biases,
the N = 1 output layer (V, dW3) and the batch sums of the bias gradients keep
full precision.

bf16 is IEEE 754 binary32 with the significand cut to 8 bits (7 stored):
8 exponent bits, normal numbers from 2^-126, subnormal spacing 2^-133, the
largest finite value (2 - 2^-7) 2^127.
"""
import numpy as np

_EMIN = -125          # frexp exponent of the smallest normal bf16 value, 2^-126 = 0.5 * 2^-125
_SIG = 8              # significand bits
_OVERFLOW = 2.0 ** 128


def bf16(x):
    """x rounded to the nearest bf16 value, ties to even (fp64 in, fp64 out).

    With x = m 2^e (0.5 <= |m| < 1), the bf16 grid near x has spacing
    2^(e - 8) (2^-133 below the normal range); np.rint rounds half-way
    cases to the even integer, which is the even significand.  A result
    that reaches 2^128 is outside the format and becomes +-inf; NaN and
    +-inf pass through.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, _EMIN)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.ldexp(np.rint(np.ldexp(x, _SIG - e)), e - _SIG)
        r = np.where(np.abs(r) >= _OVERFLOW, np.copysign(np.inf, x), r)
    r = np.where(np.isfinite(x), r, x)
    return r
