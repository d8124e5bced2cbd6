"""Pins for the oracle's bf16-operand mode (oracle/precision.py and the
gemm_operand argument of oracle/iql.py).

The rounding itself is pinned to a library routine (torch's float32 ->
bfloat16 conversion, round to nearest even) and to hand-worked cases of the
format.  The mode is pinned by what it must and must not change: on a
network whose every GEMM operand is already a bf16 value it equals the exact
oracle bit for bit; a perturbation below half a bf16 step of the operands
that are rounded (X, W1, W2, dz2) leaves its GEMM results unchanged, while a
perturbation of a value that is not a GEMM operand (w3, b2, b3, Q) reaches
V and the sums that use it unrounded.
"""
import numpy as np
import pytest
import torch

from oracle import iql
from oracle.precision import bf16


def test_bf16_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-90, 85, 200_000))).astype(np.float32)
    # exact half-way cases: bit 15 set, bits 0-14 clear, any upper half
    ties = ((rng.integers(0, 2 ** 16, 50_000).astype(np.uint32) << 16) | (1 << 15)).view(np.float32)
    ties = ties[np.isfinite(ties)]
    sub = (rng.integers(1, 2 ** 23, 20_000).astype(np.uint32)).view(np.float32)   # fp32 subnormals
    x = np.concatenate([x, ties, sub])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = bf16(x.astype(np.float64))
    assert np.array_equal(got.view(np.uint64), want.view(np.uint64))


@pytest.mark.parametrize("x, want", [
    (1.0, 1.0),
    (1 + 2 ** -8, 1.0),                       # half-way, even significand below
    (1 + 3 * 2 ** -8, 1 + 2 ** -6),           # half-way, even significand above
    (1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -7),    # just above half-way
    (-(1 + 2 ** -8), -1.0),
    (255.0, 255.0),                           # integers up to 256 are exact
    (257.0, 256.0),                           # spacing 2 above 256: half-way, even
    (259.0, 260.0),
    (0.1, 0.10009765625),                     # 0x3DCD
    (2.0 ** -130, 2.0 ** -130),               # subnormal, on the 2^-133 grid
    (3 * 2.0 ** -134, 2.0 ** -132),           # half-way on the subnormal grid, even above
    (2.0 ** -134, 0.0),                       # half of the smallest subnormal: even is zero
    ((2 - 2 ** -7) * 2.0 ** 127, (2 - 2 ** -7) * 2.0 ** 127),   # largest finite
    ((2 - 2 ** -8) * 2.0 ** 127, np.inf),     # half-way to 2^128: rounds out of range
    (np.inf, np.inf), (-np.inf, -np.inf),
])
def test_bf16_hand_cases(x, want):
    assert bf16(np.float64(x)) == want


def test_bf16_keeps_signed_zero_and_nan():
    assert np.signbit(bf16(-0.0)) and bf16(-0.0) == 0.0
    assert np.isnan(bf16(np.nan))


def _integer_net():
    """A net whose GEMM operands are all bf16 values: integer states and
    weights, half-integer biases, tau = 0.5 and B = 4 so dL/dV = -(q - V) / 4, and the targets
    q = V + small integers, so dz2, dh1 and dz1 are multiples of 1/4 below 64."""
    rng = np.random.default_rng(5)
    s, h, b = 4, 3, 4
    w1 = rng.integers(-1, 2, (h, s)).astype(float)
    b1 = np.array([1.5, 2.0, 0.0])
    w2 = rng.integers(-1, 2, (h, h)).astype(float)
    b2 = np.array([3.0, 1.0, 2.0])
    w3 = np.array([[1.0, -1.0, 2.0]])
    b3 = np.array([0.5])
    flat = iql.flatten(w1, b1, w2, b2, w3, b3)
    x = rng.integers(-2, 3, (b, s)).astype(float)
    v, _ = iql.forward(flat, x, s, h)
    qt = v + np.array([2.0, -1.0, 1.0, -2.0])
    return flat, x, qt, s, h


def test_bf16_mode_is_exact_on_bf16_operands():
    flat, x, qt, s, h = _integer_net()
    v, loss, g = iql.value_fwd_bwd(flat, x, qt, 0.5, s, h)
    vb, lossb, gb = iql.value_fwd_bwd(flat, x, qt, 0.5, s, h, gemm_operand=bf16)
    # every operand is representable: nothing is rounded
    _, act = iql.forward(flat, x, s, h)
    for a in (act["x"], act["h1"]):
        assert np.array_equal(bf16(a), a)
    assert np.count_nonzero(g) > 10   # a non-trivial gradient
    assert np.array_equal(v, vb) and loss == lossb and np.array_equal(g, gb)


def _bump(a, delta):
    """a + delta on the entries with |a| >= 1 (half a bf16 step there is >= 2^-8 > delta)."""
    a = a.copy()
    a[np.abs(a) >= 1] += delta
    return a


def test_bf16_mode_rounds_gemm_operands_only():
    flat, x, qt, s, h = _integer_net()
    d = 2.0 ** -12
    base_v, _, base_g = iql.value_fwd_bwd(flat, x, qt, 0.5, s, h, gemm_operand=bf16)
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
    seg = iql.unflatten(np.arange(len(flat)), s, h)
    idx = {k: np.asarray(a, dtype=int).ravel() for k, a in zip(("w1", "b1", "w2", "b2", "w3", "b3"), seg)}

    # X, W1, W2: rounded before their products; b1 reaches z2 only through
    # h1, which is rounded before G2 and dW2.  V and every gradient entry are
    # unchanged (no gradient entry involves these values except through
    # rounded operands)
    _, act = iql.forward(flat, x, s, h)
    assert (act["z1"][:, np.abs(b1) >= 1] != 0).all()   # no ReLU kink moves with b1
    for name, args in (("x", (flat, _bump(x, d))),
                       ("w1", (iql.flatten(_bump(w1, d), b1, w2, b2, w3, b3), x)),
                       ("b1", (iql.flatten(w1, _bump(b1, d), w2, b2, w3, b3), x)),
                       ("w2", (iql.flatten(w1, b1, _bump(w2, d), b2, w3, b3), x))):
        v, _, g = iql.value_fwd_bwd(args[0], args[1], qt, 0.5, s, h, gemm_operand=bf16)
        assert np.array_equal(v, base_v), name
        assert np.array_equal(g, base_g), name
        # the exact mode does see the perturbation
        ve, _, _ = iql.value_fwd_bwd(args[0], args[1], qt, 0.5, s, h)
        assert not np.array_equal(ve, iql.value_fwd_bwd(flat, x, qt, 0.5, s, h)[0]), name

    # w3, b2, b3 are not GEMM operands: V moves
    for name, p in (("w3", iql.flatten(w1, b1, w2, b2, w3 + d, b3)),
                    ("b2", iql.flatten(w1, b1, w2, b2 + d, w3, b3)),
                    ("b3", iql.flatten(w1, b1, w2, b2, w3, b3 + d))):
        v, _, _ = iql.value_fwd_bwd(p, x, qt, 0.5, s, h, gemm_operand=bf16)
        assert (v != base_v).all(), name

    # Q moved by 4 * 2^-12 per row moves dV by 2^-12: dz2 = dV w3 is rounded
    # back before dW2 and dh1 (so dW2, dW1 and db1 stay), while db2, dW3 and
    # db3 sum the unrounded values
    _, _, g = iql.value_fwd_bwd(flat, x, qt + 4 * d, 0.5, s, h, gemm_operand=bf16)
    for k in ("w1", "b1", "w2"):
        assert np.array_equal(g[idx[k]], base_g[idx[k]]), k
    for k in ("b2", "w3", "b3"):
        assert not np.array_equal(g[idx[k]], base_g[idx[k]]), k


def test_bf16_mode_hand_case():
    # S = 1, H = 2, B = 1, tau = 0.5, worked by hand.  z1 = h1 = 1 + 2^-8
    # (not a bf16 value: rounds to 1), so z2 = 1 + 1 = 2 per unit (the exact
    # value is 2 + 2^-7) and V = 2 w3_0 + 2 w3_1 = 2 + 2^-7.  With q = V - 1:
    # dV = 1, dz2 = w3 = (1, 2^-8), dW3 = dV h2 = (2, 2), dW2 = dz2^T r(h1) =
    # [[1, 1], [2^-8, 2^-8]], dh1 = dz2 W2 = 1 + 2^-8 per unit, which rounds
    # to 1 in dW1 = r(dz1)^T x, while db1 sums the unrounded dz1.
    e = 2.0 ** -8
    w1, b1 = np.array([[1.0], [1.0]]), np.array([e, e])
    w2, b2 = np.ones((2, 2)), np.zeros(2)
    w3, b3 = np.array([[1.0, e]]), np.array([0.0])
    flat = iql.flatten(w1, b1, w2, b2, w3, b3)
    x = np.array([[1.0]])
    v, act = iql.forward(flat, x, 1, 2, gemm_operand=bf16)
    assert v[0] == 2 + 2 * e
    qt = v - 1.0
    _, loss, g = iql.value_fwd_bwd(flat, x, qt, 0.5, 1, 2, gemm_operand=bf16)
    assert loss == 0.5
    want = iql.flatten(np.array([[1.0], [1.0]]), np.array([1 + e, 1 + e]), np.array([[1.0, 1.0], [e, e]]),
                       np.array([1.0, e]), np.array([[2.0, 2.0]]), np.array([1.0]))
    assert np.array_equal(g, want)
    # the exact oracle differs where the rounding acted
    ve, _ = iql.forward(flat, x, 1, 2)
    assert ve[0] == (2 + 2 * e) * (1 + e)


def test_bf16_mode_on_a_random_network_stays_within_first_order_rounding():
    # generic inputs: the mode rounds (results differ from the exact ones) and
    # the difference in V is within first-order bf16 rounding of every operand
    # of the two forward products (relative 2^-8 per operand and per product
    # term, 2^-9 from each operand's own rounding)
    rng = np.random.default_rng(9)
    s, h, b = 12, 16, 64
    flat = rng.uniform(-0.5, 0.5, h * s + h + h * h + h + h + 1)
    x = rng.standard_normal((b, s))
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
    v, act = iql.forward(flat, x, s, h)
    vb, _ = iql.forward(flat, x, s, h, gemm_operand=bf16)
    assert (v != vb).any()
    u = 2.0 ** -8
    dz1 = u * (np.abs(x) @ np.abs(w1).T) * 1.01
    dz2 = (u * (np.abs(act["h1"]) @ np.abs(w2).T) + (dz1 + u * np.abs(act["h1"])) @ np.abs(w2).T) * 1.01
    bound = (dz2 @ np.abs(w3).T)[:, 0]
    assert (np.abs(vb - v) <= bound).all()
