"""How far an fp32 evaluation of the V forward/backward may land from the
exact (fp64) value, element by element.

Used by the parity tests to tell "the CUDA path computed something else"
from "fp32 arithmetic does not fix this element".  Three effects are bounded
from quantities of the oracle's fp64 evaluation and from the known
difference between the two sides' weights (zero on the first step):

  * rounding: a sum of n products evaluated in fp32 in any order is off by
    about sqrt(n) u times the sum of |terms| (probabilistic rounding-error
    analysis, Higham & Mary, SIAM J. Sci. Comput. 2019); LAM is the safety
    factor over that growth, u = 2^-24;
  * propagated uncertainty: pre-activations, V and dL/dV = -2 w (q - V) / B
    inherit the upstream uncertainty (independent errors add in quadrature
    through a weight matrix); the expectile weight may switch where |q - V|
    is inside it;
  * ReLU masks: where |z| is inside z's own uncertainty, 1[z > 0] = 0 and 1
    are both fp32-correct; the contribution of every such entry is added in
    full;
  * split products: the tensor-core kernels form fp32 products from a
    three-term bf16 split (x = x0 + x1 + x2 with |x - x0| <= 2^-9 |x|, so
    |x1| <= 2^-9 |x| and |x2| <= 2^-18 |x|), and their backward GEMMs (dh1
    and the weight gradients) take only the three leading products x1 y0 +
    x0 y1 + x0 y0: the dropped x2 y0 + x1 y1 + x0 y2 (and smaller) are
    within SPLIT_REL = 3.1 * 2^-18 of |x y|, added linearly to dh1 (so to
    dz1) and to dW1, db1 and dW2.

The tests accept a CUDA value inside the stated tolerance (1e-4 relative /
1e-5 absolute) or inside this bound; a CPU test checks that an independent fp32 evaluation stays
inside it and that it stays tight on the bulk of the elements.
"""
import numpy as np

from oracle import iql
from oracle.precision import bf16

U = 2.0 ** -24
LAM = 8.0
SPLIT_REL = 3.1 * 2.0 ** -18


def _rnd(abs_sum, n):
    return LAM * U * np.sqrt(n) * abs_sum


def _rss(unc, w):
    """Uncertainty of unc-perturbed inputs through y = x W^T (independent errors)."""
    return np.sqrt((unc * unc) @ (w * w).T)


def value_uncertainty(flat, x, qt, tau, state_dim, hidden, batch=None, dparams=None, info=None):
    """Per-element uncertainty of (V, grad) of iql.value_fwd_bwd in fp32.

    x: states [B, >= S]; qt: Q(s, a_taken) [B]; dparams: |p_cuda - p_oracle|
    per flat parameter (the two sides' weight difference), or None.
    Returns (v, grad, v_unc, grad_unc); with a dict `info`, also stores in it
    the number of ReLU masks decided inside their own uncertainty
    ("ambiguous_masks").

    Every per-row quantity carries a random part (rounding, independent from
    row to row, so it adds in quadrature over the batch sums) and a
    systematic part (weight differences and ReLU-mask flips, which add
    linearly).
    """
    s, h = state_dim, hidden
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
    same = dparams is None or not np.any(dparams)   # both sides evaluate the same weights
    if dparams is None:
        dparams = np.zeros(len(flat))
    dw1, db1, dw2, db2, dw3, db3 = iql.unflatten(np.abs(dparams), s, h)
    x = np.asarray(x, dtype=np.float64)[:, :s]
    qt = np.asarray(qt, dtype=np.float64)
    n = x.shape[0] if batch is None else batch
    v, act = iql.forward(flat, x, s, h)
    z1, h1, z2, h2 = act["z1"], act["h1"], act["z2"], act["h2"]
    ax = np.abs(x)
    aw1, aw2, aw3 = np.abs(w1), np.abs(w2), np.abs(w3)
    sq = lambda a: a * a

    # ---- forward: random (r) and systematic (s) uncertainty per row ----
    z1r = _rnd(ax @ aw1.T + np.abs(b1), s + 1)
    z1s = 0.0 if same else ax @ dw1.T + db1
    amb1 = np.abs(z1) <= z1r + z1s
    on1 = (z1 > 0.0) | amb1
    h1r, h1s = z1r * on1, z1s * on1
    h1abs = np.abs(h1) + h1r + h1s
    z2r = _rnd(h1abs @ aw2.T + np.abs(b2), h + 1) + _rss(h1r, aw2)
    z2s = 0.0 if same else h1s @ aw2.T + h1abs @ dw2.T + db2
    amb2 = np.abs(z2) <= z2r + z2s
    on2 = (z2 > 0.0) | amb2
    h2r, h2s = z2r * on2, z2s * on2
    h2abs = np.abs(h2) + h2r + h2s
    vr = (_rnd(h2abs @ aw3.T + np.abs(b3), h + 1) + _rss(h2r, aw3))[:, 0]
    vs = 0.0 if same else (h2s @ aw3.T + h2abs @ dw3.T + db3)[:, 0]

    # ---- dL/dV = -2 w (q - V) / B ----
    d = qt - v
    w = np.where(d >= 0.0, tau, 1.0 - tau)
    dv = -2.0 * w * d / n
    adv = np.abs(dv)
    wmax = max(tau, 1.0 - tau)
    dvr = 2.0 * wmax * (vr + _rnd(np.abs(qt) + np.abs(v), 2)) / n + _rnd(adv, 3)
    du = vr + vs + _rnd(np.abs(qt) + np.abs(v), 2)
    dvs = 2.0 * wmax * vs / n + np.where(np.abs(d) <= du, 2.0 * abs(2.0 * tau - 1.0) * (np.abs(d) + du) / n, 0.0)

    # ---- backward rows ----
    dz2 = (dv[:, None] * w3) * (z2 > 0.0)
    adz2 = np.abs(dz2)
    dz2r = dvr[:, None] * aw3 * on2 + _rnd(adz2, 1)
    dz2s = amb2 * (adv[:, None] * aw3)
    if not same:
        dz2s = dz2s + dvs[:, None] * aw3 * on2 + adv[:, None] * dw3 * on2
    adz2x = adz2 + dz2r + dz2s                         # any admissible |dz2|
    dh1 = dz2 @ w2
    dh1r = _rnd(adz2 @ aw2, h) + np.sqrt(sq(dz2r) @ sq(aw2))
    dh1s = (dz2s @ aw2 if same else dz2s @ aw2 + adz2x @ dw2) + SPLIT_REL * (adz2 @ aw2)
    adh1x = np.abs(dh1) + dh1r + dh1s
    dz1 = dh1 * (z1 > 0.0)
    adz1 = np.abs(dz1)
    dz1r = dh1r * on1
    dz1s = dh1s * on1 + amb1 * adh1x

    # ---- batch sums: rounding of the sum, random in quadrature, systematic linearly ----
    def bsum(a_abs, ar, as_, xa, xr, xs):
        """Uncertainty of sum_r a[r, i] * x[r, k] given both factors' uncertainties."""
        rounding = _rnd(a_abs.T @ xa, n)
        rand = np.sqrt(sq(ar).T @ sq(xa) + sq(a_abs).T @ sq(xr))
        syst = as_.T @ (xa + xr + xs) + (a_abs + ar).T @ xs
        return rounding + rand + syst

    one = np.ones((x.shape[0], 1))
    zero1 = np.zeros((x.shape[0], 1))
    zx = np.zeros_like(ax)
    u_w1 = bsum(adz1, dz1r, dz1s, ax, zx, zx) + SPLIT_REL * (adz1.T @ ax)
    u_b1 = bsum(adz1, dz1r, dz1s, one, zero1, zero1)[:, 0] + SPLIT_REL * adz1.sum(axis=0)
    u_w2 = bsum(adz2, dz2r, dz2s, np.abs(h1), h1r, h1s) + SPLIT_REL * (adz2.T @ np.abs(h1))
    u_b2 = bsum(adz2, dz2r, dz2s, one, zero1, zero1)[:, 0]
    u_w3 = bsum(adv[:, None], dvr[:, None], dvs[:, None], np.abs(h2), h2r, h2s)
    u_b3 = bsum(adv[:, None], dvr[:, None], dvs[:, None], one, zero1, zero1)[:, 0]
    grad = iql.backward(flat, act, dv, s, h)
    if info is not None:
        info["ambiguous_masks"] = int(amb1.sum() + amb2.sum())
    return v, grad, vr + vs, iql.flatten(u_w1, u_b1, u_w2, u_b2, u_w3, u_b3)


def _rounding_spread(a, au):
    """Largest difference between the bf16 rounding of a value in [a - au,
    a + au] and the rounding of a (rounding is monotone: the ends bound it)."""
    r = bf16(a)
    return np.maximum(bf16(a + au) - r, r - bf16(a - au))


def _ulp_bf16(a):
    """Spacing of the bf16 values around |a| (the step of one rounding flip)."""
    _, e = np.frexp(np.abs(a))
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


def bf16_uncertainty(flat, x, qt, tau, state_dim, hidden, batch=None):
    """Per-element bound on how far an fp32 evaluation of the bf16-operand
    mode may land from the oracle's (iql.forward / iql.backward with
    gemm_operand=bf16).  Returns (v_unc [B], grad_unc [P]).

    The fp32 evaluation sums the products of the same bf16 operands in fp32
    (X, W1, W2 are fp32 values on both sides, so their roundings agree) and
    rounds h1, dz2 and dz1 to bf16 from its own fp32 values.  As in
    value_uncertainty, every per-row quantity carries a random part, which
    adds in quadrature through a weight matrix and over the batch sums, and
    a systematic part, which adds linearly:
      * random: fp32 summation (LAM sqrt(n) u times the sum of |terms|), and
        the bf16 rounding of an operand whose fp32 value may lie anywhere in
        its random interval: the largest difference between an admissible
        rounding and the oracle's (_rounding_spread), nonzero where a
        rounding midpoint lies inside the interval (either neighbour is then
        correct, and which one depends on the summation's rounding noise);
      * systematic: ReLU masks and the expectile weight decided inside their
        own uncertainty (the entry's contribution in full, plus one bf16 step
        where the entry is a rounded operand);
      * db1 as the sum of the rounded dz1 (the tensor-core kernels take it
        from the dW1 contraction's ones column): the exact offset
        |sum_rows (bf16(dz1) - dz1)|.
    """
    s, h = state_dim, hidden
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
    xr = bf16(np.asarray(x, dtype=np.float64)[:, :s])
    qt = np.asarray(qt, dtype=np.float64)
    n = xr.shape[0] if batch is None else batch
    w1r, w2r = bf16(w1), bf16(w2)
    axr, aw2, aw3 = np.abs(xr), np.abs(w2r), np.abs(w3)
    sq = lambda a: a * a

    # ---- forward (random parts only: both sides use the same weights) ----
    z1 = xr @ w1r.T + b1
    z1r = _rnd(axr @ np.abs(w1r).T + np.abs(b1), s + 1)
    amb1 = np.abs(z1) <= z1r
    on1 = (z1 > 0.0) | amb1
    h1r = bf16(np.maximum(z1, 0.0))
    hi = np.where(on1, bf16(np.maximum(z1, 0.0) + z1r), 0.0)
    lo = np.where(on1, bf16(np.maximum(z1 - z1r, 0.0)), 0.0)
    h1f = np.maximum(hi - h1r, h1r - lo)         # any admissible bf16(h1) minus the oracle's
    z2 = h1r @ w2r.T + b2
    z2r = _rnd(np.abs(h1r) @ aw2.T + np.abs(b2), h + 1) + np.sqrt(sq(h1f) @ sq(aw2).T)
    amb2 = np.abs(z2) <= z2r
    on2 = (z2 > 0.0) | amb2
    h2 = np.maximum(z2, 0.0)
    h2r = z2r * on2
    v = (h2 @ w3.T + b3)[:, 0]
    # V: one flipped h1_j moves every z2_i of its row together, so its effect
    # on V is bounded by |h1 flip_j| sum_i |w3_i W2_ij| (active units), and
    # flips of different j are independent; masks inside z2's uncertainty
    # add their entry in full
    c = (on2 * aw3) @ aw2
    vr = (_rnd(np.abs(h2) @ aw3.T + np.abs(b3), h + 1)[:, 0] + _rnd(np.abs(h1r) @ aw2.T + np.abs(b2), h + 1) @ aw3[0]
          + np.sqrt((sq(h1f) * sq(c)).sum(axis=1)) + (amb2 * (np.abs(z2) + z2r)) @ aw3[0])

    # ---- dL/dV = -2 w (q - V) / B ----
    d = qt - v
    wgt = np.where(d >= 0.0, tau, 1.0 - tau)
    dv = -2.0 * wgt * d / n
    adv = np.abs(dv)
    du = vr + _rnd(np.abs(qt) + np.abs(v), 2)
    dvr = 2.0 * max(tau, 1.0 - tau) * du / n + _rnd(adv, 3)
    dvs = np.where(np.abs(d) <= du, 2.0 * abs(2.0 * tau - 1.0) * (np.abs(d) + du) / n, 0.0)

    # ---- backward rows ----
    dz2 = dv[:, None] * w3 * (z2 > 0.0)
    dz2r = dvr[:, None] * aw3 * on2 + _rnd(np.abs(dz2), 1)
    dz2s = amb2 * (adv[:, None] * aw3) + dvs[:, None] * aw3 * on2
    dz2q = bf16(dz2)
    dz2qr = _rounding_spread(dz2, dz2r)
    dz2qs = dz2s + (dz2s > 0.0) * _ulp_bf16(np.abs(dz2) + dz2s)
    dh1 = dz2q @ w2r
    dh1r = _rnd(np.abs(dz2q) @ aw2, h) + np.sqrt(sq(dz2qr) @ sq(aw2))
    dh1s = dz2qs @ aw2
    dz1 = dh1 * (z1 > 0.0)
    dz1r = dh1r * on1
    dz1s = dh1s * on1 + amb1 * (np.abs(dh1) + dh1r + dh1s)
    dz1q = bf16(dz1)
    dz1qr = _rounding_spread(dz1, dz1r)
    dz1qs = dz1s + (dz1s > 0.0) * _ulp_bf16(np.abs(dz1) + dz1s)

    # ---- batch sums: rounding of the sum, random in quadrature, systematic linearly ----
    def bsum(a_abs, ar, as_, xa, xr_, xs):
        """Uncertainty of sum_r a[r, i] * x[r, k] given both factors' uncertainties."""
        return (_rnd(a_abs.T @ xa, n) + np.sqrt(sq(ar).T @ sq(xa) + sq(a_abs).T @ sq(xr_))
                + as_.T @ (xa + xr_ + xs) + (a_abs + ar).T @ xs)

    one = np.ones((xr.shape[0], 1))
    zero1 = np.zeros((xr.shape[0], 1))
    zx = np.zeros_like(axr)
    u_w1 = bsum(np.abs(dz1q), dz1qr, dz1qs, axr, zx, zx)
    u_b1 = (bsum(np.abs(dz1), dz1r, dz1s, one, zero1, zero1)[:, 0] + np.abs((dz1q - dz1).sum(axis=0))
            + np.sqrt(sq(dz1qr).sum(axis=0)) + dz1qs.sum(axis=0))
    u_w2 = bsum(np.abs(dz2q), dz2qr, dz2qs, np.abs(h1r), h1f, np.zeros_like(h1r))
    u_b2 = bsum(np.abs(dz2), dz2r, dz2s, one, zero1, zero1)[:, 0]
    u_w3 = bsum(adv[:, None], dvr[:, None], dvs[:, None], np.abs(h2), h2r, np.zeros_like(h2))
    u_b3 = bsum(adv[:, None], dvr[:, None], dvs[:, None], one, zero1, zero1)[:, 0]
    return vr, iql.flatten(u_w1, u_b1, u_w2, u_b2, u_w3, u_b3)


def bf16_value_uncertainty(flat, x, state_dim, hidden):
    """The V part of bf16_uncertainty (V does not depend on Q)."""
    b = np.asarray(x).shape[0]
    return bf16_uncertainty(flat, x, np.zeros(b), 0.5, state_dim, hidden)[0]


def grad_ok(gpu, ref, unc, rtol=1e-4, atol=1e-5, norm_rtol=1e-4):
    """Element-wise inside the tolerance or the fp32 bound, and norm-wise close.

    The norm-wise check measures the error beyond each element's fp32 bound
    (max(|gpu - ref| - unc, 0)), so a ReLU mask that fp32 decides the other
    way (a legitimate result) does not count, while a systematic error (a
    wrong sign, index or scale) does.  Returns (ok, number of elements outside
    the tolerance but inside the bound, relative norm of the excess).
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    tol = err <= atol + rtol * np.abs(ref)
    bnd = err <= unc
    excess = np.maximum(err - unc, 0.0)
    rel = float(np.linalg.norm(excess) / max(np.linalg.norm(ref), 1e-300))
    return bool((tol | bnd).all() and rel <= norm_rtol), int((~tol & bnd).sum()), rel


def within(gpu, ref, unc, rtol, atol):
    """Element-wise: inside the stated tolerance (rtol / atol) or inside the fp32 bound."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    return (err <= atol + rtol * np.abs(ref)) | (err <= unc)
