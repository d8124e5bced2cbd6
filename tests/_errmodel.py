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
    full.

The tests accept a CUDA value inside the benchmark spec's tolerance or inside
this bound; a CPU test checks that an independent fp32 evaluation stays
inside it and that it stays tight on the bulk of the elements.
"""
import numpy as np

from oracle import iql

U = 2.0 ** -24
LAM = 8.0


def _rnd(abs_sum, n):
    return LAM * U * np.sqrt(n) * abs_sum


def _rss(unc, w):
    """Uncertainty of unc-perturbed inputs through y = x W^T (independent errors)."""
    return np.sqrt((unc * unc) @ (w * w).T)


def value_uncertainty(flat, x, qt, tau, state_dim, hidden, batch=None, dparams=None):
    """Per-element uncertainty of (V, grad) of iql.value_fwd_bwd in fp32.

    x: states [B, >= S]; qt: Q(s, a_taken) [B]; dparams: |p_cuda - p_oracle|
    per flat parameter (the two sides' weight difference), or None.
    Returns (v, grad, v_unc, grad_unc).

    Every per-row quantity carries a random part (rounding, independent from
    row to row, so it adds in quadrature over the batch sums) and a
    systematic part (weight differences and ReLU-mask flips, which add
    linearly).
    """
    s, h = state_dim, hidden
    w1, b1, w2, b2, w3, b3 = iql.unflatten(flat, s, h)
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
    z1s = ax @ dw1.T + db1
    amb1 = np.abs(z1) <= z1r + z1s
    on1 = (z1 > 0.0) | amb1
    h1r, h1s = z1r * on1, z1s * on1
    h1abs = np.abs(h1) + h1r + h1s
    z2r = _rnd(h1abs @ aw2.T + np.abs(b2), h + 1) + _rss(h1r, aw2)
    z2s = h1s @ aw2.T + h1abs @ dw2.T + db2
    amb2 = np.abs(z2) <= z2r + z2s
    on2 = (z2 > 0.0) | amb2
    h2r, h2s = z2r * on2, z2s * on2
    h2abs = np.abs(h2) + h2r + h2s
    vr = (_rnd(h2abs @ aw3.T + np.abs(b3), h + 1) + _rss(h2r, aw3))[:, 0]
    vs = (h2s @ aw3.T + h2abs @ dw3.T + db3)[:, 0]

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
    dz2s = dvs[:, None] * aw3 * on2 + adv[:, None] * dw3 * on2 + amb2 * (adv[:, None] * aw3)
    adz2x = adz2 + dz2r + dz2s                         # any admissible |dz2|
    dh1 = dz2 @ w2
    dh1r = _rnd(adz2 @ aw2, h) + np.sqrt(sq(dz2r) @ sq(aw2))
    dh1s = dz2s @ aw2 + adz2x @ dw2
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
    u_w1 = bsum(adz1, dz1r, dz1s, ax, zx, zx)
    u_b1 = bsum(adz1, dz1r, dz1s, one, zero1, zero1)[:, 0]
    u_w2 = bsum(adz2, dz2r, dz2s, np.abs(h1), h1r, h1s)
    u_b2 = bsum(adz2, dz2r, dz2s, one, zero1, zero1)[:, 0]
    u_w3 = bsum(adv[:, None], dvr[:, None], dvs[:, None], np.abs(h2), h2r, h2s)
    u_b3 = bsum(adv[:, None], dvr[:, None], dvs[:, None], one, zero1, zero1)[:, 0]
    grad = iql.backward(flat, act, dv, s, h)
    return v, grad, vr + vs, iql.flatten(u_w1, u_b1, u_w2, u_b2, u_w3, u_b3)


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
    """Element-wise: inside the benchmark spec's tolerance or inside the fp32 bound."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    return (err <= atol + rtol * np.abs(ref)) | (err <= unc)
