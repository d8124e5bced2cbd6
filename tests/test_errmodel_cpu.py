"""CPU check of the fp32 error model used by the parity tests: an fp32
evaluation of the same network (numpy float32, its own summation order) must
stay inside the bound everywhere, and the bound must stay tight on the bulk
of the elements (it may not excuse everything)."""
import dataclasses

import numpy as np
import pytest

import synth
from _errmodel import grad_ok, value_uncertainty, within
from oracle import iql


def _fp32_fwd_bwd(flat, x, qt, tau, s, h):
    f = np.float32
    w1, b1, w2, b2, w3, b3 = [a.astype(f) for a in iql.unflatten(flat, s, h)]
    x = x[:, :s].astype(f)
    qt = qt.astype(f)
    n = x.shape[0]
    z1 = x @ w1.T + b1
    h1 = np.maximum(z1, f(0))
    z2 = h1 @ w2.T + b2
    h2 = np.maximum(z2, f(0))
    v = (h2 @ w3.T + b3)[:, 0]
    d = qt - v
    w = np.where(d >= 0, f(tau), f(1 - tau)).astype(f)
    dv = (f(-2) * w * d / f(n)).astype(f)
    dz2 = (dv[:, None] * w3) * (z2 > 0)
    dz1 = (dz2 @ w2) * (z1 > 0)
    g = np.concatenate([(dz1.T @ x).ravel(), dz1.sum(0), (dz2.T @ h1).ravel(), dz2.sum(0),
                        (dv[None, :] @ h2).ravel(), [dv.sum()]])
    return v.astype(np.float64), g.astype(np.float64)


@pytest.mark.parametrize("s,h,b,seed", [(48, 64, 256, 0), (50, 128, 4096, 1), (50, 256, 2048, 2),
                                        (50, 128, 16384, 3)])
def test_fp32_evaluation_inside_bound(s, h, b, seed):
    w = dataclasses.replace(synth.PROD, state_dim=s, hidden=h, net_seeds=(seed,))
    flat = synth.make_params(w).astype(np.float64)
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((b, s)).astype(np.float32).astype(np.float64)
    qt = (rng.standard_normal(b) * 2).astype(np.float32).astype(np.float64)
    v, g, vu, gu = value_uncertainty(flat, x, qt, 0.7, s, h)
    v32, g32 = _fp32_fwd_bwd(flat, x, qt, 0.7, s, h)
    assert (np.abs(v32 - v) <= vu).all()
    assert (np.abs(g32 - g) <= gu).all()
    assert within(g32, g, gu, 1e-4, 1e-5).all()
    ok, _, rel = grad_ok(g32, g, gu)
    assert ok and rel < 1e-5
    # tight on the bulk: the bound is a small fraction of |g| for most elements
    big = np.abs(g) > 1e-6
    r = gu[big] / np.abs(g[big])
    assert np.median(r) < 5e-3
    assert np.quantile(r, 0.95) < 0.1


@pytest.mark.parametrize("mistake", ["sign", "shift", "scale"])
def test_planted_mistakes_are_not_excused(mistake):
    # a plausible kernel bug in any one tensor of the gradient must fall
    # outside both the tolerance and the fp32 bound on most of its elements
    s, h, b = 50, 128, 4096
    w = dataclasses.replace(synth.PROD, state_dim=s, hidden=h)
    flat = synth.make_params(w).astype(np.float64)
    rng = np.random.default_rng(11)
    x = rng.standard_normal((b, s))
    qt = rng.standard_normal(b) * 2
    _, g, _, gu = value_uncertainty(flat, x, qt, 0.7, s, h)
    seg = iql.flatten(*[np.full(np.shape(a), i) for i, a in enumerate(iql.unflatten(np.zeros(len(flat)), s, h))])
    for t in range(6):
        m = seg == t
        bad = g.copy()
        if mistake == "sign":
            bad[m] = -bad[m]
        elif mistake == "shift":
            bad[m] = np.roll(bad[m], 1)
        else:
            bad[m] = bad[m] * 1.1
        if m.sum() == 1 and mistake == "shift":
            continue
        assert not grad_ok(bad, g, gu)[0], (t, mistake)
        if m.sum() > 1 and mistake != "scale":
            caught = ~within(bad[m], g[m], gu[m], 1e-4, 1e-5)
            assert caught.mean() > 0.9, (t, mistake, caught.mean())


def test_weight_difference_widens_the_bound():
    s, h, b = 50, 128, 512
    w = dataclasses.replace(synth.PROD, state_dim=s, hidden=h)
    flat = synth.make_params(w).astype(np.float64)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((b, s))
    qt = rng.standard_normal(b) * 2
    dp = np.abs(flat) * 1e-4
    v, g, vu, gu = value_uncertainty(flat, x, qt, 0.7, s, h)
    v2, g2, vu2, gu2 = value_uncertainty(flat, x, qt, 0.7, s, h, dparams=dp)
    assert (gu2 >= gu).all() and (vu2 >= vu).all()
    # the perturbed network's exact result is inside the widened bound
    vp, _, gp = iql.value_fwd_bwd(flat + dp * np.sign(rng.standard_normal(len(flat))), x, qt, 0.7, s, h)
    assert (np.abs(vp - v) <= vu2).all()
    assert (np.abs(gp - g) <= gu2).all()
