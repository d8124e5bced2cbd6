"""Pins for the oracle's budgeted clipping and Adam."""
import os

import numpy as np
import pytest
import torch

from oracle import optim

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _budget():
    vals = {}
    with open(os.path.join(GOLDEN, "constants.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return (vals["budget_primary"], vals["budget_cql"], vals["budget_iqn"], vals["budget_ens"])


def test_budget_fractions_match_pages_and_sum_to_one():
    assert optim.BUDGET == _budget()
    assert sum(optim.BUDGET) == pytest.approx(1.0, abs=1e-15)


@pytest.mark.parametrize("scale", [1e-3, 0.5, 1.0, 3.0, 1e4])
def test_single_source_norm_is_min_of_norm_and_budget(scale):
    g = np.random.default_rng(1).standard_normal(1000)
    g *= scale / np.linalg.norm(g)
    out, norms = optim.budgeted_combine([g], (0.7,), (1.0,), 1.0)
    assert norms[0] == pytest.approx(scale, rel=1e-14)
    assert norms[-1] == pytest.approx(min(scale, 0.7), rel=1e-13)
    assert np.linalg.norm(out) == pytest.approx(min(scale, 0.7), rel=1e-13)


def test_sources_below_budget_add_unchanged():
    rng = np.random.default_rng(2)
    srcs = []
    for f in optim.BUDGET:
        s = rng.standard_normal(500)
        srcs.append(s * (0.5 * f / np.linalg.norm(s)))
    out, _ = optim.budgeted_combine(srcs, optim.BUDGET, (1, 1, 1, 1), 1.0)
    np.testing.assert_array_equal(out, srcs[0] + srcs[1] + srcs[2] + srcs[3])


@pytest.mark.parametrize("mgn", [0.1, 1.0, 7.5])
def test_combined_norm_never_exceeds_max_grad_norm(mgn):
    rng = np.random.default_rng(3)
    for _ in range(50):
        scales = 10.0 ** rng.uniform(-3, 3, size=4)
        srcs = [rng.standard_normal(300) * sc for sc in scales]
        out, norms = optim.budgeted_combine(srcs, optim.BUDGET, (1, 1, 1, 1), mgn)
        assert norms[-1] <= mgn * (1 + 1e-12)
        # the per-source clips are exactly the budgets when the source is above it
        for k in range(4):
            c = optim.BUDGET[k] * mgn
            assert optim.clip_scale(norms[k], c) * norms[k] == pytest.approx(min(norms[k], c), rel=1e-13)


def test_clip_scale_formula_edge_cases():
    assert optim.clip_scale(0.0, 1.0) == 1.0
    assert optim.clip_scale(0.5, 1.0) == 1.0
    assert optim.clip_scale(1.0, 1.0) == 1.0     # strict '>'
    assert optim.clip_scale(4.0, 1.0) == 0.25
    assert optim.clip_scale(float("nan"), 1.0) == 1.0
    assert optim.clip_scale(float("inf"), 1.0) == 0.0


def test_adam_first_step_closed_form():
    # from m = v = 0 at t = 1: m_hat = g, v_hat = g^2, so
    # p1 = p0 - lr * (g / (|g| + eps) + wd * p0)
    rng = np.random.default_rng(4)
    p0 = rng.standard_normal(1000)
    g = rng.standard_normal(1000) * 0.1
    lr, eps, wd = 3e-4, 1e-8, 1e-4
    p, m, v, skipped = optim.adam(p0, g, np.zeros(1000), np.zeros(1000), 1, lr, 0.9, 0.999, eps,
                                  wd, 1e9, np.linalg.norm(g))
    assert skipped == 0
    np.testing.assert_allclose(p, p0 - lr * (g / (np.abs(g) + eps) + wd * p0), rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-14)
    np.testing.assert_allclose(v, 0.001 * g * g, rtol=1e-12)


def test_adam_constant_gradient_closed_form():
    # a constant gradient keeps m_hat = g and v_hat = g^2 at every t
    g = np.array([0.3, -2.0, 1e-3])
    p = np.zeros(3)
    m = np.zeros(3)
    v = np.zeros(3)
    lr, eps = 1e-2, 1e-8
    for t in range(1, 11):
        p, m, v, _ = optim.adam(p, g, m, v, t, lr, 0.9, 0.999, eps, 0.0, 1e9, 1.0)
        np.testing.assert_allclose(m / (1 - 0.9 ** t), g, rtol=1e-12)
        np.testing.assert_allclose(v / (1 - 0.999 ** t), g * g, rtol=1e-11)
    np.testing.assert_allclose(p, -10 * lr * g / (np.abs(g) + eps), rtol=1e-10)


def test_adam_matches_torch_adamw():
    rng = np.random.default_rng(5)
    n = 257
    p0 = rng.standard_normal(n)
    lr, b1, b2, eps, wd = 3e-4, 0.9, 0.999, 1e-8, 1e-4
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 31):
        g = rng.standard_normal(n)
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v, _ = optim.adam(p, g, m, v, t, lr, b1, b2, eps, wd, 1e9, np.linalg.norm(g))
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-12, atol=1e-15)


def test_adam_safety_clip_matches_torch_clip_grad_norm():
    rng = np.random.default_rng(6)
    n = 100
    p0 = rng.standard_normal(n)
    g = rng.standard_normal(n) * 5
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    tp.grad = torch.tensor(g, dtype=torch.float64)
    torch.nn.utils.clip_grad_norm_([tp], max_norm=1.0)   # scale 1 / (||g|| + 1e-6)
    opt = torch.optim.AdamW([tp], lr=1e-2, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0)
    opt.step()
    p, _, _, _ = optim.adam(p0, g, np.zeros(n), np.zeros(n), 1, 1e-2, 0.9, 0.999, 1e-8, 0.0, 1.0,
                            np.linalg.norm(g))
    # first step is ~ lr * sign(g) either way; the clip only changes the eps ratio
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=0, atol=1e-9)
    # and the moments follow the clipped gradient
    _, m, _, _ = optim.adam(p0, g, np.zeros(n), np.zeros(n), 1, 1e-2, 0.9, 0.999, 1e-8, 0.0, 1.0,
                            np.linalg.norm(g))
    np.testing.assert_allclose(m, 0.1 * g / np.linalg.norm(g), rtol=1e-12)


def test_adam_skips_non_finite_elements():
    p0 = np.arange(6, dtype=np.float64)
    g = np.array([1.0, np.nan, -1.0, np.inf, -np.inf, 0.5])
    m0 = np.full(6, 0.25)
    v0 = np.full(6, 0.5)
    p, m, v, skipped = optim.adam(p0, g, m0, v0, 3, 1e-3, 0.9, 0.999, 1e-8, 0.0, np.inf, np.nan)
    assert skipped == 3
    for i in (1, 3, 4):
        assert p[i] == p0[i] and m[i] == m0[i] and v[i] == v0[i]
    for i in (0, 2, 5):
        assert p[i] != p0[i]


# ---- isfinite guard on the sources, weight bound, Polyak target -------------

def _sources(seed=11, n=4, p=257, scales=(3.0, 1.0, 0.5, 2.0)):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(p) * s for s in scales[:n]]


def test_sanitize_is_identity_on_finite_sources():
    srcs = _sources()
    g0, n0 = optim.budgeted_combine(srcs, optim.BUDGET, (1, 1, 1, 1), 1.0)
    g1, n1 = optim.budgeted_combine(srcs, optim.BUDGET, (1, 1, 1, 1), 1.0, sanitize_sources=True)
    assert np.array_equal(g0, g1) and np.array_equal(n0, n1)


def test_sanitized_sources_keep_the_budget_bound():
    # NaN and +-inf planted in every source: the guarded combination stays
    # finite and inside the budget sum (sum f_k mgn = mgn)
    srcs = _sources(seed=12)
    for k, s in enumerate(srcs):
        s[[k, 40 + k, 99]] = [np.nan, np.inf, -np.inf]
    g, norms = optim.budgeted_combine(srcs, optim.BUDGET, (1, 1, 1, 1), 1.0, sanitize_sources=True)
    assert np.isfinite(g).all() and np.isfinite(norms).all()
    assert norms[-1] <= 1.0 * (1 + 1e-12)
    # without the guard the planted values reach the sum
    g_raw, _ = optim.budgeted_combine(srcs, optim.BUDGET, (1, 1, 1, 1), 1.0)
    assert not np.isfinite(g_raw).all()


def test_an_all_nonfinite_source_contributes_nothing():
    srcs = _sources(seed=13, n=3)
    bad = np.full_like(srcs[2], np.nan)
    g, norms = optim.budgeted_combine([srcs[0], srcs[1], bad], optim.BUDGET[:3], (1, 1, 1), 1.0,
                                      sanitize_sources=True)
    g2, _ = optim.budgeted_combine(srcs[:2], optim.BUDGET[:2], (1, 1), 1.0)
    assert norms[2] == 0.0
    assert np.allclose(g, g2, rtol=0, atol=0)


def test_weight_bound_closed_form():
    # first step from m = v = 0 moves p by ~lr sign(g); 0.99995 + 3e-4 is
    # past the bound 1.0, so the weight ends exactly on it
    p = np.array([0.99995, -0.5, 0.2])
    g = np.array([-1.0, 1.0, 1e-3])
    z = np.zeros(3)
    pc, _, _, _ = optim.adam(p, g, z, z, 1, 3e-4, 0.9, 0.999, 1e-8, 0.0, np.inf, 0.0, weight_clamp=1.0)
    pu, _, _, _ = optim.adam(p, g, z, z, 1, 3e-4, 0.9, 0.999, 1e-8, 0.0, np.inf, 0.0)
    assert pc[0] == 1.0 and pu[0] > 1.0
    assert np.array_equal(pc[1:], pu[1:])
    assert (np.abs(pc) <= 1.0).all()


def test_weight_bound_leaves_skipped_elements_alone():
    p = np.array([5.0, 0.1])
    g = np.array([np.nan, 1.0])
    z = np.zeros(2)
    pc, _, _, skipped = optim.adam(p, g, z, z, 1, 3e-4, 0.9, 0.999, 1e-8, 0.0, np.inf, 0.0, weight_clamp=1.0)
    assert skipped == 1 and pc[0] == 5.0


def test_polyak_rates_and_closed_form():
    rng = np.random.default_rng(14)
    t0, p = rng.standard_normal(50), rng.standard_normal(50)
    assert np.array_equal(optim.polyak(t0, p, 1.0), p)
    assert np.array_equal(optim.polyak(t0, p, 0.0), t0)
    # k updates toward a fixed p: target_k = p + (1 - r)^k (target_0 - p)
    t, r = t0.copy(), 0.05
    for _ in range(20):
        t = optim.polyak(t, p, r)
    assert np.allclose(t, p + (1 - r) ** 20 * (t0 - p), rtol=1e-13, atol=1e-14)
