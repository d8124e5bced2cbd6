"""GPU parity: budgeted clipped SAXPY and Adam against the oracle."""
import numpy as np
import pytest
import torch

from _gpu import assert_close, dev, f32, need_gpu
from oracle import optim

pytestmark = pytest.mark.gpu

BUDGET = tuple(f32(b) for b in optim.BUDGET)


def _ctx():
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    return ofrl.Context(8, 64, 4, max_batch=1)


@pytest.mark.parametrize("n", [1, 33, 79105, 1_000_003])
@pytest.mark.parametrize("n_src", [1, 2, 4])
def test_budgeted_clip_saxpy(n, n_src):
    import offline_rl_step_gb300 as ofrl
    ctx = _ctx()
    rng = np.random.default_rng(n + n_src)
    scales = [3.0, 1e-3, 0.5, 4.0][:n_src]
    srcs = [(rng.standard_normal(n) * sc / np.sqrt(n) * 2).astype(np.float32) for sc in scales]
    alpha = [1.0, 0.5, 1.0, 2.0][:n_src]
    out = torch.empty(n, device="cuda")
    norms = torch.empty(n_src + 1, device="cuda")
    ofrl.budgeted_clip_saxpy(ctx, [dev(s) for s in srcs], BUDGET, alpha, 1.0, out, norms)
    torch.cuda.synchronize()
    rg, rn = optim.budgeted_combine(srcs, BUDGET[:n_src], alpha, 1.0)
    assert_close(norms.cpu().numpy(), rn, what="norms")
    assert_close(out.cpu().numpy(), rg, rtol=1e-4, atol=1e-5 * np.abs(rg).max(), what="combined")
    ctx.close()


@pytest.mark.parametrize("t", [1, 7])
@pytest.mark.parametrize("given_norm", [False, True])
def test_adam_step(t, given_norm):
    import offline_rl_step_gb300 as ofrl
    ctx = _ctx()
    n = 23169
    rng = np.random.default_rng(t)
    p = rng.standard_normal(n).astype(np.float32) * 0.1
    g = (rng.standard_normal(n) * 0.3).astype(np.float32)
    m = (rng.standard_normal(n) * 0.01).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    v = (np.abs(rng.standard_normal(n)) * 1e-3).astype(np.float32) if t > 1 else np.zeros(n, np.float32)
    opt = ofrl.Opt(lr=3e-4, weight_decay=1e-4, max_grad_norm=1.0)
    tp, tm, tv = dev(p), dev(m), dev(v)
    gn = torch.tensor([7.5], device="cuda") if given_norm else None
    ofrl.adam_step(ctx, tp, dev(g), tm, tv, t, opt, grad_norm=gn)
    torch.cuda.synchronize()
    norm = 7.5 if given_norm else float(np.linalg.norm(g.astype(np.float64)))
    rp, rm, rv, skipped = optim.adam(p, g, m, v, t, f32(3e-4), f32(0.9), f32(0.999), f32(1e-8), f32(1e-4),
                                     1.0, norm)
    assert skipped == 0
    assert_close(tm.cpu().numpy(), rm, what="m")
    assert_close(tv.cpu().numpy(), rv, what="v")
    assert_close(tp.cpu().numpy(), rp, what="p")
    assert ctx.poll_status()["nonfinite_grad"] == 0
    ctx.close()


def test_adam_skips_and_counts_non_finite():
    import offline_rl_step_gb300 as ofrl
    ctx = _ctx()
    n = 1000
    rng = np.random.default_rng(5)
    p = rng.standard_normal(n).astype(np.float32)
    g = rng.standard_normal(n).astype(np.float32)
    bad = rng.choice(n, 37, replace=False)
    g[bad[:20]] = np.nan
    g[bad[20:30]] = np.inf
    g[bad[30:]] = -np.inf
    m = np.full(n, 0.01, np.float32)
    v = np.full(n, 0.02, np.float32)
    tp, tm, tv = dev(p), dev(m), dev(v)
    opt = ofrl.Opt(lr=1e-3, max_grad_norm=float("inf"))
    ofrl.adam_step(ctx, tp, dev(g), tm, tv, 4, opt, grad_norm=torch.tensor([1.0], device="cuda"))
    torch.cuda.synchronize()
    rp, rm, rv, skipped = optim.adam(p, g, m, v, 4, f32(1e-3), f32(0.9), f32(0.999), f32(1e-8), 0.0,
                                     float("inf"), 1.0)
    assert skipped == 37
    assert ctx.poll_status()["nonfinite_grad"] == 37
    gp = tp.cpu().numpy()
    assert np.array_equal(gp[bad], p[bad])
    assert_close(gp, rp, what="p")
    ctx.close()


def test_budget_with_non_finite_source_follows_ieee_reading():
    import offline_rl_step_gb300 as ofrl
    ctx = _ctx()
    n = 4096
    rng = np.random.default_rng(6)
    srcs = [rng.standard_normal(n).astype(np.float32) for _ in range(3)]
    srcs[1][17] = np.nan          # NaN norm -> coefficient 1, NaN combined norm
    out = torch.empty(n, device="cuda")
    norms = torch.empty(4, device="cuda")
    ofrl.budgeted_clip_saxpy(ctx, [dev(s) for s in srcs], BUDGET, [1, 1, 1], 1.0, out, norms)
    torch.cuda.synchronize()
    rg, rn = optim.budgeted_combine(srcs, BUDGET[:3], [1, 1, 1], 1.0)
    gn = norms.cpu().numpy()
    assert np.isnan(gn[1]) and np.isnan(gn[3]) and np.isnan(rn[1]) and np.isnan(rn[3])
    go = out.cpu().numpy()
    assert np.isnan(go[17]) and np.isnan(rg[17])
    ok = np.isfinite(rg)
    assert_close(go[ok], rg[ok], what="finite elements")
    ctx.close()


def test_adam_step_weight_bound():
    import offline_rl_step_gb300 as ofrl
    ctx = _ctx()
    n = 23169
    rng = np.random.default_rng(21)
    p = (rng.standard_normal(n) * 0.1).astype(np.float32)
    g = (rng.standard_normal(n) * 0.3).astype(np.float32)
    z = np.zeros(n, np.float32)
    opt = ofrl.Opt(lr=3e-4, max_grad_norm=np.inf, weight_clamp_max_abs=0.12)
    tp, tm, tv = dev(p), dev(z), dev(z)
    ofrl.adam_step(ctx, tp, dev(g), tm, tv, 1, opt, grad_norm=torch.tensor([1.0], device="cuda"))
    torch.cuda.synchronize()
    rp, _, _, _ = optim.adam(p, g, z, z, 1, f32(3e-4), f32(0.9), f32(0.999), f32(1e-8), 0.0, np.inf, 1.0,
                             weight_clamp=f32(0.12))
    gp = tp.cpu().numpy()
    assert (np.abs(gp) <= f32(0.12)).all()
    assert ((np.abs(rp) >= f32(0.12) * (1 - 1e-7)) == (np.abs(gp) >= f32(0.12) * (1 - 1e-7))).mean() > 0.999
    assert_close(gp, rp, what="p")
    ctx.close()


@pytest.mark.parametrize("n,rate", [(1, 0.5), (23169, 0.005), (1_000_003, 1.0), (4096, 0.0)])
def test_target_ema(n, rate):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    rng = np.random.default_rng(n)
    p = rng.standard_normal(n).astype(np.float32)
    t = rng.standard_normal(n).astype(np.float32)
    tp, tt = dev(p), dev(t)
    ofrl.target_ema(tp, tt, f32(rate))
    torch.cuda.synchronize()
    ref = optim.polyak(t, p, f32(rate))
    got = tt.cpu().numpy().astype(np.float64)
    # two fp32 products and a sum: a few units in the last place of the inputs' scale
    assert (np.abs(got - ref) <= 3 * np.finfo(np.float32).eps * (np.abs(t) + np.abs(p))).all()
    if rate == 1.0:
        assert np.array_equal(tt.cpu().numpy(), p)
    if rate == 0.0:
        assert np.array_equal(tt.cpu().numpy(), t)
