"""GPU parity: V forward/backward, expectile loss and policy against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from _errmodel import bf16_uncertainty, bf16_value_uncertainty, grad_ok, value_uncertainty, within
from _gpu import (ATOL, BF16_RTOL, RTOL, argmax_check, assert_close, bf16_grad_check, dev, f32, need_gpu)
from oracle.precision import bf16
from oracle import iql

pytestmark = pytest.mark.gpu


def _fwd_bwd(s, h, b, tau, prec="fp32", seed=0, stride=None, path=None):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    w = dataclasses.replace(synth.PROD, state_dim=s, hidden=h, net_seeds=(seed + 7,))
    params = synth.make_params(w)
    rng = np.random.default_rng(seed)
    st = stride or ((s + 7) & ~7)
    x = np.zeros((b, st), dtype=np.float32)
    x[:, :s] = rng.standard_normal((b, s))
    qt = (rng.standard_normal(b) * 2).astype(np.float32)
    ctx = ofrl.Context(s, h, 5, prec, max_batch=b)
    if path is not None:
        ctx.select_vnet_path(path)
    v = torch.empty(b, device="cuda")
    loss = torch.empty(1, device="cuda")
    grad = torch.empty(w.n_params, device="cuda")
    ofrl.iql_value_fwd_bwd(ctx, dev(params), dev(x), dev(qt), tau, v, loss, grad)
    torch.cuda.synchronize()
    ctx.close()
    got = (v.cpu().numpy(), float(loss.cpu()[0]), grad.cpu().numpy())
    if prec == "bf16":
        return got, (params.astype(np.float64), x, qt.astype(np.float64))
    rv, rgrad, vu, gu = value_uncertainty(params.astype(np.float64), x, qt, f32(tau), s, h)
    rloss = iql.value_fwd_bwd(params, x, qt, f32(tau), s, h)[1]
    return got, (rv, rloss, rgrad, vu, gu)


@pytest.mark.parametrize("s,h,b", [(48, 64, 256), (50, 128, 16384), (50, 128, 300), (50, 256, 200),
                                   (50, 256, 16384), (7, 64, 1), (64, 128, 129), (63, 128, 1000),
                                   (50, 128, 40000), (64, 128, 40000), (64, 64, 40000)])
def test_value_fwd_bwd_fp32(s, h, b):
    # B = 40000: 313 tiles, so the fused kernel's CTAs run two or three tiles
    # each and build the state tiles themselves (no relabel images), for G1
    # and again for G5; S = 64 leaves no ones column, so db1 comes from
    # column sums (at H = 64 only the warps of the 64 units' columns run)
    (v, loss, g), (rv, rl, rg, vu, gu) = _fwd_bwd(s, h, b, 0.7, seed=s + h + b)
    assert within(v, rv, vu, RTOL, ATOL).all(), "V outside tolerance and fp32 bound"
    assert_close(loss, rl, what="loss")
    ok, n_bound, rel = grad_ok(g, rg, gu)
    assert ok, f"gradient outside tolerance and fp32 bound (norm rel {rel:.3g}, {n_bound} by bound)"


@pytest.mark.parametrize("s,h,b,path", [(50, 128, 1000, "tc_layered"), (63, 128, 300, "tc_layered"),
                                        (1, 256, 129, "tc_layered"), (50, 256, 1000, "cuda_cores"),
                                        (48, 64, 256, "cuda_cores"), (50, 64, 16384, "tc_fused")])
def test_value_fwd_bwd_each_path(s, h, b, path):
    # the implementations the default choice does not take for these shapes
    (v, loss, g), (rv, rl, rg, vu, gu) = _fwd_bwd(s, h, b, 0.7, seed=s + h + b, path=path)
    assert within(v, rv, vu, RTOL, ATOL).all(), "V outside tolerance and fp32 bound"
    assert_close(loss, rl, what="loss")
    ok, n_bound, rel = grad_ok(g, rg, gu)
    assert ok, f"gradient outside tolerance and fp32 bound (norm rel {rel:.3g}, {n_bound} by bound)"


@pytest.mark.parametrize("h,b", [(128, 16384), (256, 333), (64, 1000)])
def test_value_fwd_bwd_bf16(h, b):
    # against the oracle's bf16-operand mode (the same GEMM operands rounded
    # to bf16, exact sums), element by element
    (v, loss, g), (params, x, qt) = _fwd_bwd(50, h, b, 0.9, prec="bf16", seed=h + b)
    rv, act = iql.forward(params, x, 50, h, gemm_operand=bf16)
    rl, dv = iql.expectile_loss(qt, rv, f32(0.9))
    rg = iql.backward(params, act, dv, 50, h, gemm_operand=bf16)
    vu, gu = bf16_uncertainty(params, x, qt, f32(0.9), 50, h)
    assert abs(loss - rl) <= BF16_RTOL * abs(rl)
    assert within(v, rv, vu, BF16_RTOL, ATOL).all(), "V (bf16)"
    ok, n_bound, worst = bf16_grad_check(g, rg, gu, 50, h)
    assert ok, f"gradient (bf16): outside 2e-2 and the bf16 bound (worst tensor norm rel {worst:.3g})"


@pytest.mark.parametrize("b", [1, 1000, 65536])
@pytest.mark.parametrize("tau", [0.5, 0.7, 0.9])
def test_expectile_loss(b, tau):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    rng = np.random.default_rng(b)
    q = (rng.standard_normal(b) * 2).astype(np.float32)
    v = rng.standard_normal(b).astype(np.float32)
    ctx = ofrl.Context(8, 64, 4, max_batch=1)
    loss = torch.empty(1, device="cuda")
    dv = torch.empty(b, device="cuda")
    ofrl.expectile_loss(ctx, dev(q), dev(v), tau, loss, dv)
    torch.cuda.synchronize()
    rl, rdv = iql.expectile_loss(q, v, f32(tau))
    assert_close(float(loss.cpu()[0]), rl, what="loss")
    assert_close(dv.cpu().numpy(), rdv, what="dL/dV")
    ctx.close()


@pytest.mark.parametrize("b,a", [(1, 1), (777, 5), (16384, 9), (65536, 16)])
def test_policy(b, a):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    rng = np.random.default_rng(a * 100 + b)
    q = (rng.standard_normal((b, a)) * 6).astype(np.float32)   # many advantages hit the clamp
    v = (rng.standard_normal(b) * 3).astype(np.float32)
    ctx = ofrl.Context(8, 64, 4, max_batch=1)
    pi = torch.empty(b, a, device="cuda")
    am = torch.empty(b, dtype=torch.int32, device="cuda")
    ofrl.adv_weighted_policy(ctx, dev(q), dev(v), 3.0, pi, am)
    torch.cuda.synchronize()
    rpi, ram = iql.policy(q, v, f32(3.0))
    assert_close(pi.cpu().numpy(), rpi, what="pi")
    np.testing.assert_allclose(pi.cpu().numpy().sum(axis=1), 1.0, atol=1e-5)
    # same V on both sides: exact, except where fp32 rounding of q - V lands
    # on the clamp and makes a tie the fp64 difference does not have
    argmax_check(am.cpu().numpy(), q, v, v, ram)
    ctx.close()


def _forward_case(s, h, b, prec="fp32", seed=0, path=None):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    w = dataclasses.replace(synth.PROD, state_dim=s, hidden=h, net_seeds=(seed + 11,))
    params = synth.make_params(w)
    rng = np.random.default_rng(seed)
    st = (s + 7) & ~7
    x = np.zeros((b, st), dtype=np.float32)
    x[:, :s] = rng.standard_normal((b, s))
    r = rng.standard_normal(b).astype(np.float32)
    d = (rng.random(b) < 0.1).astype(np.float32)
    ctx = ofrl.Context(s, h, 5, prec, max_batch=b)
    if path is not None:
        ctx.select_vnet_path(path)
    # forward_values and iql_target run on the tensor cores wherever the
    # step takes the fused kernel (hidden 64 / 128), else on the CUDA cores
    want = path or ("tc_fused" if h <= 128 else "tc_layered")
    assert ctx.vnet_path(1) == want, (h, path)
    return ofrl, ctx, w, params, x, r, d


@pytest.mark.parametrize("path", [None, "cuda_cores"], ids=["default", "cuda_cores"])
@pytest.mark.parametrize("s,h,b", [(50, 128, 16384), (50, 128, 65536), (48, 64, 256), (50, 256, 333), (7, 64, 1),
                                   (64, 128, 129), (50, 128, 1000)])
def test_forward_values_fp32(s, h, b, path):
    ofrl, ctx, w, params, x, _, _ = _forward_case(s, h, b, seed=s + b, path=path)
    v = torch.empty(b, device="cuda")
    ofrl.forward_values(ctx, dev(params), dev(x), v)
    torch.cuda.synchronize()
    rv, _, vu, _ = value_uncertainty(params.astype(np.float64), x, np.zeros(b, np.float32), f32(0.7), s, h)
    ctx.close()
    assert within(v.cpu().numpy(), rv, vu, RTOL, ATOL).all(), "V outside tolerance and fp32 bound"


@pytest.mark.parametrize("path", [None, "cuda_cores"], ids=["default", "cuda_cores"])
@pytest.mark.parametrize("s,h,b", [(50, 128, 16384), (50, 256, 1000), (48, 64, 777)])
def test_iql_target_fp32(s, h, b, path):
    ofrl, ctx, w, params, x, r, d = _forward_case(s, h, b, seed=3 * b, path=path)
    gamma = 0.99
    t = torch.empty(b, device="cuda")
    vn = torch.empty(b, device="cuda")
    ofrl.iql_target(ctx, dev(params), dev(x), dev(r), dev(d), gamma, t, v_next_out=vn)
    torch.cuda.synchronize()
    rt, rv = iql.iql_target(params, x, r, d, f32(gamma), s, h)
    _, _, vu, _ = value_uncertainty(params.astype(np.float64), x, np.zeros(b, np.float32), f32(0.7), s, h)
    ctx.close()
    tg, vg = t.cpu().numpy(), vn.cpu().numpy()
    assert within(vg, rv, vu, RTOL, ATOL).all()
    # target = r + gamma (1 - d) V: V's bound scaled by gamma, plus the fp32 rounding of the sum
    tu = float(gamma) * (1.0 - d) * vu + 4 * np.finfo(np.float32).eps * (np.abs(rt) + 1.0)
    assert within(tg, rt, tu, RTOL, ATOL).all()
    # terminal rows bootstrap nothing: exactly the reward
    term = d == 1.0
    assert np.array_equal(tg[term], r[term])


@pytest.mark.parametrize("path", [None, "cuda_cores"], ids=["default", "cuda_cores"])
def test_iql_target_in_a_cuda_graph(path):
    # the forward path captured in a CUDA graph (weight pack + forward kernel,
    # launched on the capturing stream) and replayed gives the direct call's
    # results bit for bit, on new inputs copied into the captured buffers
    b = 3000
    ofrl, ctx, w, params, x, r, d = _forward_case(50, 128, b, seed=11, path=path)
    p_d, x_d, r_d, d_d = dev(params), dev(x), dev(r), dev(d)
    t, vn = torch.empty(b, device="cuda"), torch.empty(b, device="cuda")
    call = lambda: ofrl.iql_target(ctx, p_d, x_d, r_d, d_d, 0.99, t, v_next_out=vn)
    call()
    torch.cuda.synchronize()
    v0 = vn.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    rng = np.random.default_rng(12)
    x_d.copy_(dev(x + rng.standard_normal(x.shape).astype(np.float32)))
    p_d.copy_(dev(params * np.float32(0.9)))
    g.replay()
    torch.cuda.synchronize()
    tg, vg = t.clone(), vn.clone()
    call()
    torch.cuda.synchronize()
    ctx.close()
    assert torch.equal(tg.view(torch.int32), t.view(torch.int32))
    assert torch.equal(vg.view(torch.int32), vn.view(torch.int32))
    assert not torch.equal(vg, v0)   # the replay read the new inputs


@pytest.mark.parametrize("path", [None, "cuda_cores"], ids=["default", "cuda_cores"])
def test_forward_values_bf16(path):
    ofrl, ctx, w, params, x, _, _ = _forward_case(50, 128, 4096, prec="bf16", seed=5, path=path)
    v = torch.empty(4096, device="cuda")
    ofrl.forward_values(ctx, dev(params), dev(x), v)
    torch.cuda.synchronize()
    rv, _ = iql.forward(params, x, 50, 128, gemm_operand=bf16)
    ctx.close()
    # against the oracle's bf16-operand mode, element by element: 2e-2, or
    # inside the bf16 bound (h1 roundings decided the other way)
    vu = bf16_value_uncertainty(params.astype(np.float64), x, 50, 128)
    assert within(v.cpu().numpy(), rv, vu, BF16_RTOL, ATOL).all(), "V (bf16)"


def test_forward_rejects_bad_arguments():
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    ctx = ofrl.Context(50, 128, 5, "fp32", max_batch=64)
    p = torch.zeros(synth.PROD.n_params, device="cuda")
    x = torch.zeros(65, 56, device="cuda")
    v = torch.empty(65, device="cuda")
    with pytest.raises(Exception):
        ofrl.forward_values(ctx, p, x, v)           # batch above max_batch
    r = torch.zeros(8, device="cuda")
    with pytest.raises(Exception):
        ofrl.iql_target(ctx, p, x[:8], r, r, 1.5, r)   # gamma outside [0, 1]
    ctx.close()
