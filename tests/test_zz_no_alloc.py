"""The allocation-free V forward/backward entry point.

For callers that may not allocate device memory (a host framework owns the
GPU memory pool, a CUDA graph recorded under the global capture mode, a
latency-critical loop), ofrl_iql_value_fwd_bwd_noalloc runs the same
computation as ofrl_iql_value_fwd_bwd out of the library's fixed scratch
array.  This test calls both through the C ABI on the same inputs, twice in a
row (the scratch keeps the previous call's contents), and requires the same
results within the parity tolerance, and the allocation-free results to match
the oracle (V, loss and gradient within 1e-4 / 1e-5 or the fp32 error bound);
it also checks the size limit.  It sits in a file of its own that pytest
collects last.
"""
import numpy as np
import pytest
import torch

import synth
from _errmodel import grad_ok, value_uncertainty, within
from _gpu import ATOL, RTOL, assert_close, dev, need_gpu
from oracle import iql

pytestmark = pytest.mark.gpu


def _inputs(s, h, b, seed):
    import dataclasses
    w = dataclasses.replace(synth.PROD, state_dim=s, hidden=h, net_seeds=(seed,))
    rng = np.random.default_rng(seed)
    x = np.zeros((b, (s + 7) & ~7), dtype=np.float32)
    x[:, :s] = rng.standard_normal((b, s))
    q = (rng.standard_normal(b) * 2).astype(np.float32)
    return synth.make_params(w), x, q, w.n_params


@pytest.mark.parametrize("s,h,b", [(50, 128, 3000), (48, 64, 257), (50, 256, 500)])
def test_noalloc_matches_context_entry_point_twice(s, h, b):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    assert b <= ofrl.noalloc_max_batch(s, h, 5)
    ctx = ofrl.Context(s, h, 5, max_batch=b)
    for call in range(2):
        params, x, q, p = _inputs(s, h, b, seed=100 * call + h)
        tp, tx, tq = dev(params), dev(x), dev(q)
        want = (torch.empty(b, device="cuda"), torch.empty(1, device="cuda"), torch.empty(p, device="cuda"))
        got = (torch.empty(b, device="cuda"), torch.empty(1, device="cuda"), torch.empty(p, device="cuda"))
        ofrl.iql_value_fwd_bwd(ctx, tp, tx, tq, 0.7, *want)
        ofrl.iql_value_fwd_bwd_noalloc(s, h, 5, tp, tx, tq, 0.7, *got)
        torch.cuda.synchronize()
        for name, g, r in zip(("V", "loss", "gradient"), got, want):
            assert_close(g.cpu().numpy(), r.cpu().numpy(), rtol=RTOL, atol=ATOL, what=f"call {call} {name}")
        # against the oracle (fp64), on the same inputs
        v_ref, loss_ref, g_ref = iql.value_fwd_bwd(params, x, q, 0.7, s, h)
        _, _, vu, gu = value_uncertainty(params, x, q, 0.7, s, h)
        v_got, loss_got, g_got = (t.cpu().numpy() for t in got)
        assert within(v_got, v_ref, vu, RTOL, ATOL).all(), f"call {call}: V against the oracle"
        assert_close(loss_got[0], loss_ref, what=f"call {call}: loss against the oracle")
        ok, _, rel = grad_ok(g_got, g_ref, gu)
        assert ok, f"call {call}: gradient against the oracle (norm rel {rel:.3g})"
    ctx.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    import offline_rl_step_gb300 as ofrl
    from offline_rl_step_gb300 import _abi
    need_gpu()
    limit = ofrl.noalloc_max_batch(50, 128, 5)
    assert limit > 0
    b = limit + 1
    params, x, q, p = _inputs(50, 128, b, seed=3)
    outs = (torch.empty(b, device="cuda"), torch.empty(1, device="cuda"), torch.empty(p, device="cuda"))
    with pytest.raises(ofrl.OfrlError) as e:
        ofrl.iql_value_fwd_bwd_noalloc(50, 128, 5, dev(params), dev(x), dev(q), 0.7, *outs)
    assert e.value.code == _abi.EINVAL
