"""GPU: argument errors are refused before launch; device anomalies are counted.

Every failure here is made on the host (bad arguments, NaN/Inf written into
inputs, out-of-range actions written into the replay buffer); no test faults,
traps or hangs the GPU.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from _gpu import GpuStep, dev, need_gpu

pytestmark = pytest.mark.gpu


def test_invalid_arguments_are_refused():
    import offline_rl_step_gb300 as ofrl
    from offline_rl_step_gb300 import _abi
    need_gpu()
    with pytest.raises(ofrl.OfrlError) as e:
        ofrl.Context(50, 96, 5)                    # hidden outside {64, 128, 256}
    assert e.value.code == _abi.EUNSUPPORTED
    with pytest.raises(ofrl.OfrlError) as e:
        ofrl.Context(65, 128, 5)                   # state_dim above 64
    assert e.value.code == _abi.EINVAL
    w = synth.TINY
    g = GpuStep(w)
    try:
        q = dev(synth.make_q(w, 0))
        bad_opt = dataclasses.replace(g.opt, max_grad_norm=0.0)
        with pytest.raises(ofrl.OfrlError) as e:
            ofrl.train_step(g.ctx, g.replay, g.her, 0, g.batch, q, g.nets, bad_opt)
        assert e.value.code == _abi.EINVAL
        big = ofrl.HerConfig(w.batch + 1, 0, "final", 0.01, 1)   # above max_batch
        with pytest.raises(ofrl.OfrlError):
            ofrl.train_step(g.ctx, g.replay, big, 0, g.batch, q, g.nets, g.opt)
        her = ofrl.HerConfig(w.batch, w.batch + 1, "final", 0.01, 1)  # more HER rows than rows
        with pytest.raises(ofrl.OfrlError):
            ofrl.her_relabel(g.ctx, g.replay, her, 0, g.batch)
        nohist = dataclasses.replace(g.replay, episode_ends=None)       # Final needs boundaries
        with pytest.raises(ofrl.OfrlError):
            ofrl.her_relabel(g.ctx, nohist, g.her, 0, g.batch)
        # nothing was launched: the weights are untouched and t did not move
        torch.cuda.synchronize()
        assert np.array_equal(g.nets[0].params.cpu().numpy(), g.params0[0])
        assert g.nets[0].t == 0
    finally:
        g.close()


def test_nan_in_aux_source_is_skipped_and_counted():
    need_gpu()
    w = dataclasses.replace(synth.BUDGETED, batch=512, capacity=1 << 14)
    g = GpuStep(w)
    try:
        aux = [synth.make_aux(w, 0)]
        aux[0][1, :5] = np.nan
        aux[0][2, 5:8] = np.inf
        before = g.nets[0].params.cpu().numpy().copy()
        got = g.step(0, synth.make_q(w, 0), aux)
        st = g.ctx.poll_status()
        # NaN norm -> coefficient 1 (NaN survives at its 5 elements);
        # inf norm -> coefficient 0, 0 * inf = NaN at its 3 elements: 8 skipped
        assert st["nonfinite_grad"] == 8, st
        assert np.array_equal(got["params"][0][:8], before[:8])
        assert np.isfinite(got["params"][0]).all()
    finally:
        g.close()


def test_out_of_range_actions_are_counted():
    need_gpu()
    w = synth.TINY
    g = GpuStep(w)
    try:
        acts = g.replay.actions.clone()
        acts[:] = w.num_actions + 3                   # every stored action invalid
        g.replay.actions = acts
        got = g.step(0, synth.make_q(w, 0))
        st = g.ctx.poll_status()
        assert st["bad_action"] == w.batch * w.n_nets, st
        assert np.isfinite(got["loss"]).all() and np.isfinite(got["params"][0]).all()
    finally:
        g.close()


def test_nan_in_q_is_skipped_by_adam():
    need_gpu()
    w = synth.TINY
    g = GpuStep(w)
    try:
        q = synth.make_q(w, 0)
        q[:, :] = np.nan
        got = g.step(0, q)
        st = g.ctx.poll_status()
        assert np.isnan(got["loss"][0])
        # the norms are NaN, so no clip applies; Adam skips exactly the
        # non-finite gradient elements, counts them and leaves those weights
        bad = ~np.isfinite(got["grad"][0])
        assert bad.sum() > 0.9 * w.n_params
        assert st["nonfinite_grad"] == int(bad.sum()), st
        assert np.array_equal(got["params"][0][bad], g.params0[0][bad])
    finally:
        g.close()


def test_two_runs_are_bit_identical():
    need_gpu()
    w = dataclasses.replace(synth.PROD, steps=3)
    outs = []
    for _ in range(2):
        g = GpuStep(w)
        try:
            for k in range(3):
                o = g.step(k, synth.make_q(w, k))
            outs.append(o)
        finally:
            g.close()
    for key in ("v", "pi", "loss", "norms", "grad"):
        assert np.array_equal(outs[0][key].view(np.uint32), outs[1][key].view(np.uint32)), key
    assert np.array_equal(outs[0]["params"][0].view(np.uint32), outs[1]["params"][0].view(np.uint32))


def test_grid_barrier_timeout_writes_nothing_and_context_stays_usable():
    # The fused reduce + Adam launch is given a grid-barrier target one above
    # what its grid can reach and a 2 ms wait limit (a test-only setting of
    # the context): every CTA gives up, writes no weights, moments or norms,
    # and counts a timeout.  Nothing faults or hangs: the wait is bounded.
    # Afterwards the same step runs normally, bit for bit as on a fresh context.
    need_gpu()
    from offline_rl_step_gb300 import _abi
    lib = _abi.load()
    w = dataclasses.replace(synth.PROD, batch=4096, capacity=1 << 16, steps=1)
    q0 = synth.make_q(w, 0)
    g = GpuStep(w)
    try:
        assert g.kernels() == 3   # relabel, V, and the cooperative reduce + Adam
        net = g.nets[0]
        before = [t.cpu().numpy().copy() for t in (net.params, net.m, net.v)]
        assert lib.ofrl_selftest_barrier(g.ctx.handle, 2_000_000, 1) == _abi.OK
        g.step(0, q0)
        st = g.ctx.poll_status()
        assert st["timeout"] > 0, st
        after = [t.cpu().numpy() for t in (net.params, net.m, net.v)]
        for name, b, a in zip(("params", "m", "v"), before, after):
            assert np.array_equal(b.view(np.uint32), a.view(np.uint32)), f"{name} written after the timeout"
        # back to the normal barrier; the step again from t = 0
        assert lib.ofrl_selftest_barrier(g.ctx.handle, 0, 0) == _abi.OK
        net.t = 0
        got = g.step(0, q0)
        st = g.ctx.poll_status()
        assert st["timeout"] == 0, st
    finally:
        g.close()
    fresh = GpuStep(w)
    try:
        want = fresh.step(0, q0)
    finally:
        fresh.close()
    for key in ("v", "pi", "loss", "norms", "grad"):
        assert np.array_equal(got[key].view(np.uint32), want[key].view(np.uint32)), key
    assert np.array_equal(got["params"][0].view(np.uint32), want["params"][0].view(np.uint32))


def test_barrier_selftest_arguments():
    need_gpu()
    from offline_rl_step_gb300 import _abi
    lib = _abi.load()
    g = GpuStep(synth.TINY)
    try:
        assert lib.ofrl_selftest_barrier(None, 0, 0) == _abi.EINVAL
        assert lib.ofrl_selftest_barrier(g.ctx.handle, 10, 0) == _abi.EINVAL          # below 1 us
        assert lib.ofrl_selftest_barrier(g.ctx.handle, 0, 2) == _abi.EINVAL
        assert lib.ofrl_selftest_barrier(g.ctx.handle, 1_000_000, 0) == _abi.OK
    finally:
        g.close()
