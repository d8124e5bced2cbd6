"""GPU parity: the fused train step on all five workloads, against the oracle,
at every step of each workload's full run (1 / 100 / 100 / 50 / 200 steps).

How a run is checked.  The GPU runs the steps on its own state: nothing is
ever loaded into it from the oracle.  Before each step the test reads every
network's state off the GPU (weights, Adam moments, t, the Polyak target;
fp32 values are exact in fp64), and the oracle computes that same step from
exactly that state.  So every step of the run is compared element by
element, from the same starting point, and the state the GPU carries from
one step to the next is the GPU's.  (A chained fp32 run departs from the
fp64 one legitimately: Adam's first updates are about lr sign(g), so a
gradient element whose sign fp32 does not fix moves its weight by 2 lr, and
that difference feeds the later steps.  test_production_trajectory compares
the two free-running 100-step trajectories norm-wise as well.)

Per step and network:
  * batch (indices, relabelled states, actions, rewards, dones): bit-exact;
  * loss, V, pi, norms: 1e-4 relative / 1e-5 absolute (fp32 workloads); a V
    or pi element outside that must lie inside the fp32 error bound of
    tests/_errmodel.py (rounding, propagated uncertainty, ReLU masks decided
    inside their own uncertainty), computed only when needed;
  * argmax: bit-exact against the argmax of the GPU's own clamped advantages
    on every row, and equal to the oracle's except on rows where a +-10
    clamp breakpoint lies between the two V values (counted);
  * primary gradient: 1e-4 / 1e-5 element-wise, or inside the fp32 bound,
    and norm-wise beyond each element's bound to 1e-4 (the bound-excused
    elements are counted);
  * the Adam step twice: (1) the weights, moments and target the GPU wrote
    equal the oracle's clipped combination and Adam applied to the GPU's own
    primary gradient from the same state, every element, to fp32 rounding
    (no exceptions); (2) they equal the oracle's own post-step values within
    1e-4 / 1e-5, except weights whose gradient element was itself outside
    that tolerance (counted; (1) shows those weights follow the GPU's
    gradient, the gradient check shows that gradient is fp32-correct).
bf16 workload (twin networks): the oracle's bf16-operand mode (GEMM operands
rounded to bf16, exact sums) with 2e-2 relative on V, pi, the gradient, the
norms, the loss and the post-Adam weights.  A V or pi element outside that
must lie inside the bf16 bound (tests/_errmodel.py bf16_uncertainty: fp32
sums, operands within their fp32 uncertainty of a bf16 rounding midpoint,
which the GPU may round the other way, and ReLU masks that decides), and
every gradient tensor must match norm-wise to 2e-2 (tests/_gpu.py
bf16_grad_check).  The Adam steps follow the fp32 master weights, so check
(1) is the fp32 one.

With OFRL_PARITY_LOG=<file> each checked step appends one JSON record (the
counts above and the largest errors).
"""
import copy
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import synth
from _errmodel import bf16_uncertainty, grad_ok, value_uncertainty, within
from _gpu import (ATOL, BF16_RTOL, RTOL, GpuStep, argmax_check, assert_bits, assert_close, bf16_grad_check,
                  need_gpu, oracle_cfg, oracle_nets, replay_np)
from oracle import iql, optim
from oracle import step as ostep

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24
LOG = os.environ.get("OFRL_PARITY_LOG")


def _log(rec):
    if LOG:
        with open(LOG, "a") as f:
            f.write(json.dumps(rec) + "\n")


def adam_given_gradient(cfg, pre, g0, aux=None, dg=None):
    """The oracle's budgeted combination and Adam step (and Polyak target)
    applied to a given primary gradient g0, from the network state `pre`.

    Returns (G, G_scale, p, m, v, target): G the combined gradient, G_scale
    the sum of |terms| of each of its elements.  dg (optional, per element)
    shifts G before Adam, to probe how far a rounding of G moves the update.
    """
    sources = [np.asarray(g0, dtype=np.float64)]
    if aux is not None:
        sources += [np.asarray(a, dtype=np.float64) for a in aux]
    if cfg.sanitize_sources:
        sources = [optim.sanitize(x) for x in sources]
    n = len(sources)
    g, norms = optim.budgeted_combine(sources, cfg.budget[:n], cfg.alpha[:n], cfg.max_grad_norm)
    gsc = np.zeros_like(g)
    for k, x in enumerate(sources):
        c = abs(float(cfg.alpha[k]) * optim.clip_scale(norms[k], float(cfg.budget[k]) * cfg.max_grad_norm))
        gsc += c * np.abs(x)
    if dg is not None:
        g = g + dg
    p, m, v, _ = optim.adam(pre.params, g, pre.m, pre.v, pre.t + 1, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
                            cfg.weight_decay, cfg.max_grad_norm, norms[-1], cfg.weight_clamp_max_abs)
    tgt = None if pre.target is None else optim.polyak(pre.target, p, pre.polyak)
    return g, gsc, p, m, v, tgt


def _close_to_rounding(got, want, scale, rel, what):
    """|got - want| <= 4 u |want| + rel * scale, every element (u = 2^-24)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    bad = err > 4 * U32 * np.abs(want) + rel * scale
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements off (max abs err "
                           f"{float(err.max()):.3g}); first at {int(np.argmax(bad))}")


class _Bound:
    """The error bounds of one network's V and gradient (fp32 workloads:
    tests/_errmodel.py value_uncertainty; bf16: bf16_uncertainty), computed
    once and only when an element is outside the plain tolerance."""

    def __init__(self, w, pre, states, qt):
        self.w, self.pre, self.states, self.qt = w, pre, states, qt
        self.vu = self.gu = None
        self.info = {}

    def _get(self):
        if self.vu is None:
            w, p = self.w, self.pre
            if w.prec == "bf16":
                self.vu, self.gu = bf16_uncertainty(p.params, self.states, self.qt, p.tau, w.state_dim, w.hidden)
            else:
                _, _, self.vu, self.gu = value_uncertainty(p.params, self.states, self.qt, p.tau, w.state_dim,
                                                           w.hidden, info=self.info)
        return self.vu, self.gu

    def v(self):
        return self._get()[0]

    def g(self):
        return self._get()[1]


def _check_step(w, cfg, k, got, ref, post, pre, q, aux):
    s = w.state_dim
    bt, rb = got["batch"], ref["batch"]
    for key in ("src_idx", "donor_idx", "actions", "rewards", "dones"):
        assert_bits(bt[key], rb[key], f"step {k} {key}")
    assert_bits(bt["states"][:, :s], rb["states"][:, :s], f"step {k} states")
    assert_bits(bt["next_states"][:, :s], rb["next_states"][:, :s], f"step {k} next_states")
    bf = w.prec == "bf16"
    rtol = BF16_RTOL if bf else RTOL
    qt = iql.q_taken(q, rb["actions"])
    for n in range(w.n_nets):
        tag = f"step {k} net {n}"
        bound = _Bound(w, pre[n], rb["states"], qt)
        rec = dict(test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], workload=w.name, step=k, net=n,
                   n_params=int(w.n_params))

        # ---- loss, V, pi ----
        assert_close(got["loss"][n], ref["loss"][n], rtol=rtol, what=f"{tag} loss")
        gv, rv = got["v"][n], ref["v"][n]
        v_ok = within(gv, rv, 0.0, rtol, ATOL)
        rec["v_bound_rows"] = int((~v_ok).sum())
        if not v_ok.all():
            v_ok = within(gv, rv, bound.v(), rtol, ATOL)
        assert v_ok.all(), f"{tag} V: {int((~v_ok).sum())} rows outside tolerance and bound"
        gp, rp = got["pi"][n], ref["pi"][n]
        pi_ok = within(gp, rp, 0.0, rtol, ATOL)
        rec["pi_bound_entries"] = int((~pi_ok).sum())
        if not pi_ok.all():
            pi_ok = within(gp, rp, w.beta * bound.v()[:, None], rtol, ATOL)
        assert pi_ok.all(), f"{tag} pi: {int((~pi_ok).sum())} entries outside tolerance and bound"
        rec["argmax_breakpoint_rows"] = argmax_check(got["argmax"][n], q, gv, rv, ref["argmax"][n], f"{tag} argmax")

        # ---- primary gradient ----
        gg, rg = got["grad"][n].astype(np.float64), ref["grad"][n]
        plain = np.abs(gg - rg) <= ATOL + RTOL * np.abs(rg)
        if bf:
            ok, n_bound, worst = bf16_grad_check(gg, rg, 0.0, s, w.hidden)
            if not ok:
                ok, n_bound, worst = bf16_grad_check(gg, rg, bound.g(), s, w.hidden)
            rec["grad_excused_by_bound"], rec["grad_tensor_norm_rel"] = n_bound, worst
            assert ok, f"{tag} gradient (bf16): outside 2e-2 and the bf16 bound (worst tensor norm rel {worst:.3g})"
        elif plain.all():
            rec["grad_excused_by_bound"] = 0
        else:
            ok, n_bound, rel = grad_ok(gg, rg, bound.g())
            rec["grad_excused_by_bound"], rec["grad_norm_excess"] = n_bound, rel
            assert ok, f"{tag} gradient: outside tolerance and bound (norm-wise excess {rel:.3g})"
        rec["grad_max_rel_err"] = float((np.abs(gg - rg) / np.maximum(np.abs(rg), 1e-30)).max())
        ns = 1 + (w.n_aux if aux is not None else 0)
        assert_close(got["norms"][n][:ns], ref["norms"][n][:ns], rtol=rtol, what=f"{tag} norms")
        assert_close(got["norms"][n][4], ref["norms"][n][4], rtol=rtol, what=f"{tag} combined norm")

        # ---- (1) Adam on the GPU's own gradient, same state: to fp32 rounding ----
        # The GPU forms G in fp32 (off by up to a few u times G's sum of
        # |terms|); where G is small by cancellation, near Adam's eps, that
        # rounding moves the update, so the weight tolerance adds the update's
        # spread over G +- 8 u |terms|.
        a_n = None if aux is None else aux[n]
        G, gsc, pc, mc, vc, tc = adam_given_gradient(cfg, pre[n], gg, a_n)
        dg = 8 * U32 * gsc
        spread = np.maximum(np.abs(adam_given_gradient(cfg, pre[n], gg, a_n, dg)[2] - pc),
                            np.abs(adam_given_gradient(cfg, pre[n], gg, a_n, -dg)[2] - pc))
        _close_to_rounding(got["params"][n], pc, cfg.lr + spread / 1e-4, 1e-4,
                           f"{tag} weights vs Adam on the GPU gradient")
        _close_to_rounding(got["m"][n], mc, cfg.beta1 * np.abs(pre[n].m) + (1 - cfg.beta1) * gsc, 1e-5,
                           f"{tag} m vs Adam on the GPU gradient")
        _close_to_rounding(got["vmom"][n], vc, cfg.beta2 * pre[n].v + (1 - cfg.beta2) * gsc * gsc, 1e-5,
                           f"{tag} v vs Adam on the GPU gradient")
        if tc is not None:
            _close_to_rounding(got["target"][n], tc, (1 - pre[n].polyak) * np.abs(pre[n].target)
                               + pre[n].polyak * (np.abs(pc) + spread), 1e-5,
                               f"{tag} target vs Adam on the GPU gradient")
        rec["adam_spread_weights"] = int((spread > 1e-4 * cfg.lr).sum())
        assert got["t"][n] == pre[n].t + 1, f"{tag}: t"

        # ---- (2) against the oracle's own update ----
        # a weight may be off only where the two gradients differ beyond 1e-4
        # relative (Adam's first updates are about lr sign(g), so a gradient
        # element inside the 1e-5 absolute tolerance with the other sign moves
        # its weight by 2 lr)
        p_off = np.abs(got["params"][n] - post[n].params) > ATOL + rtol * np.abs(post[n].params)
        unexplained = p_off & (np.abs(gg - rg) <= RTOL * np.abs(rg))
        assert not unexplained.any(), (f"{tag} weights: {int(unexplained.sum())} off tolerance where the gradient "
                                       f"agrees (first at {int(np.argmax(unexplained))})")
        rec["weights_off_tolerance"] = int(p_off.sum())
        rec["v_max_abs_err"] = float(np.abs(gv - rv).max())
        rec["loss_rel"] = float(abs(got["loss"][n] / ref["loss"][n] - 1))
        if "ambiguous_masks" in bound.info:
            rec["ambiguous_relu_masks"] = bound.info["ambiguous_masks"]
        _log(rec)


def _run(w, graph=False, path=None, host_io=False, polyak=None, plant=None, **opts):
    """Every step of workload w on the GPU, each checked against the oracle
    computed from the GPU's own state before the step."""
    need_gpu()
    g = GpuStep(w, graph=graph, path=path, host_io=host_io, polyak=polyak, **opts)
    cfg = oracle_cfg(w, **opts)
    rep = replay_np(w)
    try:
        for k in range(w.steps):
            q = synth.make_q(w, k)
            aux = [synth.make_aux(w, k, n) for n in range(w.n_nets)] if w.n_aux else None
            if plant is not None:
                plant(aux)
            pre = g.state()
            got = g.step(k, q, aux)
            post = copy.deepcopy(pre)
            ref = ostep.train_step(cfg, rep, k, q, post, aux)
            _check_step(w, cfg, k, got, ref, post, pre, q, aux)
            if w.n_aux:
                # the combined norm never exceeds the budget sum
                assert (got["norms"][:, 4] <= w.max_grad_norm * (1 + 1e-5)).all()
        st = g.ctx.poll_status()   # reading the status word clears it
        assert st["bad_action"] == 0 and st["bad_index"] == 0 and st["nonfinite_grad"] == 0, st
        assert all(n.t == w.steps for n in g.nets)
        return st
    finally:
        g.close()


@pytest.mark.parametrize("w", synth.ALL, ids=lambda w: w.name)
def test_train_step_matches_oracle(w):
    _run(w)


def test_production_trajectory():
    # the GPU's and the oracle's free-running 100-step production runs (each
    # on its own state throughout): the loss each step within 1e-4, V and
    # the weights within 1e-3 in norm.  Element-wise agreement is what
    # test_train_step_matches_oracle checks, step by step.
    need_gpu()
    w = synth.PROD
    g = GpuStep(w)
    cfg = oracle_cfg(w)
    rep = replay_np(w)
    nets = oracle_nets(w)
    try:
        for k in range(w.steps):
            q = synth.make_q(w, k)
            got = g.step(k, q)
            ref = ostep.train_step(cfg, rep, k, q, nets)
            p, rp = got["params"][0].astype(np.float64), nets[0].params
            assert abs(got["loss"][0] - ref["loss"][0]) <= RTOL * abs(ref["loss"][0]), f"step {k} loss"
            assert np.linalg.norm(got["v"][0] - ref["v"][0]) <= 1e-3 * np.linalg.norm(ref["v"][0]), f"step {k} V"
            assert np.linalg.norm(p - rp) <= 1e-3 * np.linalg.norm(rp), f"step {k} weights"
            _log(dict(test="test_production_trajectory", workload=w.name, step=k, phase="free trajectory",
                      weights_norm_rel=float(np.linalg.norm(p - rp) / np.linalg.norm(rp)),
                      weights_off_tolerance=int((np.abs(p - rp) > ATOL + RTOL * np.abs(rp)).sum()),
                      loss_rel=float(abs(got["loss"][0] / ref["loss"][0] - 1))))
    finally:
        g.close()


def test_ragged_batch_step():
    # a batch that is not a multiple of the tile rows, H = 256 (layered
    # tensor-core path: 8 tiles, the last one ragged)
    _run(dataclasses.replace(synth.BUDGETED, batch=1000, capacity=1 << 14, steps=3))


def test_vnet_path_choice():
    # the default implementation per hidden width, and which choices a shape allows
    need_gpu()
    import offline_rl_step_gb300 as ofrl
    from offline_rl_step_gb300 import _abi
    want = {64: "tc_fused", 128: "tc_fused", 256: "tc_layered"}
    for h, path in want.items():
        for nets in (1, 2):
            ctx = ofrl.Context(50, h, 5, "fp32", max_batch=4096, max_nets=nets)
            try:
                assert ctx.vnet_path(nets) == path, (h, nets)
                ctx.select_vnet_path("cuda_cores")
                assert ctx.vnet_path(nets) == "cuda_cores"
                for other in ("tc_fused", "tc_layered"):
                    ok = (other == "tc_fused" and h <= 128) or (other == "tc_layered" and h in (128, 256))
                    if ok:
                        ctx.select_vnet_path(other)
                        assert ctx.vnet_path(nets) == other
                    else:
                        with pytest.raises(_abi.OfrlError):
                            ctx.select_vnet_path(other)
            finally:
                ctx.close()
    # a 64-column state leaves no ones column: no layered path
    ctx = ofrl.Context(64, 256, 5, "fp32", max_batch=1024)
    try:
        assert ctx.vnet_path(1) == "cuda_cores"
    finally:
        ctx.close()


@pytest.mark.parametrize("w, path", [
    (dataclasses.replace(synth.PROD, batch=2000, capacity=1 << 16, steps=3), "tc_layered"),
    (dataclasses.replace(synth.TWIN, batch=1000, capacity=1 << 14, steps=3), "tc_layered"),
    (dataclasses.replace(synth.TWIN, batch=1000, capacity=1 << 14, steps=3), "cuda_cores"),
    (dataclasses.replace(synth.PROD, batch=1000, capacity=1 << 14, steps=3), "cuda_cores"),
    (dataclasses.replace(synth.BUDGETED, batch=1000, capacity=1 << 14, steps=3), "cuda_cores"),
    (dataclasses.replace(synth.BUDGETED, batch=128, capacity=1 << 14, steps=3), "tc_layered"),
    (dataclasses.replace(synth.TINY, steps=3), "cuda_cores"),
    (dataclasses.replace(synth.TINY, batch=1000, capacity=1 << 14, steps=3), "tc_fused"),
    (dataclasses.replace(synth.PROD, batch=32768, steps=3), "tc_fused"),
], ids=["prod_layered", "twin_bf16_layered", "twin_bf16_cuda_cores", "prod_cuda_cores", "budgeted_cuda_cores",
        "budgeted_one_tile", "tiny_cuda_cores", "h64_ragged_fused", "prod_256_tiles_two_per_cta"])
def test_step_on_each_vnet_path(w, path):
    # every implementation against the oracle (the default ones run in the tests above)
    _run(w, path=path)


@pytest.mark.parametrize("w", [
    dataclasses.replace(synth.PROD, state_dim=64, num_actions=16, batch=1000, capacity=1 << 14, steps=3),
    dataclasses.replace(synth.PROD, state_dim=63, hidden=256, num_actions=16, batch=300, capacity=1 << 14, steps=3),
    dataclasses.replace(synth.TINY, state_dim=64, num_actions=1, batch=700, capacity=1 << 14, steps=3),
], ids=["s64_a16_h128", "s63_a16_h256", "s64_a1_h64"])
def test_step_at_shape_limits(w):
    # the largest state (no ones column in the state-tile image: db1 from
    # column sums), the most and the fewest actions, hidden 256 with S = 63
    _run(w)


def test_single_row_batch_step():
    _run(dataclasses.replace(synth.TINY, batch=1, her_ratio=1.0, steps=3))


def test_step_with_source_guard_weight_bound_and_target():
    # three auxiliary sources with planted NaN / +-inf elements and the
    # isfinite guard on; a weight bound below the initial weight range (it
    # binds from the first step); a Polyak target copy of every network
    w = dataclasses.replace(synth.PROD, batch=1000, capacity=1 << 14, steps=4,
                            aux_sigmas=synth.BUDGETED.aux_sigmas, weight_decay=1e-4)
    planted = [0]

    def plant(aux):
        for per in aux:
            for j, src in enumerate(per):
                src[[7 + j, 1000 + 13 * j, w.n_params - 1 - j]] = [np.nan, np.inf, -np.inf]
                planted[0] += 3

    st = _run(w, polyak=0.05, plant=plant, weight_clamp_max_abs=0.15, sanitize_sources=True)
    assert st["sanitized"] == planted[0], st


def test_reduce_and_adam_launch_fusion_choice():
    # the production batch (128 tile partials: 64 element lanes, 91 blocks)
    # and the H = 256 workload (76 K-range partials of 79k parameters, or 256
    # tile partials from the CUDA-core kernel: 310 blocks) take the single
    # cooperative reduce + Adam launch; the layered path has two V kernels
    need_gpu()
    for w, expect, path in ((synth.PROD, 3, None), (dataclasses.replace(synth.BUDGETED, capacity=1 << 16), 4, None),
                            (dataclasses.replace(synth.BUDGETED, capacity=1 << 16), 3, "cuda_cores")):
        g = GpuStep(w, path=path)
        try:
            assert g.kernels() == expect, (w.name, path)
        finally:
            g.close()


@pytest.mark.parametrize("w", [dataclasses.replace(synth.PROD, steps=6),
                               dataclasses.replace(synth.BUDGETED, batch=1000, capacity=1 << 14, steps=3),
                               dataclasses.replace(synth.TWIN, steps=3)],
                         ids=["prod_graph", "budgeted_graph", "twin_graph"])
def test_step_graph_matches_oracle(w):
    # the same steps replayed from one captured CUDA graph: the step index,
    # Q and the auxiliary sources change per replay, t advances
    _run(w, graph=True)


@pytest.mark.parametrize("w", [dataclasses.replace(synth.PROD, steps=4),
                               dataclasses.replace(synth.BUDGETED, batch=1000, capacity=1 << 14, steps=3)],
                         ids=["prod_graph_io", "budgeted_graph_io"])
def test_step_graph_host_io_matches_oracle(w):
    # the graph with its host I/O: each replay copies a fresh pinned host Q in
    # and the loss and norms out (equal to the device results bit for bit)
    _run(w, graph="io")


@pytest.mark.parametrize("w", [dataclasses.replace(synth.PROD, steps=4),
                               dataclasses.replace(synth.BUDGETED, batch=1000, capacity=1 << 14, steps=3),
                               dataclasses.replace(synth.TINY, steps=3),
                               dataclasses.replace(synth.PROD, batch=1001, capacity=1 << 14, steps=3),
                               dataclasses.replace(synth.TWIN, steps=3)],
                         ids=["prod_host_buffers", "budgeted_host_buffers", "tiny_host_buffers",
                              "ragged_host_buffers", "twin_host_buffers"])
def test_train_step_with_host_buffers_matches_oracle(w):
    # Q in pinned host memory (staged into the workspace by the relabel's row
    # blocks; 1001 rows of 5 actions end in a run copied element by element),
    # loss and norms written in place into pinned host memory by the kernels
    _run(w, host_io=True)


def test_step_graph_with_host_q_matches_oracle():
    # a graph captured with Q in pinned host memory: each replay points the
    # relabel's staging copy at that step's host Q
    _run(dataclasses.replace(synth.PROD, batch=2000, capacity=1 << 16, steps=3), graph=True, host_io=True)
