"""Shared helpers of the GPU parity tests: inputs, oracle runs, comparisons.

Tolerances (fp32 GEMM workloads): 1e-4 relative / 1e-5 absolute on V, the
loss, the policy, gradients and post-Adam weights; bit-exact on HER indices,
relabelled goals, rewards and the policy argmax.  bf16-GEMM workloads: 2e-2
relative on the loss and the weights.
"""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import her as oher
from oracle import iql
from oracle import step as ostep

RTOL, ATOL = 1e-4, 1e-5
BF16_RTOL = 2e-2

_REPLAYS = {}


def f32(x):
    """The fp32 value the library receives for a hyper-parameter."""
    return float(np.float32(x))


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import offline_rl_step_gb300 as ofrl  # noqa: F401
    from offline_rl_step_gb300 import _abi
    _abi.load()   # raises if the library is not built: no silent fallback


def replay_np(w):
    key = (w.seed, w.capacity, w.state_dim, w.goal_dim, w.ep_len, w.num_actions, w.anchor_frac)
    if key not in _REPLAYS:
        if len(_REPLAYS) >= 3:
            _REPLAYS.clear()
        _REPLAYS[key] = synth.make_replay(w)
    return _REPLAYS[key]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def replay_dev(w, rep):
    import offline_rl_step_gb300 as ofrl
    return ofrl.Replay(dev(rep["states"]), dev(rep["next_states"]), dev(rep["actions"]), dev(rep["rewards"]),
                       dev(rep["dones"]), w.state_dim, w.goal_dim, dev(rep["episode_ends"]))


def oracle_cfg(w, weight_clamp_max_abs=0.0, sanitize_sources=False):
    """Oracle step config with the fp32-rounded constants the library gets."""
    c = ostep.config_from_workload(w)
    return dataclasses.replace(
        c, goal_threshold=f32(w.goal_threshold), beta=f32(w.beta), lr=f32(w.lr), beta1=f32(w.beta1),
        beta2=f32(w.beta2), eps=f32(w.eps), weight_decay=f32(w.weight_decay),
        max_grad_norm=f32(w.max_grad_norm), budget=tuple(f32(b) for b in w.budget),
        weight_clamp_max_abs=f32(weight_clamp_max_abs), sanitize_sources=bool(sanitize_sources))


def report(gpu, ref, rtol, atol):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))
    rel = err / np.maximum(np.abs(ref), 1e-30)
    return bad, float(err.max(initial=0.0)), float(rel.max(initial=0.0))


def assert_close(gpu, ref, rtol=RTOL, atol=ATOL, what="value", allow=None):
    """Element-wise |gpu - ref| <= atol + rtol |ref|; `allow` masks elements that may differ."""
    bad, emax, rmax = report(gpu, ref, rtol, atol)
    if allow is not None:
        bad &= ~np.asarray(allow, dtype=bool)
    n = int(bad.sum())
    assert n == 0, f"{what}: {n} of {bad.size} elements out of tolerance (max abs {emax:.3g}, max rel {rmax:.3g})"


def assert_bits(gpu, ref, what="value"):
    g = np.ascontiguousarray(gpu)
    r = np.ascontiguousarray(ref)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    if g.dtype.kind == "f":
        g, r = g.view(np.uint32 if g.itemsize == 4 else np.uint64), r.astype(g.dtype).view(
            np.uint32 if g.itemsize == 4 else np.uint64)
    n = int((g != r).sum())
    assert n == 0, f"{what}: {n} of {g.size} elements differ"


def bf16_grad_check(gpu, ref, unc, state_dim, hidden):
    """bf16 workload, gradient against the oracle's bf16-operand mode.

    Element-wise: within 2e-2 relative (1e-5 absolute), or inside the bf16
    bound `unc` (tests/_errmodel.py bf16_uncertainty).  Norm-wise per tensor
    (W1, b1, W2, b2, w3, b3): ||gpu - ref|| <= 2e-2 ||ref||, so a wrong
    sign, index or scale in any one tensor fails whatever the bound allows.
    Returns (ok, elements inside the bound but outside 2e-2, largest
    per-tensor relative norm error).
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    tol = err <= ATOL + BF16_RTOL * np.abs(ref)
    elem = tol | (err <= unc)
    seg = iql.unflatten(np.arange(ref.size), state_dim, hidden)
    worst = 0.0
    for ix in seg:
        ix = np.asarray(ix, dtype=np.int64).ravel()
        worst = max(worst, float(np.linalg.norm(gpu[ix] - ref[ix]) / max(np.linalg.norm(ref[ix]), 1e-300)))
    return bool(elem.all() and worst <= BF16_RTOL), int((~tol & elem).sum()), worst


def argmax_of(q, v):
    """The policy argmax the GPU must produce from its own V: the lowest index
    of the row maximum of clamp(q - v, -10, 10), the difference rounded to
    fp32 as the kernel rounds it."""
    q32 = np.asarray(q, dtype=np.float32)
    v32 = np.asarray(v, dtype=np.float32)
    adv = np.clip(q32 - v32[:, None], np.float32(-10.0), np.float32(10.0))
    return np.argmax(adv, axis=1).astype(np.int32)


def argmax_check(gpu_am, q, v_gpu, v_ref, ref_am, what="argmax"):
    """The policy argmax, exact.

    (1) On every row it is the argmax of the GPU's own clamped advantages
    (argmax_of): bit-exact, no exceptions.  (2) It equals the oracle's argmax
    on every row, except where a clamp breakpoint (q_a - V = +-10, where an
    entry enters or leaves a tie at the clamp) lies between the GPU's V and
    the oracle's V: there the argmax over that interval of V takes more than
    one value and the GPU's must be one of them.  V itself is compared
    separately.  Returns the number of such rows.
    """
    gpu_am = np.asarray(gpu_am)
    own = argmax_of(q, v_gpu)
    n_own = int((gpu_am != own).sum())
    assert n_own == 0, f"{what}: {n_own} rows differ from the argmax of the GPU's own clamped advantages"
    diff = np.nonzero(gpu_am != np.asarray(ref_am))[0]
    if diff.size == 0:
        return 0
    q = np.asarray(q, dtype=np.float64)
    for r in diff:
        lo, hi = sorted((float(v_gpu[r]), float(v_ref[r])))
        slack = 4 * np.spacing(np.float32(10.0))   # fp32 rounding of q - V near the clamp
        lo, hi = lo - slack, hi + slack
        cand = [lo, hi] + [c for a in q[r] for c in (a - 10.0, a + 10.0) if lo <= c <= hi]
        cand = sorted(set(cand + [c + d for c in cand for d in (-1e-9, 1e-9)]))
        accept = {int(np.argmax(np.clip(q[r] - c, -10.0, 10.0))) for c in cand if lo <= c <= hi}
        assert len(accept) > 1 and int(gpu_am[r]) in accept, \
            f"{what}: row {r} argmax {int(gpu_am[r])} vs oracle {int(ref_am[r])} with no clamp breakpoint between " \
            f"V {float(v_gpu[r])!r} and {float(v_ref[r])!r}"
    return int(diff.size)


class GpuStep:
    """The fused train step of one workload on the GPU, through the C ABI."""

    def __init__(self, w, weight_clamp_max_abs=0.0, sanitize_sources=False, polyak=None, graph=False, path=None,
                 host_io=False):
        import offline_rl_step_gb300 as ofrl
        self.ofrl = ofrl
        self.w = w
        self.rep = replay_np(w)
        self.replay = replay_dev(w, self.rep)
        self.her = ofrl.HerConfig(w.batch, w.her_count, w.strategy, w.goal_threshold, w.seed)
        self.ctx = ofrl.Context(w.state_dim, w.hidden, w.num_actions, w.prec, max_batch=w.batch,
                                max_nets=w.n_nets)
        if path is not None:
            self.ctx.select_vnet_path(path)
            assert self.ctx.vnet_path(w.n_nets) == path
        self.params0 = [synth.make_params(w, k) for k in range(w.n_nets)]
        self.nets = [ofrl.VNet.from_params(torch.from_numpy(p), w.taus[k], polyak=polyak)
                     for k, p in enumerate(self.params0)]
        self.opt = ofrl.Opt(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                            max_grad_norm=w.max_grad_norm, beta=w.beta, budget=w.budget,
                            weight_clamp_max_abs=weight_clamp_max_abs, sanitize_sources=sanitize_sources)
        self.batch = ofrl.Batch.empty(w.batch, w.state_stride)
        n, b, a, p = w.n_nets, w.batch, w.num_actions, w.n_params
        self.v = torch.empty(n, b, device="cuda")
        self.pi = torch.empty(n, b, a, device="cuda")
        self.am = torch.empty(n, b, dtype=torch.int32, device="cuda")
        # host_io: Q read in place from pinned host memory, loss and norms
        # written in place into pinned host memory by the kernels
        self.host_io = host_io
        self.loss = torch.empty(n, pin_memory=True) if host_io else torch.empty(n, device="cuda")
        self.norms = torch.empty(n, 5, pin_memory=True) if host_io else torch.empty(n, 5, device="cuda")
        self.grad = torch.empty(n, p, device="cuda")
        self.use_graph = graph
        self.sg = None

    def step(self, k, q, aux=None):
        aux_dev = None if aux is None else [[dev(a) for a in per] for per in aux]
        if self.use_graph == "io":
            # the graph with its host I/O: Q copied in from pinned host memory,
            # loss and norms copied out to pinned host memory, one launch
            qh = torch.from_numpy(np.ascontiguousarray(q)).pin_memory()
            if self.sg is None:
                self.qd = torch.empty(qh.shape, device="cuda")
                self.loss_h = torch.empty(self.w.n_nets, pin_memory=True)
                self.norms_h = torch.empty(self.w.n_nets, 5, pin_memory=True)
                self.sg = self.ofrl.StepGraph(self.ctx, self.replay, self.her, self.batch, self.nets, self.opt,
                                              self.qd, aux=aux_dev, v_out=self.v, pi_out=self.pi, argmax_out=self.am,
                                              loss_out=self.loss, norms_out=self.norms, grad_out=self.grad,
                                              q_host=qh, loss_host=self.loss_h, norms_host=self.norms_h)
            self.sg.launch_io(k, qh, aux_dev, self.loss_h, self.norms_h)
            torch.cuda.synchronize()
            self.sg.sync_t()
            # the host copies are the device results, bit for bit
            assert np.array_equal(self.loss_h.numpy(), self.loss.cpu().numpy())
            assert np.array_equal(self.norms_h.numpy(), self.norms.cpu().numpy())
            return self._results()
        qd = torch.from_numpy(np.ascontiguousarray(q)).pin_memory() if self.host_io else dev(q)
        if self.use_graph:
            # the step as a replayed CUDA graph (captured at the first step)
            if self.sg is None:
                self.sg = self.ofrl.StepGraph(self.ctx, self.replay, self.her, self.batch, self.nets, self.opt, qd,
                                              aux=aux_dev, v_out=self.v, pi_out=self.pi, argmax_out=self.am,
                                              loss_out=self.loss, norms_out=self.norms, grad_out=self.grad)
            self.sg.launch(k, qd, aux_dev)
            torch.cuda.synchronize()
            self.sg.sync_t()
        else:
            self.ofrl.train_step(self.ctx, self.replay, self.her, k, self.batch, qd, self.nets, self.opt,
                                 aux=aux_dev, v_out=self.v, pi_out=self.pi, argmax_out=self.am,
                                 loss_out=self.loss, norms_out=self.norms, grad_out=self.grad)
            torch.cuda.synchronize()
        return self._results()

    def _results(self):
        cpu = lambda t: t.cpu().numpy()
        return dict(batch={k2: cpu(getattr(self.batch, k2)) for k2 in
                           ("states", "next_states", "actions", "rewards", "dones", "src_idx", "donor_idx")},
                    v=cpu(self.v), pi=cpu(self.pi), argmax=cpu(self.am), loss=cpu(self.loss),
                    norms=cpu(self.norms), grad=cpu(self.grad),
                    params=[cpu(n.params) for n in self.nets], m=[cpu(n.m) for n in self.nets],
                    vmom=[cpu(n.v) for n in self.nets],
                    target=[cpu(n.target) if n.target is not None else None for n in self.nets],
                    t=[n.t for n in self.nets])

    def state(self):
        """Each network's trainable state as it is on the GPU now, as oracle
        networks (fp32 values are exact in fp64)."""
        out = []
        for n in self.nets:
            f64 = lambda t: t.cpu().numpy().astype(np.float64)
            out.append(ostep.NetState(params=f64(n.params), m=f64(n.m), v=f64(n.v), t=int(n.t), tau=f32(n.tau),
                                      target=None if n.target is None else f64(n.target), polyak=f32(n.polyak)))
        return out

    def kernels(self):
        return self.ofrl.train_step_kernels(self.ctx, self.batch, self.w.batch, self.w.n_nets)

    def close(self):
        if self.sg is not None:
            self.sg.close()
        self.ctx.close()


def oracle_nets(w, polyak=None):
    return [ostep.NetState.fresh(synth.make_params(w, k), f32(w.taus[k]), None if polyak is None else f32(polyak))
            for k in range(w.n_nets)]


def her_rows(w):
    return oher.her_count(w.batch, w.her_ratio)
