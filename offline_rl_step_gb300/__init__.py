"""GB300 (sm_103a) fused offline-RL train step: HER relabel + IQL value update.

A thin Python binding over the C ABI of include/ofrl.h.  Every function
marshals torch CUDA tensors into device pointers and calls the library on
the current torch stream; all arithmetic runs in the library's CUDA kernels.
There is no CPU path: if libofrl.so is missing, importing the binding's
calls raises.

Functions (same names as the C entry points, without the ofrl_ prefix):
  Context(...)                  ofrl_create / ofrl_destroy / ofrl_poll_status
  her_relabel(...)              HER index sampling + gather + relabel
  iql_value_fwd_bwd(...)        V forward + expectile loss + V backward
  expectile_loss(...)           expectile loss and dL/dV
  adv_weighted_policy(...)      softmax(beta * clamp(Q - V, -10, 10)), argmax
  budgeted_clip_saxpy(...)      budgeted per-source clip + SAXPY, norms
  adam_step(...)                Adam with the safety clip
  train_step(...)               the fused step composed of the above
"""
import ctypes as C
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

from . import _abi
from ._abi import (HER_EPISODE, HER_FINAL, HER_FUTURE, HER_RANDOM, PREC_BF16, PREC_FP32,  # noqa: F401
                   STAT_BAD_ACTION, STAT_BAD_INDEX, STAT_NONFINITE_GRAD, STAT_SANITIZED, STAT_TIMEOUT, OfrlError)

STRATEGY = {"final": HER_FINAL, "future": HER_FUTURE, "random": HER_RANDOM, "episode": HER_EPISODE}
PRECISION = {"fp32": PREC_FP32, "bf16": PREC_BF16}
BUDGET = (0.70, 0.15, 0.10, 0.05)


def n_params(state_dim: int, hidden: int) -> int:
    return hidden * state_dim + hidden + hidden * hidden + hidden + hidden + 1


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor", host_ok=False):
    """Address of a CUDA tensor; with host_ok also of a pinned CPU tensor (page-locked host memory the
    kernels read or write in place over the host link)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (host_ok and t.is_pinned())):
        raise TypeError(f"{name} must be a CUDA tensor" + (" or a pinned CPU tensor" if host_ok else ""))
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _host_ptr(t: Optional[torch.Tensor], name="tensor"):
    """A page-locked float32 CPU tensor (the graph's host copies need pinned memory)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
        raise TypeError(f"{name} must be a pinned CPU tensor")
    if t.dtype != F32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous float32 tensor")
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


F32, I32 = torch.float32, torch.int32


@dataclass
class Replay:
    """Replay buffer (device tensors): states/next_states [capacity, stride]."""
    states: torch.Tensor
    next_states: torch.Tensor
    actions: torch.Tensor
    rewards: torch.Tensor
    dones: torch.Tensor
    state_dim: int
    goal_dim: int
    episode_ends: Optional[torch.Tensor] = None

    def c(self):
        cap, stride = self.states.shape
        ne = 0 if self.episode_ends is None else int(self.episode_ends.numel())
        return _abi.Replay(_ptr(self.states, F32, "states"), _ptr(self.next_states, F32, "next_states"),
                           _ptr(self.actions, I32, "actions"), _ptr(self.rewards, F32, "rewards"),
                           _ptr(self.dones, F32, "dones"), _ptr(self.episode_ends, I32, "episode_ends"),
                           cap, ne, self.state_dim, stride, self.goal_dim)


@dataclass
class HerConfig:
    batch: int
    her_count: int
    strategy: str = "future"
    goal_threshold: float = 0.01
    seed: int = 0

    def c(self):
        return _abi.HerCfg(self.batch, self.her_count, STRATEGY[self.strategy], self.goal_threshold,
                           self.seed & ((1 << 64) - 1))


@dataclass
class Batch:
    """Relabelled batch (device tensors), written by her_relabel / train_step."""
    states: torch.Tensor
    next_states: torch.Tensor
    actions: torch.Tensor
    rewards: torch.Tensor
    dones: torch.Tensor
    src_idx: torch.Tensor
    donor_idx: torch.Tensor

    @classmethod
    def empty(cls, batch: int, stride: int, device="cuda"):
        f = dict(device=device, dtype=F32)
        i = dict(device=device, dtype=I32)
        return cls(torch.empty(batch, stride, **f), torch.empty(batch, stride, **f), torch.empty(batch, **i),
                   torch.empty(batch, **f), torch.empty(batch, **f), torch.empty(batch, **i),
                   torch.empty(batch, **i))

    def c(self):
        return _abi.Batch(_ptr(self.states, F32, "batch.states"), _ptr(self.next_states, F32, "batch.next_states"),
                          _ptr(self.actions, I32, "batch.actions"), _ptr(self.rewards, F32, "batch.rewards"),
                          _ptr(self.dones, F32, "batch.dones"), _ptr(self.src_idx, I32, "batch.src_idx"),
                          _ptr(self.donor_idx, I32, "batch.donor_idx"), self.states.shape[1])


@dataclass
class VNet:
    """One V network's trainable state: params, Adam moments m and v, step t; optionally a Polyak target copy
    that train_step moves toward the weights after every update (target = (1 - polyak) target + polyak params)."""
    params: torch.Tensor
    m: torch.Tensor
    v: torch.Tensor
    tau: float
    t: int = 0
    target: Optional[torch.Tensor] = None
    polyak: float = 0.0

    @classmethod
    def from_params(cls, params: torch.Tensor, tau: float, polyak: Optional[float] = None):
        p = params.detach().to(device="cuda", dtype=F32).contiguous().clone()
        tgt = p.clone() if polyak is not None else None
        return cls(p, torch.zeros_like(p), torch.zeros_like(p), float(tau), 0, tgt, float(polyak or 0.0))

    def c(self):
        return _abi.VNet(_ptr(self.params, F32, "params"), _ptr(self.m, F32, "m"), _ptr(self.v, F32, "v"),
                         self.t, self.tau, _ptr(self.target, F32, "target"), self.polyak)


@dataclass
class Opt:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    max_grad_norm: float = 1.0
    beta: float = 3.0
    budget: Sequence[float] = BUDGET
    alpha: Sequence[float] = (1.0, 1.0, 1.0, 1.0)
    weight_clamp_max_abs: float = 0.0    # > 0: |weight| bound after every Adam update
    sanitize_sources: bool = False       # non-finite gradient-source elements count as 0

    def c(self):
        b = (C.c_float * 4)(*[float(x) for x in (list(self.budget) + [0.0] * 4)[:4]])
        a = (C.c_float * 4)(*[float(x) for x in (list(self.alpha) + [0.0] * 4)[:4]])
        return _abi.Opt(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, self.max_grad_norm,
                        self.beta, b, a, self.weight_clamp_max_abs, 1 if self.sanitize_sources else 0)


# V forward/backward implementations (OFRL_VNET_* in ofrl.h)
VNET_PATHS = {"auto": 0, "tc_fused": 1, "tc_layered": 2, "cuda_cores": 3}


class Context:
    """Device workspace for one V-network shape (ofrl_create); the only allocation."""

    def __init__(self, state_dim: int, hidden: int, num_actions: int, prec: str = "fp32",
                 max_batch: int = 16384, max_nets: int = 1):
        self._lib = _abi.load()
        self.shape = _abi.VShape(state_dim, hidden, num_actions, PRECISION[prec])
        self.state_dim, self.hidden, self.num_actions, self.prec = state_dim, hidden, num_actions, prec
        self.max_batch, self.max_nets = max_batch, max_nets
        self.n_params = n_params(state_dim, hidden)
        h = C.c_void_p()
        _abi.check("ofrl_create", self._lib.ofrl_create(C.byref(self.shape), max_batch, max_nets, C.byref(h)))
        self.handle = h

    def close(self):
        if self.handle is not None and self.handle.value:
            _abi.check("ofrl_destroy", self._lib.ofrl_destroy(self.handle))
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def poll_status(self, stream=None):
        words = (C.c_int32 * _abi.STAT_WORDS)()
        _abi.check("ofrl_poll_status", self._lib.ofrl_poll_status(self.handle, _stream(stream), words))
        return {"nonfinite_grad": words[_abi.STAT_NONFINITE_GRAD], "bad_action": words[_abi.STAT_BAD_ACTION],
                "bad_index": words[_abi.STAT_BAD_INDEX], "timeout": words[_abi.STAT_TIMEOUT],
                "sanitized": words[_abi.STAT_SANITIZED]}

    def workspace_bytes(self) -> int:
        return int(self._lib.ofrl_workspace_bytes(C.byref(self.shape), self.max_batch, self.max_nets))

    def select_vnet_path(self, path: str):
        """Which V forward/backward implementation later calls take: auto, tc_fused, tc_layered, cuda_cores."""
        _abi.check("ofrl_select_vnet_path", self._lib.ofrl_select_vnet_path(self.handle, VNET_PATHS[path]))

    def vnet_path(self, n_nets: int = 1) -> str:
        """The implementation a train step of n_nets networks takes on this context."""
        k = int(self._lib.ofrl_vnet_path(self.handle, n_nets))
        names = {v: n for n, v in VNET_PATHS.items()}
        if k not in names:
            raise ValueError(f"ofrl_vnet_path: invalid arguments (n_nets={n_nets})")
        return names[k]


def her_relabel(ctx: Context, replay: Replay, her: HerConfig, step: int, out: Batch, stream=None):
    r, h, b = replay.c(), her.c(), out.c()
    _abi.check("ofrl_her_relabel", ctx._lib.ofrl_her_relabel(ctx.handle, C.byref(r), C.byref(h), step,
                                                              C.byref(b), _stream(stream)))


def her_relabel_sources(ctx: Context, replay: Replay, her: HerConfig, step: int, src_idx, out: Batch,
                        is_weights=None, is_weights_out=None, stream=None):
    """her_relabel with the caller's (e.g. PER-sampled) source of every row; HER rows get importance weight 1."""
    r, h, b = replay.c(), her.c(), out.c()
    _abi.check("ofrl_her_relabel_sources", ctx._lib.ofrl_her_relabel_sources(
        ctx.handle, C.byref(r), C.byref(h), step, _ptr(src_idx, I32, "src_idx"), _ptr(is_weights, F32, "is_weights"),
        C.byref(b), _ptr(is_weights_out, F32, "is_weights_out"), _stream(stream)))


def episode_ends_append(ctx: Context, dones, first_index: int, episode_ends, num_episodes, stream=None):
    """Append the exclusive end of every done transition among the n = dones.numel() new ones stored at
    first_index.. to episode_ends (device int32, in order), growing the device counter num_episodes."""
    _abi.check("ofrl_episode_ends_append", ctx._lib.ofrl_episode_ends_append(
        ctx.handle, _ptr(dones, F32, "dones"), int(first_index), int(dones.numel()), _ptr(episode_ends, I32, "episode_ends"),
        _ptr(num_episodes, I32, "num_episodes"), int(episode_ends.numel()), _stream(stream)))


def iql_value_fwd_bwd(ctx: Context, params, states, q_taken, tau: float, v_out, loss_out, grad_out,
                      stream=None):
    batch = int(q_taken.numel())
    _abi.check("ofrl_iql_value_fwd_bwd", ctx._lib.ofrl_iql_value_fwd_bwd(
        ctx.handle, _ptr(params, F32, "params"), _ptr(states, F32, "states"), states.shape[1], batch,
        _ptr(q_taken, F32, "q_taken"), tau, _ptr(v_out, F32, "v_out"), _ptr(loss_out, F32, "loss_out"),
        _ptr(grad_out, F32, "grad_out"), _stream(stream)))


def forward_values(ctx: Context, params, states, v_out, stream=None):
    """V(s) of every row of `states` [batch, stride] into v_out [batch] (forward only)."""
    _abi.check("ofrl_forward_values", ctx._lib.ofrl_forward_values(
        ctx.handle, _ptr(params, F32, "params"), _ptr(states, F32, "states"), states.shape[1],
        int(states.shape[0]), _ptr(v_out, F32, "v_out"), _stream(stream)))


def iql_target(ctx: Context, params, next_states, rewards, dones, gamma: float, target_out, v_next_out=None,
               stream=None):
    """target_out = rewards + gamma (1 - dones) V(next_states); V(s') into v_next_out when given."""
    _abi.check("ofrl_iql_target", ctx._lib.ofrl_iql_target(
        ctx.handle, _ptr(params, F32, "params"), _ptr(next_states, F32, "next_states"), next_states.shape[1],
        _ptr(rewards, F32, "rewards"), _ptr(dones, F32, "dones"), int(next_states.shape[0]), gamma,
        _ptr(v_next_out, F32, "v_next_out"), _ptr(target_out, F32, "target_out"), _stream(stream)))


def noalloc_max_batch(state_dim: int, hidden: int, num_actions: int, prec: str = "fp32") -> int:
    """Largest batch iql_value_fwd_bwd_noalloc accepts for this shape."""
    shape = _abi.VShape(state_dim, hidden, num_actions, PRECISION[prec])
    return int(_abi.load().ofrl_noalloc_max_batch(C.byref(shape)))


def iql_value_fwd_bwd_noalloc(state_dim: int, hidden: int, num_actions: int, params, states, q_taken,
                              tau: float, v_out, loss_out, grad_out, prec: str = "fp32", stream=None):
    """iql_value_fwd_bwd for callers that may not allocate device memory.

    No Context: the library's own fixed scratch array is used (see the C
    header), so nothing is allocated.  Calls that overlap on the GPU share
    that scratch and race: issue them on one stream.
    """
    lib = _abi.load()
    shape = _abi.VShape(state_dim, hidden, num_actions, PRECISION[prec])
    batch = int(q_taken.numel())
    _abi.check("ofrl_iql_value_fwd_bwd_noalloc", lib.ofrl_iql_value_fwd_bwd_noalloc(
        C.byref(shape), _ptr(params, F32, "params"), _ptr(states, F32, "states"), states.shape[1], batch,
        _ptr(q_taken, F32, "q_taken"), tau, _ptr(v_out, F32, "v_out"), _ptr(loss_out, F32, "loss_out"),
        _ptr(grad_out, F32, "grad_out"), _stream(stream)))


def expectile_loss(ctx: Context, q_taken, v, tau: float, loss_out, dv_out=None, stream=None):
    _abi.check("ofrl_expectile_loss", ctx._lib.ofrl_expectile_loss(
        ctx.handle, _ptr(q_taken, F32, "q_taken"), _ptr(v, F32, "v"), int(v.numel()), tau,
        _ptr(loss_out, F32, "loss_out"), _ptr(dv_out, F32, "dv_out"), _stream(stream)))


def adv_weighted_policy(ctx: Context, q, v, beta: float, pi_out, argmax_out=None, stream=None):
    b, a = q.shape
    _abi.check("ofrl_adv_weighted_policy", ctx._lib.ofrl_adv_weighted_policy(
        ctx.handle, _ptr(q, F32, "q"), _ptr(v, F32, "v"), b, a, beta, _ptr(pi_out, F32, "pi_out"),
        _ptr(argmax_out, I32, "argmax_out"), _stream(stream)))


def budgeted_clip_saxpy(ctx: Context, sources: List[torch.Tensor], budget_frac, alpha, max_grad_norm: float,
                        grad_out, norms_out=None, stream=None):
    k = len(sources)
    n = int(sources[0].numel())
    ptrs = (C.c_void_p * k)(*[_ptr(s, F32, "source").value for s in sources])
    bf = (C.c_float * k)(*[float(x) for x in budget_frac[:k]])
    al = (C.c_float * k)(*[float(x) for x in alpha[:k]])
    _abi.check("ofrl_budgeted_clip_saxpy", ctx._lib.ofrl_budgeted_clip_saxpy(
        ctx.handle, ptrs, bf, al, k, n, max_grad_norm, _ptr(grad_out, F32, "grad_out"),
        _ptr(norms_out, F32, "norms_out"), _stream(stream)))


def adam_step(ctx: Context, p, g, m, v, t: int, opt: Opt, grad_norm=None, stream=None):
    o = opt.c()
    _abi.check("ofrl_adam_step", ctx._lib.ofrl_adam_step(
        ctx.handle, _ptr(p, F32, "p"), _ptr(g, F32, "g"), _ptr(m, F32, "m"), _ptr(v, F32, "v"), int(p.numel()),
        t, C.byref(o), _ptr(grad_norm, F32, "grad_norm"), _stream(stream)))


def train_step(ctx: Context, replay: Replay, her: HerConfig, step: int, batch: Batch, q, nets: List[VNet],
               opt: Opt, aux: Optional[List[List[torch.Tensor]]] = None, v_out=None, pi_out=None,
               argmax_out=None, loss_out=None, norms_out=None, grad_out=None, stream=None):
    """One fused step; increments every net's t."""
    r, h, b, o = replay.c(), her.c(), batch.c(), opt.c()
    n_nets = len(nets)
    cn = (_abi.VNet * n_nets)(*[x.c() for x in nets])
    n_aux = 0 if not aux else len(aux[0])
    aux_arr = None
    if n_aux:
        flat = [_ptr(t, F32, "aux").value for per in aux for t in per]
        aux_arr = (C.c_void_p * len(flat))(*flat)
    _abi.check("ofrl_train_step", ctx._lib.ofrl_train_step(
        ctx.handle, C.byref(r), C.byref(h), step, C.byref(b), _ptr(q, F32, "q", host_ok=True), cn, n_nets, C.byref(o),
        aux_arr, n_aux, _ptr(v_out, F32, "v_out"), _ptr(pi_out, F32, "pi_out"),
        _ptr(argmax_out, I32, "argmax_out"), _ptr(loss_out, F32, "loss_out", host_ok=True),
        _ptr(norms_out, F32, "norms_out", host_ok=True), _ptr(grad_out, F32, "grad_out"), _stream(stream)))
    for k in range(n_nets):
        nets[k].t = cn[k].t


class StepPlan:
    """train_step with every argument marshalled once.

    Per call only the step index, the Q pointer and the optional auxiliary
    source pointers change; the networks' t counters live in the C array and
    advance there.  Same semantics as train_step.
    """

    def __init__(self, ctx: Context, replay: Replay, her: HerConfig, batch: Batch, nets: List[VNet], opt: Opt,
                 n_aux: int = 0, v_out=None, pi_out=None, argmax_out=None, loss_out=None, norms_out=None,
                 grad_out=None):
        self.ctx, self.nets = ctx, nets
        self._keep = (replay, batch, nets, v_out, pi_out, argmax_out, loss_out, norms_out, grad_out)
        self.r, self.h, self.b, self.o = replay.c(), her.c(), batch.c(), opt.c()
        self.n_nets = len(nets)
        self.cn = (_abi.VNet * self.n_nets)(*[x.c() for x in nets])
        self.n_aux = n_aux
        self.aux_arr = (C.c_void_p * max(1, self.n_nets * n_aux))()
        self.outs = [_ptr(v_out, F32), _ptr(pi_out, F32), _ptr(argmax_out, I32), _ptr(loss_out, F32, host_ok=True),
                     _ptr(norms_out, F32, host_ok=True), _ptr(grad_out, F32)]
        self.fn = ctx._lib.ofrl_train_step
        self.rp, self.hp, self.bp, self.op = C.byref(self.r), C.byref(self.h), C.byref(self.b), C.byref(self.o)

    def run(self, step: int, q: torch.Tensor, aux=None, stream=None):
        if self.n_aux:
            flat = [t.data_ptr() for per in aux for t in per]
            for i, p in enumerate(flat):
                self.aux_arr[i] = p
        code = self.fn(self.ctx.handle, self.rp, self.hp, step, self.bp, C.c_void_p(q.data_ptr()), self.cn,
                       self.n_nets, self.op, self.aux_arr if self.n_aux else None, self.n_aux, *self.outs,
                       _stream(stream))
        if code != _abi.OK:
            _abi.check("ofrl_train_step", code)

    def sync_t(self):
        for k in range(self.n_nets):
            self.nets[k].t = self.cn[k].t

    def reload_t(self):
        """Take each network's t from the VNet objects (after steps made by other means, e.g. a StepGraph)."""
        for k in range(self.n_nets):
            self.cn[k].t = self.nets[k].t

    def kernels(self) -> int:
        """Kernel launches one run() makes (4, or 3 when the reduce and Adam run as one launch)."""
        return int(self.ctx._lib.ofrl_train_step_kernels(self.ctx.handle, self.bp, self.h.batch, self.n_nets))


def target_ema(params, target, polyak: float, stream=None):
    """target = (1 - polyak) target + polyak params, element-wise (Polyak averaging of a target network)."""
    if params.numel() != target.numel():
        raise ValueError("params and target differ in size")
    _abi.check("ofrl_target_ema", _abi.load().ofrl_target_ema(
        _ptr(params, F32, "params"), _ptr(target, F32, "target"), int(params.numel()), polyak, _stream(stream)))


class StepGraph:
    """train_step captured once as a CUDA graph; launch() replays it as a given step.

    Same semantics as train_step: per launch the step index, and optionally the Q tensor and the auxiliary
    sources, change; each network's t advances.  Every other tensor is the one given here (keep them alive).
    One graph launch on the host per step.
    """

    def __init__(self, ctx: Context, replay: Replay, her: HerConfig, batch: Batch, nets: List[VNet], opt: Opt, q,
                 aux=None, v_out=None, pi_out=None, argmax_out=None, loss_out=None, norms_out=None, grad_out=None,
                 q_host=None, loss_host=None, norms_host=None):
        """q, loss_out and norms_out may be pinned CPU tensors, as for train_step (Q staged by the relabel,
        loss and norms written in place).  q_host / loss_host / norms_host (pinned CPU tensors, with device
        q, loss_out, norms_out): the graph also copies Q in from q_host and the loss and norms out to
        loss_host / norms_host; replay it with launch_io."""
        self.ctx, self.nets = ctx, nets
        self._keep = [replay, batch, nets, q, aux, v_out, pi_out, argmax_out, loss_out, norms_out, grad_out,
                      q_host, loss_host, norms_host]
        self.r, self.h, self.b, self.o = replay.c(), her.c(), batch.c(), opt.c()
        self.n_nets = len(nets)
        self.cn = (_abi.VNet * self.n_nets)(*[x.c() for x in nets])
        self.n_aux = 0 if not aux else len(aux[0])
        self.aux_arr = (C.c_void_p * max(1, self.n_nets * self.n_aux))()
        if self.n_aux:
            for i, t in enumerate(t for per in aux for t in per):
                self.aux_arr[i] = _ptr(t, F32, "aux").value
        handle = C.c_void_p()
        args = (ctx.handle, C.byref(self.r), C.byref(self.h), C.byref(self.b), _ptr(q, F32, "q", host_ok=True), self.cn,
                self.n_nets, C.byref(self.o), self.aux_arr if self.n_aux else None, self.n_aux,
                _ptr(v_out, F32, "v_out"), _ptr(pi_out, F32, "pi_out"), _ptr(argmax_out, I32, "argmax_out"),
                _ptr(loss_out, F32, "loss_out", host_ok=True), _ptr(norms_out, F32, "norms_out", host_ok=True),
                _ptr(grad_out, F32, "grad_out"))
        self.io = q_host is not None or loss_host is not None or norms_host is not None
        if self.io:
            _abi.check("ofrl_step_graph_create_io", ctx._lib.ofrl_step_graph_create_io(
                *args, _host_ptr(q_host, "q_host"), _host_ptr(loss_host, "loss_host"),
                _host_ptr(norms_host, "norms_host"), C.byref(handle)))
        else:
            _abi.check("ofrl_step_graph_create", ctx._lib.ofrl_step_graph_create(*args, C.byref(handle)))
        self.handle = handle
        self.fn = ctx._lib.ofrl_step_graph_launch
        self.fn_io = ctx._lib.ofrl_step_graph_launch_io

    def launch_io(self, step: int, q_host=None, aux=None, loss_host=None, norms_host=None, stream=None):
        """Replay as step `step` with this step's host buffers (pinned CPU tensors; None keeps the previous)."""
        arr = None
        if aux is not None:
            self._keep.append(aux)
            for i, t in enumerate(t for per in aux for t in per):
                self.aux_arr[i] = t.data_ptr()
            arr = self.aux_arr
        for t in (q_host, loss_host, norms_host):
            if t is not None:
                self._keep.append(t)
        code = self.fn_io(self.handle, step, _host_ptr(q_host, "q_host"), arr, _host_ptr(loss_host, "loss_host"),
                          _host_ptr(norms_host, "norms_host"), _stream(stream))
        if code != _abi.OK:
            _abi.check("ofrl_step_graph_launch_io", code)
        if len(self._keep) > 64:
            del self._keep[14:-8]

    def launch(self, step: int, q=None, aux=None, stream=None):
        arr = None
        if aux is not None:
            self._keep.append(aux)
            for i, t in enumerate(t for per in aux for t in per):
                self.aux_arr[i] = t.data_ptr()
            arr = self.aux_arr
        if q is not None:
            self._keep[3] = q
        code = self.fn(self.handle, step, C.c_void_p(q.data_ptr()) if q is not None else None, arr,
                       _stream(stream))
        if code != _abi.OK:
            _abi.check("ofrl_step_graph_launch", code)
        if len(self._keep) > 64:
            del self._keep[14:-8]

    def sync_t(self):
        for k in range(self.n_nets):
            self.nets[k].t = self.cn[k].t

    def close(self):
        if self.handle:
            self.ctx._lib.ofrl_step_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def train_step_kernels(ctx: Context, batch: Batch, rows: int, n_nets: int = 1) -> int:
    """Kernel launches one train_step makes for this batch (4, or 3 when the reduce and Adam run as one launch)."""
    b = batch.c()
    return int(ctx._lib.ofrl_train_step_kernels(ctx.handle, C.byref(b), rows, n_nets))


def profile_begin(ctx: Context, max_steps: int):
    _abi.check("ofrl_profile_begin", ctx._lib.ofrl_profile_begin(ctx.handle, max_steps))


def profile_end(ctx: Context):
    """Per-phase device milliseconds summed over the profiled steps, and the step count."""
    ms = (C.c_float * len(_abi.PHASES))()
    n = C.c_int32()
    _abi.check("ofrl_profile_end", ctx._lib.ofrl_profile_end(ctx.handle, ms, C.byref(n)))
    return dict(zip(_abi.PHASES, list(ms))), int(n.value)
