"""The fused IQL + HER train step, composed from the oracle's parts.

Order of one step (for each V network; twin networks share the batch and Q):
  1. HER index sampling and relabel ("GPU IQL + HER Porting Plan", "Phase 3:
     Combined IQL + HER": HER produces the relabelled batch that feeds the
     training step; "How HER Interacts with GPU PER": normal rows, then HER).
  2. V forward, expectile loss on Q(s, a_taken) with a_taken the batch's
     (copied) action, advantage-weighted policy, V backward into the primary
     gradient ("CUDA Kernel: iql_value_kernel.cu").
  3. Budgeted clip of the primary (0.70) plus clipped SAXPY of each auxiliary
     source ("Gradient Stability ...", "Proper design", pipeline steps 2-6).
  4. t <- t + 1, then Adam with its safety clip at max_grad_norm (pipeline
     step 7; the step counter is incremented before Adam reads it, "DQN
     Backward-Path NaN Audit", Adam findings), the optional weight bound
     after the update, and the optional Polyak update of the network's
     target copy ("GPU IQL + HER Porting Plan", target_ema_update).

The twin workload runs two networks (high and low tau) with identical shapes
and independent weights on one batch ("Phase 2: Multi-Stream Graph
Parallelism", "2C. Grouped GEMM for IQL").
"""
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import her, iql, optim, precision


@dataclass
class NetState:
    params: np.ndarray          # flat, fp64
    m: np.ndarray
    v: np.ndarray
    t: int = 0
    tau: float = 0.7
    target: Optional[np.ndarray] = None   # Polyak target copy, or None
    polyak: float = 0.0

    @classmethod
    def fresh(cls, params, tau, polyak=None):
        p = np.asarray(params, dtype=np.float64).copy()
        return cls(params=p, m=np.zeros_like(p), v=np.zeros_like(p), t=0, tau=float(tau),
                   target=None if polyak is None else p.copy(), polyak=float(polyak or 0.0))


@dataclass
class StepConfig:
    state_dim: int
    hidden: int
    num_actions: int
    goal_dim: int
    batch: int
    her_rows: int
    strategy: int
    goal_threshold: float
    seed: int
    beta: float
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    max_grad_norm: float
    budget: tuple = optim.BUDGET
    alpha: tuple = (1.0, 1.0, 1.0, 1.0)
    weight_clamp_max_abs: float = 0.0
    sanitize_sources: bool = False
    prec: str = "fp32"          # 'bf16': GEMM operands rounded to bf16 (oracle/precision.py)

    def gemm_operand(self):
        return precision.bf16 if self.prec == "bf16" else None


def config_from_workload(w) -> StepConfig:
    return StepConfig(
        state_dim=w.state_dim, hidden=w.hidden, num_actions=w.num_actions,
        goal_dim=w.goal_dim, batch=w.batch, her_rows=her.her_count(w.batch, w.her_ratio),
        strategy=her.STRATEGY[w.strategy], goal_threshold=w.goal_threshold, seed=w.seed,
        beta=w.beta, lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
        weight_decay=w.weight_decay, max_grad_norm=w.max_grad_norm,
        budget=tuple(w.budget), prec=w.prec)


def train_step(cfg: StepConfig, replay: dict, step: int, q, nets, aux=None):
    """One fused step.  `nets` (list of NetState) is updated in place.

    aux: per network, an [n_aux, P] array of auxiliary gradient sources (or
    None).  Returns a dict of the step's outputs, per network where relevant.
    """
    src, donor = her.sample_indices(cfg.seed, step, cfg.batch, cfg.her_rows, cfg.strategy,
                                    replay["states"].shape[0], replay.get("episode_ends"))
    batch = her.relabel(replay, src, donor, cfg.goal_dim, cfg.goal_threshold)
    qt = iql.q_taken(q, batch["actions"])
    out = dict(batch=batch, v=[], loss=[], pi=[], argmax=[], grad=[], combined=[],
               combined_abs=[], norms=[], skipped=[])
    for k, net in enumerate(nets):
        rnd = cfg.gemm_operand()
        v, act = iql.forward(net.params, batch["states"], cfg.state_dim, cfg.hidden, rnd)
        loss, dv = iql.expectile_loss(qt, v, net.tau)
        pi, am = iql.policy(q, v, cfg.beta)
        g0 = iql.backward(net.params, act, dv, cfg.state_dim, cfg.hidden, rnd)
        g0_abs = iql.backward_abs(net.params, act, dv, cfg.state_dim, cfg.hidden)
        sources = [g0]
        if aux is not None and aux[k] is not None:
            sources += [np.asarray(a, dtype=np.float64) for a in aux[k]]
        n = len(sources)
        if cfg.sanitize_sources:
            sources = [optim.sanitize(x) for x in sources]
        g, norms = optim.budgeted_combine(sources, cfg.budget[:n], cfg.alpha[:n], cfg.max_grad_norm)
        # magnitude scale of each combined element: |coef_0| * sum|terms of g0|
        # plus |coef_k g_k| for the (exact) auxiliary inputs
        g_abs = np.zeros_like(g)
        for k, src in enumerate(sources):
            c = abs(float(cfg.alpha[k]) * optim.clip_scale(norms[k], float(cfg.budget[k]) * cfg.max_grad_norm))
            g_abs += c * (g0_abs if k == 0 else np.abs(src))
        net.t += 1
        net.params, net.m, net.v, skipped = optim.adam(
            net.params, g, net.m, net.v, net.t, cfg.lr, cfg.beta1, cfg.beta2, cfg.eps,
            cfg.weight_decay, cfg.max_grad_norm, norms[-1], cfg.weight_clamp_max_abs)
        if net.target is not None:
            net.target = optim.polyak(net.target, net.params, net.polyak)
        full = np.zeros(5)
        full[:n] = norms[:n]
        full[4] = norms[-1]
        out["v"].append(v)
        out["loss"].append(loss)
        out["pi"].append(pi)
        out["argmax"].append(am)
        out["grad"].append(g0)
        out["combined"].append(g)
        out["combined_abs"].append(g_abs)
        out["norms"].append(full)
        out["skipped"].append(skipped)
    return out
