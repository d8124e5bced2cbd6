"""The five synthetic workloads of the fused IQL + HER train step.

Each workload is named by what it is and its sizes.  The values follow the
workload list of the method's benchmark; where a field is left open there,
the default of the tiny workload (Adam lr 3e-4, max_grad_norm 1.0, weight
decay 0, beta 3.0) or of the production-shaped workload (HER 'future' over a
2^20-transition buffer of 256-step episodes, goal_dim 4, Q ~ N(0, 2)) is used.

This module holds sizes and hyper-parameters only, none of the method's
arithmetic.
"""
from dataclasses import dataclass, field
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    state_dim: int
    goal_dim: int
    hidden: int
    num_actions: int
    q_sigma: float
    taus: Tuple[float, ...]          # one per V network (two for the twin workload)
    net_seeds: Tuple[int, ...]       # weight-init seed per V network
    beta: float                      # advantage temperature
    her_ratio: float
    strategy: str                    # 'final' | 'future' | 'random'
    capacity: int
    ep_len: Tuple[int, int]          # episode length range [lo, hi] (lo == hi: fixed)
    steps: int
    prec: str = "fp32"               # GEMM operand precision: 'fp32' or 'bf16'
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    max_grad_norm: float = 1.0
    goal_threshold: float = 0.01
    aux_sigmas: Tuple[float, ...] = ()   # one N(0, sigma) gradient source each
    budget: Tuple[float, ...] = (0.70, 0.15, 0.10, 0.05)
    anchor_frac: float = 0.0         # fraction of observations whose goal slice sits near one anchor

    @property
    def state_stride(self) -> int:
        """Row stride in floats: state_dim rounded up to a multiple of 8."""
        return (self.state_dim + 7) & ~7

    @property
    def n_nets(self) -> int:
        return len(self.taus)

    @property
    def her_count(self) -> int:
        """floor(batch * her_ratio): HER rows are the last her_count rows."""
        return int(self.batch * self.her_ratio)

    @property
    def n_params(self) -> int:
        s, h = self.state_dim, self.hidden
        return h * s + h + h * h + h + h + 1

    @property
    def n_aux(self) -> int:
        return len(self.aux_sigmas)


TINY = Workload(
    name="tiny_fp32_B256_S48_H64_A4", seed=1001, batch=256, state_dim=48, goal_dim=4,
    hidden=64, num_actions=4, q_sigma=1.0, taus=(0.7,), net_seeds=(1101,), beta=3.0,
    her_ratio=0.5, strategy="final", capacity=4096, ep_len=(16, 16), steps=1)

PROD = Workload(
    name="prod_fp32_B16384_S50_H128_A5", seed=1002, batch=16384, state_dim=50, goal_dim=4,
    hidden=128, num_actions=5, q_sigma=2.0, taus=(0.7,), net_seeds=(1102,), beta=3.0,
    her_ratio=0.25, strategy="future", capacity=1 << 20, ep_len=(256, 256), steps=100)

TWIN = Workload(
    name="twin_bf16_B16384_S50_H128_A5", seed=1003, batch=16384, state_dim=50, goal_dim=4,
    hidden=128, num_actions=5, q_sigma=2.0, taus=(0.9, 0.5), net_seeds=(2003, 2004), beta=3.0,
    her_ratio=0.25, strategy="future", capacity=1 << 20, ep_len=(256, 256), steps=100,
    prec="bf16")

HER_HEAVY = Workload(
    name="her_heavy_fp32_B65536_S50_H128_A5", seed=1004, batch=65536, state_dim=50, goal_dim=8,
    hidden=128, num_actions=5, q_sigma=2.0, taus=(0.7,), net_seeds=(1104,), beta=3.0,
    her_ratio=0.8, strategy="random", capacity=1 << 22, ep_len=(64, 512), steps=50,
    anchor_frac=0.4472)

BUDGETED = Workload(
    name="budgeted_fp32_B16384_S50_H256_A9", seed=1005, batch=16384, state_dim=50, goal_dim=4,
    hidden=256, num_actions=9, q_sigma=2.0, taus=(0.7,), net_seeds=(1105,), beta=3.0,
    her_ratio=0.25, strategy="future", capacity=1 << 20, ep_len=(256, 256), steps=200,
    weight_decay=1e-4, aux_sigmas=(0.5, 1.0, 4.0))

ALL = (TINY, PROD, TWIN, HER_HEAVY, BUDGETED)
BY_NAME = {w.name: w for w in ALL}
