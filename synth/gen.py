"""Seeded synthetic inputs for the fused IQL + HER train step.

Both the CUDA path (through the tests and the benchmark) and the CPU oracle
take their inputs from here.  Everything is numpy on the host, seeded from
the workload's seed, so that any step's inputs can be regenerated on either
side.  Nothing here computes any part of the method: no index sampling, no
relabelling, no network, no loss, no optimiser.

Replay buffer (structure-of-arrays, the layout of the GPU replay buffer the
method reads): states and next_states [capacity, stride] fp32 (stride =
state_dim rounded up to 8, pad columns zero), actions [capacity] int32,
rewards [capacity] fp32, dones [capacity] fp32, episode_ends [num_episodes]
int32 (exclusive, ascending, last == capacity) and episode_id [capacity]
int32.  Episodes are contiguous; next_states[i] = states[i+1] inside an
episode and a fresh N(0,1) observation after its last step, where done = 1.
The features stand in for the 42 market + 8 order-flow features of the
source pipeline (all N(0,1)).
"""
import dataclasses

import numpy as np

from .configs import Workload


def scaled(w: Workload, batch=None, capacity=None, steps=None) -> Workload:
    """The same workload with a smaller batch / buffer (structure kept)."""
    kw = {}
    if batch is not None:
        kw["batch"] = batch
    if capacity is not None:
        kw["capacity"] = capacity
    if steps is not None:
        kw["steps"] = steps
    return dataclasses.replace(w, **kw)


def episode_lengths(w: Workload, rng) -> np.ndarray:
    lo, hi = w.ep_len
    if lo == hi:
        n = -(-w.capacity // lo)
        lens = np.full(n, lo, dtype=np.int64)
    else:
        # enough draws to cover the buffer, then truncate the last episode
        n = 2 * w.capacity // lo + 16
        lens = rng.integers(lo, hi + 1, size=n, dtype=np.int64)
    cum = np.cumsum(lens)
    k = int(np.searchsorted(cum, w.capacity, side="left"))
    lens = lens[: k + 1].copy()
    lens[-1] -= int(cum[k] - w.capacity)
    return lens


def make_replay(w: Workload) -> dict:
    rng = np.random.default_rng([w.seed, 0])
    cap, s, st, g = w.capacity, w.state_dim, w.state_stride, w.goal_dim
    lens = episode_lengths(w, rng)
    ends = np.cumsum(lens).astype(np.int32)
    n_eps = len(ends)

    states = np.zeros((cap, st), dtype=np.float32)
    states[:, :s] = rng.standard_normal((cap, s), dtype=np.float32)
    terminal = np.zeros((n_eps, st), dtype=np.float32)
    terminal[:, :s] = rng.standard_normal((n_eps, s), dtype=np.float32)

    if w.anchor_frac > 0.0:
        # A fraction of all observations get a goal slice within 0.0025 of one
        # anchor point, so two of them are within 0.005 of each other.  With
        # fraction f, a random pair of observations is near with probability
        # about f^2 (0.4472^2 = 0.2).
        anchor = rng.standard_normal(g).astype(np.float32)

        def place(arr):
            m = rng.random(arr.shape[0]) < w.anchor_frac
            k = int(m.sum())
            d = rng.standard_normal((k, g))
            d /= np.linalg.norm(d, axis=1, keepdims=True)
            d *= rng.uniform(0.0, 0.0025, size=(k, 1))
            arr[m, :g] = (anchor[None, :].astype(np.float64) + d).astype(np.float32)

        place(states)
        place(terminal)

    next_states = np.empty_like(states)
    next_states[:-1] = states[1:]
    next_states[ends - 1] = terminal

    actions = rng.integers(0, w.num_actions, size=cap, dtype=np.int32)
    rewards = rng.standard_normal(cap, dtype=np.float32)
    dones = np.zeros(cap, dtype=np.float32)
    dones[ends - 1] = 1.0
    episode_id = np.repeat(np.arange(n_eps, dtype=np.int32), lens)
    return dict(states=states, next_states=next_states, actions=actions, rewards=rewards,
                dones=dones, episode_ends=ends, episode_id=episode_id)


def make_params(w: Workload, net: int = 0) -> np.ndarray:
    """Flat V parameters W1[H,S], b1[H], W2[H,H], b2[H], W3[1,H], b3[1], fp32.

    Kaiming-uniform with ReLU gain for weights (U(+-sqrt(6/fan_in))), and
    U(+-1/sqrt(fan_in)) for biases.
    """
    rng = np.random.default_rng(w.net_seeds[net])
    s, h = w.state_dim, w.hidden

    def lin(fan_out, fan_in):
        wb = np.sqrt(6.0 / fan_in)
        bb = 1.0 / np.sqrt(fan_in)
        return (rng.uniform(-wb, wb, size=(fan_out, fan_in)),
                rng.uniform(-bb, bb, size=fan_out))

    w1, b1 = lin(h, s)
    w2, b2 = lin(h, h)
    w3, b3 = lin(1, h)
    flat = np.concatenate([w1.ravel(), b1, w2.ravel(), b2, w3.ravel(), b3]).astype(np.float32)
    assert flat.size == w.n_params
    return flat


def make_q(w: Workload, step: int, batch=None) -> np.ndarray:
    """Q[B, A] ~ N(0, q_sigma^2), fp32, with entries of a row at least 1e-4 apart."""
    b = w.batch if batch is None else batch
    rng = np.random.default_rng([w.seed, 1, step])
    q = (rng.standard_normal((b, w.num_actions)) * w.q_sigma).astype(np.float32)
    while True:
        srt = np.sort(q, axis=1)
        bad = np.nonzero((np.diff(srt, axis=1) < 1e-4).any(axis=1))[0]
        if bad.size == 0:
            return q
        q[bad] = (rng.standard_normal((bad.size, w.num_actions)) * w.q_sigma).astype(np.float32)


def make_aux(w: Workload, step: int, net: int = 0) -> np.ndarray:
    """Auxiliary gradient sources [n_aux, P] ~ N(0, sigma_k^2), fp32."""
    rng = np.random.default_rng([w.seed, 2, step, net])
    out = np.empty((w.n_aux, w.n_params), dtype=np.float32)
    for k, sg in enumerate(w.aux_sigmas):
        out[k] = (rng.standard_normal(w.n_params) * sg).astype(np.float32)
    return out
