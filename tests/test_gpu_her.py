"""GPU parity: HER index sampling + relabel, bit-exact against the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from _gpu import assert_bits, dev, f32, need_gpu, replay_dev, replay_np
from oracle import her as oher

pytestmark = pytest.mark.gpu


def _run(w, step=0, her_rows=None, batch=None):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    b = w.batch if batch is None else batch
    nh = oher.her_count(b, w.her_ratio) if her_rows is None else her_rows
    rep = replay_np(w)
    replay = replay_dev(w, rep)
    ctx = ofrl.Context(w.state_dim, w.hidden, w.num_actions, max_batch=max(b, 1))
    out = ofrl.Batch.empty(b, w.state_stride)
    ofrl.her_relabel(ctx, replay, ofrl.HerConfig(b, nh, w.strategy, w.goal_threshold, w.seed), step, out)
    torch.cuda.synchronize()
    src, donor = oher.sample_indices(w.seed, step, b, nh, oher.STRATEGY[w.strategy], w.capacity,
                                     rep["episode_ends"])
    ref = oher.relabel(rep, src, donor, w.goal_dim, f32(w.goal_threshold))
    s = w.state_dim
    assert_bits(out.src_idx.cpu().numpy(), ref["src_idx"], "src_idx")
    assert_bits(out.donor_idx.cpu().numpy(), ref["donor_idx"], "donor_idx")
    assert_bits(out.states.cpu().numpy()[:, :s], ref["states"][:, :s], "states")
    assert_bits(out.next_states.cpu().numpy()[:, :s], ref["next_states"][:, :s], "next_states")
    assert_bits(out.actions.cpu().numpy(), ref["actions"], "actions")
    assert_bits(out.rewards.cpu().numpy(), ref["rewards"], "rewards")
    assert_bits(out.dones.cpu().numpy(), ref["dones"], "dones")
    status = ctx.poll_status()
    assert status["bad_index"] == 0
    ctx.close()
    return ref


@pytest.mark.parametrize("w", [synth.TINY, synth.PROD, synth.HER_HEAVY], ids=lambda w: w.name)
def test_relabel_full_size(w):
    ref = _run(w, step=3)
    r = ref["rewards"][ref["donor_idx"] >= 0]
    # both reward branches fire on every workload
    assert (r == np.float32(1.0)).any() and (r == np.float32(-0.01)).any()


@pytest.mark.parametrize("strategy", ["final", "future", "random"])
@pytest.mark.parametrize("batch", [1, 15, 17, 1000, 40001])   # 40001: the 16-rows-per-warp kernel, ragged
def test_relabel_ragged_batches(strategy, batch):
    w = dataclasses.replace(synth.TINY, strategy=strategy, ep_len=(5, 40), capacity=3000)
    _run(w, step=11, batch=batch)


@pytest.mark.parametrize("her_rows", [0, 1, 256])
def test_relabel_her_row_counts(her_rows):
    _run(synth.TINY, step=2, her_rows=her_rows)


def test_relabel_goal_dim_edges():
    # g = S (every column is goal) and an odd state_dim whose rows have pad columns
    w = dataclasses.replace(synth.TINY, state_dim=13, goal_dim=13, capacity=2048)
    _run(w, step=1)
    w = dataclasses.replace(synth.TINY, state_dim=13, goal_dim=1, capacity=2048)
    _run(w, step=1)


def test_relabel_later_steps_draw_new_rows():
    w = synth.PROD
    a = _run(w, step=0)
    b = _run(w, step=99)
    assert (a["src_idx"] != b["src_idx"]).mean() > 0.99


@pytest.mark.parametrize("w", [dataclasses.replace(synth.TINY, strategy="episode", ep_len=(5, 40), capacity=3000),
                               dataclasses.replace(synth.PROD, strategy="episode")],
                         ids=["tiny_episode", "prod_episode"])
def test_relabel_episode_strategy(w):
    ref = _run(w, step=5)
    assert (ref["donor_idx"] >= 0).sum() == oher.her_count(w.batch, w.her_ratio)


@pytest.mark.parametrize("strategy", ["final", "future", "episode", "random"])
def test_relabel_with_given_sources_and_weights(strategy):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    w = dataclasses.replace(synth.TINY, strategy=strategy, ep_len=(5, 40), capacity=3000, batch=777)
    nh = oher.her_count(w.batch, w.her_ratio)
    rep = replay_np(w)
    replay = replay_dev(w, rep)
    rng = np.random.default_rng(77)
    given = rng.integers(0, w.capacity, w.batch).astype(np.int32)
    given[[3, 500]] = [-5, w.capacity + 2]            # outside the buffer: clamped and counted
    isw = rng.random(w.batch).astype(np.float32)
    ctx = ofrl.Context(w.state_dim, w.hidden, w.num_actions, max_batch=w.batch)
    out = ofrl.Batch.empty(w.batch, w.state_stride)
    isw_out = torch.empty(w.batch, device="cuda")
    ofrl.her_relabel_sources(ctx, replay, ofrl.HerConfig(w.batch, nh, w.strategy, w.goal_threshold, w.seed), 6,
                             dev(given), out, is_weights=dev(isw), is_weights_out=isw_out)
    torch.cuda.synchronize()
    clamped = np.clip(given, 0, w.capacity - 1)
    src, donor = oher.sample_indices(w.seed, 6, w.batch, nh, oher.STRATEGY[strategy], w.capacity,
                                     rep["episode_ends"], sources=clamped)
    ref = oher.relabel(rep, src, donor, w.goal_dim, f32(w.goal_threshold))
    s = w.state_dim
    assert_bits(out.src_idx.cpu().numpy(), ref["src_idx"], "src_idx")
    assert_bits(out.donor_idx.cpu().numpy(), ref["donor_idx"], "donor_idx")
    assert_bits(out.states.cpu().numpy()[:, :s], ref["states"][:, :s], "states")
    assert_bits(out.next_states.cpu().numpy()[:, :s], ref["next_states"][:, :s], "next_states")
    assert_bits(out.rewards.cpu().numpy(), ref["rewards"], "rewards")
    assert_bits(isw_out.cpu().numpy(), oher.importance_weights(w.batch, nh, isw), "is_weights")
    assert ctx.poll_status()["bad_index"] == 2
    ctx.close()


@pytest.mark.parametrize("n,chunks", [(1, 1), (1000, 1), (300_000, 3), (4096, 7)])
def test_episode_ends_append(n, chunks):
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    rng = np.random.default_rng(n)
    dones = (rng.random(n) < 0.03).astype(np.float32)
    dones[-1] = 1.0
    ctx = ofrl.Context(8, 64, 4, max_batch=1)
    cap = int(dones.sum()) + 8
    ends = torch.zeros(cap, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = []
    cuts = np.linspace(0, n, chunks + 1).astype(int)
    for a, b in zip(cuts[:-1], cuts[1:]):
        ofrl.episode_ends_append(ctx, dev(dones[a:b]), int(a), ends, count)
        ref = oher.append_episode_ends(ref, dones[a:b], int(a))
    torch.cuda.synchronize()
    k = int(count.item())
    assert k == len(ref)
    assert_bits(ends.cpu().numpy()[:k], np.array(ref, dtype=np.int32), "episode_ends")
    assert ctx.poll_status()["bad_index"] == 0
    ctx.close()


def test_episode_ends_append_overflow_is_counted():
    import offline_rl_step_gb300 as ofrl
    need_gpu()
    dones = np.ones(50, dtype=np.float32)
    ctx = ofrl.Context(8, 64, 4, max_batch=1)
    ends = torch.zeros(20, dtype=torch.int32, device="cuda")
    count = torch.tensor([15], dtype=torch.int32, device="cuda")
    ofrl.episode_ends_append(ctx, dev(dones), 100, ends, count)
    torch.cuda.synchronize()
    assert int(count.item()) == 20
    assert_bits(ends.cpu().numpy()[15:], np.arange(101, 106, dtype=np.int32), "kept ends")
    assert ctx.poll_status()["bad_index"] == 45
    ctx.close()
