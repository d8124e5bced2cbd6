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
@pytest.mark.parametrize("batch", [1, 15, 17, 1000])
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
