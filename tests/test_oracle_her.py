"""Pins for the oracle's HER index sampling and relabel."""
import os

import numpy as np
import pytest

import synth
from oracle import her

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def _constants():
    return {k: float(v) for k, v in _rows("constants.txt")}


def test_her_split_matches_pages():
    for b, ratio, rows in _rows("her_split.txt"):
        assert her.her_count(int(b), float(ratio)) == int(rows)


def test_staging_size_matches_pages():
    for s, rows, nbytes in _rows("her_staging.txt"):
        w = synth.scaled(synth.TINY, batch=256)
        assert her.her_count(w.batch, w.her_ratio) == int(rows)
        assert 2 * int(rows) * int(s) * 4 == int(nbytes)


def _small(strategy, cap=2048, ep=(16, 16), batch=512, ratio=0.5, g=4):
    import dataclasses
    w = dataclasses.replace(synth.TINY, capacity=cap, ep_len=ep, batch=batch,
                            her_ratio=ratio, strategy=strategy, goal_dim=g)
    return w, synth.make_replay(w)


def _last_of_episode(episode_id, i):
    # linear scan on episode ids: an independent way to find the episode end
    j = i
    while j + 1 < len(episode_id) and episode_id[j + 1] == episode_id[i]:
        j += 1
    return j


@pytest.mark.parametrize("strategy", ["final", "future", "random"])
def test_indices_valid(strategy):
    w, rep = _small(strategy, ep=(5, 40))
    n_her = her.her_count(w.batch, w.her_ratio)
    src, donor = her.sample_indices(w.seed, 3, w.batch, n_her, her.STRATEGY[strategy],
                                    w.capacity, rep["episode_ends"])
    assert src.min() >= 0 and src.max() < w.capacity
    assert (donor[: w.batch - n_her] == -1).all()
    eid = rep["episode_id"]
    for b in range(w.batch - n_her, w.batch):
        s, d = int(src[b]), int(donor[b])
        last = _last_of_episode(eid, s)
        if strategy == "final":
            assert d == last
        elif strategy == "future":
            if s == last:
                assert d == s
            else:
                assert s + 1 <= d <= last
                assert eid[d] == eid[s]
        else:
            assert 0 <= d < w.capacity


def test_future_covers_its_range():
    # one 8-step episode per 8 rows: from source 0 the donor is uniform on 1..7
    w, rep = _small("future", cap=64, ep=(8, 8), batch=4096, ratio=1.0)
    src, donor = her.sample_indices(w.seed, 0, w.batch, w.batch, her.FUTURE, w.capacity,
                                    rep["episode_ends"])
    off = (donor - (src // 8) * 8)[src % 8 == 0]
    assert set(off.tolist()) == set(range(1, 8))


def test_steps_draw_fresh_indices():
    w, rep = _small("random")
    a = her.sample_indices(w.seed, 0, w.batch, 256, her.RANDOM, w.capacity, rep["episode_ends"])
    b = her.sample_indices(w.seed, 1, w.batch, 256, her.RANDOM, w.capacity, rep["episode_ends"])
    assert (a[0] != b[0]).mean() > 0.9


@pytest.mark.parametrize("strategy", ["final", "future", "random"])
def test_relabel_properties(strategy):
    c = _constants()
    w, rep = _small(strategy)
    n_her = her.her_count(w.batch, w.her_ratio)
    src, donor = her.sample_indices(w.seed, 0, w.batch, n_her, her.STRATEGY[strategy],
                                    w.capacity, rep["episode_ends"])
    out = her.relabel(rep, src, donor, w.goal_dim, c["goal_threshold"])
    g = w.goal_dim
    normal = donor < 0
    # normal rows are the stored transition, bit for bit
    for k in ("states", "next_states", "actions", "rewards", "dones"):
        assert np.array_equal(out[k][normal].view(np.uint8), rep[k][src[normal]].view(np.uint8))
    hr = ~normal
    # non-goal features, action and done are the source's, bit for bit
    for k in ("states", "next_states"):
        assert np.array_equal(out[k][hr][:, g:].view(np.uint32), rep[k][src[hr]][:, g:].view(np.uint32))
        # the goal slice is the donor's achieved goal (its next_state's slice)
        assert np.array_equal(out[k][hr][:, :g].view(np.uint32),
                              rep["next_states"][donor[hr]][:, :g].view(np.uint32))
    assert np.array_equal(out["actions"][hr], rep["actions"][src[hr]])
    assert np.array_equal(out["dones"][hr].view(np.uint32), rep["dones"][src[hr]].view(np.uint32))
    # rewards are exactly +1 or -0.01 (fp32), and agree with the distance rule
    r = out["rewards"][hr]
    assert set(np.unique(r).tolist()) <= {np.float32(c["reward_hit"]), np.float32(c["reward_miss"])}
    dist = np.linalg.norm(rep["next_states"][src[hr], :g].astype(np.float64)
                          - rep["next_states"][donor[hr], :g].astype(np.float64), axis=1)
    clear = np.abs(dist - c["goal_threshold"]) > 1e-6
    want = np.where(dist < c["goal_threshold"], np.float32(1.0), np.float32(-0.01))
    assert np.array_equal(r[clear], want[clear])


def test_final_from_episode_end_is_a_hit():
    # a source that is its episode's last transition is its own Final donor:
    # distance 0, reward +1
    w, rep = _small("final")
    ends = rep["episode_ends"]
    src = (ends[:10] - 1).astype(np.int32)
    donor = np.array([her.episode_end(list(ends), int(s)) - 1 for s in src], dtype=np.int32)
    assert np.array_equal(src, donor)
    out = her.relabel(rep, src, donor, w.goal_dim, 0.01)
    assert (out["rewards"] == np.float32(1.0)).all()


def test_reward_threshold_cases():
    ns = np.zeros((6, 8), dtype=np.float32)
    ns[1, 0] = 0.009          # distance 0.009 -> hit
    ns[2, 0] = 0.011          # distance 0.011 -> miss
    ns[3, :4] = 0.004         # distance 0.008 -> hit
    ns[4, :4] = 0.006         # distance 0.012 -> miss
    ns[5, 0] = np.nan         # NaN distance compares false -> miss
    r = her.goal_reward(ns, np.arange(6), np.zeros(6, dtype=np.int64), 4, 0.01)
    assert r.tolist() == [np.float32(1.0), np.float32(1.0), np.float32(-0.01),
                          np.float32(1.0), np.float32(-0.01), np.float32(-0.01)]


def test_anchor_workload_fires_both_branches():
    # the HER-heavy recipe places about 20% of random pairs within 0.005
    import dataclasses
    w = dataclasses.replace(synth.HER_HEAVY, capacity=1 << 15, batch=4096)
    rep = synth.make_replay(w)
    n_her = her.her_count(w.batch, w.her_ratio)
    src, donor = her.sample_indices(w.seed, 0, w.batch, n_her, her.RANDOM, w.capacity,
                                    rep["episode_ends"])
    out = her.relabel(rep, src, donor, w.goal_dim, w.goal_threshold)
    frac = (out["rewards"][donor >= 0] == np.float32(1.0)).mean()
    assert 0.15 < frac < 0.25


# ---- Episode strategy, caller-given sources, boundary maintenance ----------

def _first_of_episode(episode_id, i):
    # linear scan on episode ids: an independent way to find the episode start
    j = i
    while j > 0 and episode_id[j - 1] == episode_id[i]:
        j -= 1
    return j


def test_episode_donors_stay_in_the_source_episode():
    w, rep = _small("episode", ep=(5, 40))
    n_her = her.her_count(w.batch, w.her_ratio)
    src, donor = her.sample_indices(w.seed, 4, w.batch, n_her, her.EPISODE, w.capacity, rep["episode_ends"])
    eid = rep["episode_id"]
    before = after = 0
    for b in range(w.batch - n_her, w.batch):
        s, d = int(src[b]), int(donor[b])
        assert _first_of_episode(eid, s) <= d <= _last_of_episode(eid, s)
        assert eid[d] == eid[s]
        before += d < s
        after += d > s
    # the whole episode is reachable: donors before and after the source
    assert before > 0 and after > 0


def test_episode_covers_the_whole_episode():
    # 8-step episodes: from source 3 the donor is uniform on 0..7 of its episode
    w, rep = _small("episode", cap=64, ep=(8, 8), batch=4096, ratio=1.0)
    src, donor = her.sample_indices(w.seed, 0, w.batch, w.batch, her.EPISODE, w.capacity, rep["episode_ends"])
    off = (donor - (src // 8) * 8)[src % 8 == 3]
    assert set(off.tolist()) == set(range(8))


def test_given_sources_are_used_and_donors_follow_them():
    w, rep = _small("future", ep=(5, 40))
    rng = np.random.default_rng(9)
    given = rng.integers(0, w.capacity, w.batch).astype(np.int32)
    n_her = her.her_count(w.batch, w.her_ratio)
    src, donor = her.sample_indices(w.seed, 2, w.batch, n_her, her.FUTURE, w.capacity, rep["episode_ends"],
                                    sources=given)
    assert np.array_equal(src, given)
    eid = rep["episode_id"]
    for b in range(w.batch - n_her, w.batch):
        s, d = int(src[b]), int(donor[b])
        last = _last_of_episode(eid, s)
        assert d == s if s == last else s + 1 <= d <= last


def test_importance_weights_of_her_rows_are_one():
    isw = np.linspace(0.1, 0.9, 10).astype(np.float32)
    w = her.importance_weights(10, 3, isw)
    assert np.array_equal(w[:7], isw[:7]) and (w[7:] == 1.0).all()
    assert (her.importance_weights(5, 2) == 1.0).all()


def test_boundary_append_rebuilds_the_buffer_ends():
    # the generator builds episode_ends from episode lengths; appending its
    # done flags (whole, or in two chunks) gives the same array
    import dataclasses
    w = dataclasses.replace(synth.TINY, capacity=3000, ep_len=(5, 40))
    rep = synth.make_replay(w)
    ends = [int(e) for e in rep["episode_ends"]]
    assert her.append_episode_ends([], rep["dones"], 0) == ends
    cut = 1234
    part = her.append_episode_ends([], rep["dones"][:cut], 0)
    assert her.append_episode_ends(part, rep["dones"][cut:], cut) == ends
