"""HER index sampling and relabelling (oracle side).

Follows "GPU IQL + HER Porting Plan":
  * "HER (CPU)": the goal is the first goal_dim elements of the state; the
    goal slice of state and next_state is replaced by an achieved goal taken
    from another transition; the reward becomes +1.0 if the goal distance is
    below 0.01 and -0.01 otherwise; a her_ratio fraction of the batch is HER.
  * "How HER Interacts with GPU PER": her_size = batch * her_ratio truncated
    to an integer, normal rows first and HER rows after them (concat order).
    PER sampling belongs to another system; sources here are uniform over the
    buffer.
  * "Donor Index Generation": Final = episode_end - 1 with the episode end
    found by binary search over the episode boundary array; Future = uniform
    in [source_idx + 1, episode_end); Random = uniform over the buffer.
  * "CUDA Kernel: her_relabel_kernel.cu": copy state/next_state/action/done
    of the source; the goal slice comes from next_states[donor]; the reward
    compares next_states[source, :g] with next_states[donor, :g] in fp32
    (float accumulator, sqrtf, strict '<' against the threshold).

  * "HER (CPU)" item 5 names a fourth strategy, Episode, without defining
    it; "How HER Interacts with GPU PER": the HER rows' sources may come from
    the PER sampler and their importance weights are 1 (no PER bias);
    "Episode Boundary Tracking on GPU": each finished episode's end is
    appended to the boundary array.

Readings where the pages are open (each listed in the design notes):
  * episode_end is exclusive, so Final's donor is the last transition.
  * Future with an empty range (source is the episode's last transition)
    takes the source itself as donor.
  * Normal rows keep their stored reward and get donor index -1.
  * Episode: the donor is uniform over the source's whole episode
    [episode_start, episode_end), as the HER paper's "episode" strategy
    (Andrychowicz et al. 2017); episode_start is the previous episode's end.
"""
import bisect

import numpy as np

from . import rng

FINAL, FUTURE, RANDOM, EPISODE = 0, 1, 2, 3
STRATEGY = {"final": FINAL, "future": FUTURE, "random": RANDOM, "episode": EPISODE}


def her_count(batch: int, her_ratio: float) -> int:
    """her_size = (batch * her_ratio) truncated, as the pages' `as usize` cast does."""
    return int(batch * her_ratio)


def episode_end(episode_ends, src: int) -> int:
    """Exclusive end of the episode holding transition `src` (binary search)."""
    k = bisect.bisect_right(episode_ends, src)
    return int(episode_ends[k])


def episode_start(episode_ends, src: int) -> int:
    """First transition of the episode holding `src`: the previous episode's end, or 0."""
    k = bisect.bisect_right(episode_ends, src)
    return int(episode_ends[k - 1]) if k > 0 else 0


def sample_indices(seed: int, step: int, batch: int, her_rows: int, strategy: int,
                   capacity: int, episode_ends=None, sources=None):
    """Source and donor indices for one batch.

    Rows [0, batch - her_rows) are normal rows (donor -1); rows
    [batch - her_rows, batch) are HER rows with a donor by `strategy`.
    `sources`: the caller's source of every row (e.g. PER-sampled) in place
    of the drawn ones.
    """
    ends = None if episode_ends is None else [int(e) for e in episode_ends]
    src = np.empty(batch, dtype=np.int32)
    donor = np.full(batch, -1, dtype=np.int32)
    first_her = batch - her_rows
    for b in range(batch):
        s = int(sources[b]) if sources is not None else rng.below(rng.draw(seed, rng.counter(step, b, 0)), capacity)
        src[b] = s
        if b < first_her:
            continue
        if strategy == FINAL:
            donor[b] = episode_end(ends, s) - 1
        elif strategy == FUTURE:
            end = episode_end(ends, s)
            lo = s + 1
            if lo < end:
                donor[b] = lo + rng.below(rng.draw(seed, rng.counter(step, b, 1)), end - lo)
            else:
                donor[b] = s
        elif strategy == RANDOM:
            donor[b] = rng.below(rng.draw(seed, rng.counter(step, b, 1)), capacity)
        elif strategy == EPISODE:
            lo, end = episode_start(ends, s), episode_end(ends, s)
            donor[b] = lo + rng.below(rng.draw(seed, rng.counter(step, b, 1)), end - lo)
        else:
            raise ValueError(strategy)
    return src, donor


def goal_reward(next_states, src: np.ndarray, donor: np.ndarray, goal_dim: int,
                threshold: float) -> np.ndarray:
    """+1.0 if ||s'[src,:g] - s'[donor,:g]||_2 < threshold else -0.01, in fp32.

    fp32 as in the pages' kernel: diff in fp32, a float accumulator summed in
    order d = 0..g-1 (each product and sum rounded, no fused multiply-add),
    sqrtf, then a strict comparison with the fp32 threshold.
    """
    a = next_states[src, :goal_dim].astype(np.float32)
    b = next_states[donor, :goal_dim].astype(np.float32)
    dsq = np.zeros(len(src), dtype=np.float32)
    for d in range(goal_dim):
        diff = a[:, d] - b[:, d]
        dsq = dsq + diff * diff
    dist = np.sqrt(dsq)
    return np.where(dist < np.float32(threshold), np.float32(1.0), np.float32(-0.01)).astype(np.float32)


def relabel(replay: dict, src: np.ndarray, donor: np.ndarray, goal_dim: int,
            threshold: float) -> dict:
    """Gather rows `src` and relabel the rows whose donor is >= 0."""
    st = replay["states"][src].copy()
    ns = replay["next_states"][src].copy()
    act = replay["actions"][src].copy()
    rew = replay["rewards"][src].copy()
    done = replay["dones"][src].copy()
    her = donor >= 0
    if her.any():
        d = donor[her]
        goal = replay["next_states"][d, :goal_dim]
        st[her, :goal_dim] = goal
        ns[her, :goal_dim] = goal
        rew[her] = goal_reward(replay["next_states"], src[her], d, goal_dim, threshold)
    return dict(states=st, next_states=ns, actions=act, rewards=rew, dones=done,
                src_idx=src.astype(np.int32), donor_idx=donor.astype(np.int32))


def importance_weights(batch: int, her_rows: int, is_weights=None):
    """Normal rows keep their (PER) importance weight; HER rows get 1 ("How
    HER Interacts with GPU PER": uniform weight for HER samples, no PER bias)."""
    w = np.ones(batch, dtype=np.float32) if is_weights is None else np.asarray(is_weights, np.float32).copy()
    w[batch - her_rows:] = 1.0
    return w


def append_episode_ends(episode_ends, dones, first_index: int):
    """The boundary array after n new transitions stored at first_index..:
    each done transition i closes an episode ending (exclusively) at
    first_index + i + 1, appended in order."""
    new = [first_index + i + 1 for i, d in enumerate(np.asarray(dones)) if d != 0]
    return list(episode_ends) + new
