"""Pins for the oracle's counter-based RNG (SplitMix64 + Lemire map)."""
import os

import numpy as np

from oracle import rng

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_hex(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(int(line, 16))
    return vals


def test_published_splitmix64_vector():
    # published outputs of SplitMix64(seed=0), both through the stateful
    # stream and through the counter jump
    want = _golden_hex("splitmix64_seed0.txt")
    assert rng.splitmix64_stream(0, len(want)) == want
    assert [rng.draw(0, i) for i in range(len(want))] == want


def test_counter_jump_equals_stateful_stream():
    for seed in (1, 1002, 0xDEADBEEFCAFEF00D):
        stream = rng.splitmix64_stream(seed, 200)
        assert [rng.draw(seed, i) for i in range(200)] == stream


def test_counter_layout_is_injective():
    seen = set()
    for step in (0, 1, 7, (1 << 32) - 1):
        for row in (0, 1, 2, 65535, (1 << 31) - 1):
            for s in (0, 1):
                c = rng.counter(step, row, s)
                assert c not in seen
                seen.add(c)
                assert c >> 32 == step


def test_below_bucket_boundaries():
    # below(x<<32, n) = floor(x * n / 2^32): the first x of bucket j is
    # ceil(j * 2^32 / n) and the one before it is still in bucket j - 1.
    r = np.random.default_rng(5)
    for n in (1, 2, 3, 7, 255, 4096, 1 << 20, 1000003, (1 << 32) - 1, 1 << 32):
        for j in set([0, n - 1] + [int(x) for x in r.integers(0, n, 20)]):
            first = -(-(j << 32) // n)
            assert rng.below(first << 32, n) == j
            if first > 0:
                assert rng.below((first - 1) << 32, n) == j - 1
        assert rng.below(((1 << 32) - 1) << 32 | 0xFFFFFFFF, n) == n - 1
        assert rng.below(0, n) == 0


def test_below_is_uniform_on_a_sample():
    n = 10
    counts = np.zeros(n)
    for i in range(20000):
        counts[rng.below(rng.draw(77, i), n)] += 1
    chi2 = ((counts - 2000.0) ** 2 / 2000.0).sum()
    assert chi2 < 40.0   # 9 dof; p < 1e-5 above this
