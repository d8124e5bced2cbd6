"""Counter-based random numbers for HER index sampling (oracle side).

The pages draw HER source and donor indices with cuRAND ("GPU IQL + HER
Porting Plan", "Donor Index Generation", strategies Future and Random).
cuRAND has no bit-exact CPU twin, so both sides implement one published
generator independently: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-based, and
Lemire's multiply-shift map to a range (Lemire, "Fast random integer
generation in an interval", ACM TOMACS 2019), without the rejection step.

Definition used:
  draw(seed, counter) = the (counter+1)-th output of SplitMix64 seeded with
                        `seed`, i.e. mix(seed + (counter + 1) * GAMMA mod 2^64)
  counter(step, row, stream) = step * 2^32 + 2 * row + stream
                        (stream 0: source index, stream 1: donor index)
  below(r, n)         = ((r >> 32) * n) >> 32, for 1 <= n <= 2^32
"""
M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def _mix(z: int) -> int:
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def splitmix64_stream(seed: int, n: int):
    """The first n outputs of a stateful SplitMix64 generator."""
    state = seed & M64
    out = []
    for _ in range(n):
        state = (state + GAMMA) & M64
        out.append(_mix(state))
    return out


def draw(seed: int, counter: int) -> int:
    """Output number counter+1 of SplitMix64 seeded with `seed` (64-bit int)."""
    return _mix((seed + (counter + 1) * GAMMA) & M64)


def counter(step: int, row: int, stream: int) -> int:
    assert 0 <= row < (1 << 31) and stream in (0, 1) and 0 <= step < (1 << 32)
    return (step << 32) | (row << 1) | stream


def below(r: int, n: int) -> int:
    """Map a 64-bit draw to [0, n) by Lemire's multiply-shift on its top 32 bits."""
    assert 1 <= n <= (1 << 32)
    return ((r >> 32) * n) >> 32
