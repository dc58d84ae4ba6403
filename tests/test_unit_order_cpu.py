"""The band kernel's unit order (CPU only): units are numbered longest first and dealt to
the persistent CTAs in rounds of the grid size, in alternating directions -- CTA c takes
unit i*G + c in even rounds and i*G + (G-1-c) in odd ones.  Every role of a CTA walks the
same sequence, so it must cover each unit exactly once over the grid, and each CTA's
sequence must rise (a CTA stops at its first unit past the end).  Restates the kernel's
arithmetic, like the ring-protocol model."""
import random


def unit_at(i, c, grid):
    return i * grid + ((grid - 1 - c) if (i & 1) else c)


def cta_units(c, grid, n_units):
    out, i = [], 0
    while unit_at(i, c, grid) < n_units:
        out.append(unit_at(i, c, grid))
        i += 1
    return out


def test_every_unit_exactly_once_and_rising():
    rng = random.Random(5)
    cases = [(1, 1), (1, 152), (152, 152), (153, 152), (2048, 152), (1536, 152), (8192, 152)]
    cases += [(rng.randint(1, 5000), None) for _ in range(200)]
    for n_units, grid in cases:
        grid = min(n_units, grid or rng.randint(1, 200))
        seen = []
        for c in range(grid):
            seq = cta_units(c, grid, n_units)
            assert seq == sorted(seq) and len(set(seq)) == len(seq)
            seen += seq
        assert sorted(seen) == list(range(n_units)), (n_units, grid)


def test_alternating_rounds_balance_decreasing_lengths():
    """With unit lengths falling along the order (as for the early query tiles of a causal
    band), alternating rounds keep the per-CTA totals within one unit of each other where
    one-way rounds give the first CTAs every longer unit of each round."""
    grid, n_units = 152, 2048
    lengths = [33] * 1536 + [max(1, 33 - (u - 1536) // 16) for u in range(1536, n_units)]

    def spread(deal):
        tot = [0] * grid
        for c in range(grid):
            for u in deal(c):
                tot[c] += lengths[u]
        return max(tot) - min(tot)

    one_way = spread(lambda c: range(c, n_units, grid))
    alternating = spread(lambda c: cta_units(c, grid, n_units))
    assert alternating <= 33 and alternating < one_way
