"""Division by a launch-constant divisor with a multiply-high and a shift (Granlund and
Montgomery, "Division by invariant integers using multiplication", 1994), the method the
cache kernels use for their 32-bit index arithmetic: with s = ceil(log2 d) and
m = floor(2^32 (2^s - d) / d) + 1, x / d = (umulhi(x, m) + x) >> s for 0 <= x < 2^31.

This checks the claim itself, with exact integer arithmetic, over edge and random
divisors and dividends (including where the 32-bit sum umulhi + x is largest); the
kernels' results are compared bit for bit against the oracle in the GPU cache tests."""
import numpy as np


def magic(d):
    s = 0
    while (1 << s) < d:
        s += 1
    m = ((1 << 32) * ((1 << s) - d)) // d + 1
    assert 0 < m < (1 << 32)
    return m, s


def fast_div(x, m, s):
    hi = (x * np.uint64(m)) >> np.uint64(32)
    total = hi + x
    assert int(total.max()) < (1 << 32)  # the kernels add in 32 bits
    return total >> np.uint64(s)


def test_exact_for_31_bit_dividends():
    rng = np.random.default_rng(2024)
    top = (1 << 31) - 1
    divisors = set(range(1, 300))
    for k in range(1, 31):
        divisors |= {(1 << k) - 1, 1 << k, (1 << k) + 1}
    divisors |= {3 * 4096, 4096 - 4, 4100, 8 * 4096, 131072, top, top - 1, 1 << 30}
    divisors |= set(int(v) for v in rng.integers(1, top, 300))
    for d in sorted(divisors):
        if d > top:
            continue
        m, s = magic(d)
        q = rng.integers(0, top // d + 1, 2000, dtype=np.int64)
        xs = np.concatenate([
            np.array([0, 1, d - 1, d, d + 1, top, top - 1, top - (top % d), top - (top % d) - 1]),
            q * d, q * d - 1, q * d + d - 1, rng.integers(0, top + 1, 2000),
        ])
        xs = xs[(xs >= 0) & (xs <= top)].astype(np.uint64)
        np.testing.assert_array_equal(fast_div(xs, m, s), xs // np.uint64(d), err_msg=f"d={d}")


def test_small_divisors_exhaustive_on_a_range():
    xs = np.arange(0, 1 << 20, dtype=np.uint64)
    for d in range(1, 130):
        m, s = magic(d)
        np.testing.assert_array_equal(fast_div(xs, m, s), xs // np.uint64(d), err_msg=f"d={d}")
