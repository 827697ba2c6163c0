"""Division by invariant integers as the kernels do it (FastDiv in
csrc/common.cuh): for 0 <= n < 2^31 and d >= 1, with l = ceil(log2 d) and
m = ceil(2^(31+l) / d), n // d == (n * m) >> (31 + l) (Granlund and
Montgomery, "Division by invariant integers using multiplication", 1994,
the round-up method for N = 31-bit dividends). Checked here exhaustively on
small ranges and at the edges of every power of two, including that m fits
the kernels' 32-bit field."""
import random

import pytest


def make(d):
    l = 0
    while (1 << l) < d:
        l += 1
    m = ((1 << (31 + l)) + d - 1) // d
    return m, 31 + l


def divisors():
    ds = set(range(1, 4097))
    for k in range(1, 31):
        for e in (-2, -1, 0, 1, 2):
            v = (1 << k) + e
            if 1 <= v < (1 << 31):
                ds.add(v)
    rng = random.Random(5)
    ds.update(rng.randrange(1, 1 << 31) for _ in range(2000))
    return sorted(ds)


def dividends(d, rng):
    top = (1 << 31) - 1
    ns = {0, 1, d - 1, d, d + 1, top, top - 1, top - d}
    q = top // d
    for k in (q, q - 1, max(0, q - 7)):
        for e in (-1, 0, 1):
            ns.add(k * d + e)
    ns.update(rng.randrange(0, 1 << 31) for _ in range(40))
    return [n for n in ns if 0 <= n <= top]


def test_fastdiv_exact_everywhere_sampled():
    rng = random.Random(11)
    for d in divisors():
        m, sh = make(d)
        assert 0 < m < (1 << 32), d
        for n in dividends(d, rng):
            assert (n * m) >> sh == n // d, (n, d)


@pytest.mark.parametrize("d", [1, 2, 3, 5, 7, 24, 76, 100, 152, 392])
def test_fastdiv_exhaustive_small_dividends(d):
    m, sh = make(d)
    for n in range(0, 1 << 17):
        assert (n * m) >> sh == n // d
