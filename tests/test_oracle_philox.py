"""Pins of the oracle's Philox4x64-10 and uniform mapping.

The generator is checked against numpy.random.Philox, an independent
implementation of the same published generator (Salmon et al., SC'11). numpy
increments its 256-bit counter before producing each block, so a numpy stream
started at counter c - 1 yields the block for counter c.
"""
import numpy as np
import pytest

from oracle import philox


def _numpy_block(counter, key):
    c = list(counter)
    # numpy increments before generating: start one below (with borrow).
    for i in range(4):
        if c[i] > 0:
            c[i] -= 1
            break
        c[i] = (1 << 64) - 1
    g = np.random.Philox(counter=np.array(c, dtype=np.uint64),
                         key=np.array(key, dtype=np.uint64))
    return tuple(int(x) for x in g.random_raw(4))


@pytest.mark.parametrize("counter,key", [
    ((0, 0, 0, 0), (0, 0)),
    ((1, 0, 0, 0), (0, philox.KEY_HI)),
    ((5, 7, 2, 0), (123, philox.KEY_HI)),
    ((127, 16, 3, 0), (2**64 - 1, philox.KEY_HI)),
    ((2**64 - 1, 2**63, 1, 0), (0xDEADBEEF, 0x1234)),
])
def test_philox_matches_numpy(counter, key):
    assert philox.philox4x64_10(counter, key) == _numpy_block(counter, key)


def test_philox_random_counters_match_numpy():
    rng = np.random.default_rng(7)
    for _ in range(50):
        counter = tuple(int(x) for x in rng.integers(0, 2**63, size=4))
        key = tuple(int(x) for x in rng.integers(0, 2**63, size=2))
        assert philox.philox4x64_10(counter, key) == _numpy_block(counter, key)


def test_uniform_is_exact_odd_multiple_of_2_pow_minus_53():
    for r in range(20):
        for k in range(1, 5):
            for purpose in range(4):
                u = philox.uniform(3, r, k, purpose)
                assert 0.0 < u < 1.0
                n = u * 2.0 ** 53
                assert n == int(n) and int(n) % 2 == 1


def test_uniform_distribution_and_independence_of_purposes():
    us = np.array([philox.uniform(0, r, k, p) for r in range(400) for k in range(1, 6)
                   for p in range(4)])
    # Kolmogorov-Smirnov distance against U(0, 1) for 8000 draws.
    s = np.sort(us)
    n = s.size
    d = max(np.max(np.arange(1, n + 1) / n - s), np.max(s - np.arange(n) / n))
    assert d < 1.63 / np.sqrt(n)  # 1% critical value
    # purposes of the same (r, k) are different streams
    a = np.array([philox.uniform(0, r, 1, 0) for r in range(200)])
    b = np.array([philox.uniform(0, r, 1, 1) for r in range(200)])
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.25
