"""Pins of the oracle's hardware-aware prefix scheduler.

Brute force enumerates every prefix-closed choice of verification lengths
(L_1..L_R) directly from the confidences, independent of the oracle's sort and
scan; invariants and limiting tables come from the pages' statements
([GN] "Hardware-Aware Prefix Scheduler": monotone survival gives prefix
closure, greedy early stop is globally optimal only when Theta is unimodal).
"""
import itertools
import math

import numpy as np
import pytest

from oracle import schedule as S


def _a(conf):
    return S.survival(conf)


def _theta_of_lengths(a, L, sps):
    """Theta of an explicit length vector, computed from first principles."""
    R = a.shape[0]
    B = R + int(sum(L))
    if B > len(sps):
        return None
    s = 0
    for r in range(R):
        for j in range(L[r]):
            s += math.floor(float(a[r, j]) * 2.0 ** 40 + 0.5)
    return (R + s * 2.0 ** -40) * float(sps[B - 1])


def test_survival_is_sequential_fp32_product():
    c = np.array([[0.9, 0.8, 0.7], [1.0, 0.5, 0.25]], dtype=np.float32)
    a = _a(c)
    assert a.dtype == np.float32
    assert a[0, 0] == np.float32(0.9)
    assert a[0, 1] == np.float32(np.float32(0.9) * np.float32(0.8))
    assert a[0, 2] == np.float32(a[0, 1] * np.float32(0.7))
    assert list(a[1]) == [1.0, 0.5, 0.125]


def test_survival_clamps_and_rejects_nan():
    a = _a(np.array([[1.5, -0.2, 0.5]], dtype=np.float32))
    assert list(a[0]) == [1.0, 0.0, 0.0]
    with pytest.raises(S.NonFiniteInput):
        _a(np.array([[0.5, np.nan]], dtype=np.float32))


@pytest.mark.parametrize("seed", range(6))
def test_prefix_closure_and_monotone_survival(seed):
    rng = np.random.default_rng(seed)
    R, g = 7, 5
    conf = rng.uniform(0.3, 1.0, size=(R, g)).astype(np.float32)
    conf[0, 2] = 1.0  # repeated product values exercise the tie rule
    n = 60
    sps = (1.0 / (1.0 + 0.03 * np.arange(1, n + 1))).astype(np.float32)
    out = S.schedule(conf, sps, S.CAUSAL)
    a = out["a"]
    assert np.all(np.diff(a, axis=1) <= 0)
    order = S.descending_order(a)
    admitted = set(order[:out["K"]])
    for r in range(R):
        got = {i % g for i in admitted if i // g == r}
        assert got == set(range(out["L"][r]))  # each request keeps a prefix
    assert out["K"] == int(out["L"].sum())


def _unimodal(seq):
    peak = int(np.argmax(seq))
    return all(seq[i] <= seq[i + 1] for i in range(peak)) and \
        all(seq[i] >= seq[i + 1] for i in range(peak, len(seq) - 1))


@pytest.mark.parametrize("seed", range(12))
def test_greedy_equals_brute_force_when_theta_unimodal(seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(1, 4))
    g = int(rng.integers(1, 5))
    conf = rng.uniform(0.2, 1.0, size=(R, g)).astype(np.float32)
    n = R * (g + 1)
    t1 = rng.uniform(0.01, 0.3)
    sps = (1.0 / (1.0 + t1 * np.arange(1, n + 1) ** 1.5)).astype(np.float32)
    a = _a(conf)
    best_by_count = {}
    for L in itertools.product(range(g + 1), repeat=R):
        th = _theta_of_lengths(a, L, sps)
        if th is not None:
            k = sum(L)
            best_by_count[k] = max(best_by_count.get(k, -1.0), th)
    seq = [best_by_count[k] for k in sorted(best_by_count)]
    out = S.schedule(conf, sps, S.CAUSAL)
    if _unimodal(seq):
        assert out["theta"] == max(seq)
        assert out["theta"] == _theta_of_lengths(a, out["L"], sps)
    else:
        assert out["theta"] <= max(seq)  # greedy may stop early on a non-unimodal Theta


def test_constant_table_admits_up_to_table_bound():
    rng = np.random.default_rng(9)
    R, g = 5, 6
    conf = rng.uniform(0.1, 1.0, size=(R, g)).astype(np.float32)
    for n_table in (R, R + 7, R + R * g, 200):
        sps = np.ones(n_table, dtype=np.float32)
        out = S.schedule(conf, sps, S.CAUSAL)
        assert out["K"] == min(R * g, n_table - R)


def test_table_falling_faster_than_R_over_R_plus_1_admits_nothing():
    R, g = 4, 3
    conf = np.ones((R, g), dtype=np.float32)
    ratio = 0.99 * R / (R + 1)
    sps = (ratio ** np.arange(30)).astype(np.float32)
    out = S.schedule(conf, sps, S.CAUSAL)
    assert out["K"] == 0 and list(out["L"]) == [0] * R
    assert out["theta"] == float(R) * float(sps[R - 1])


def test_R_beyond_table_admits_nothing():
    conf = np.full((6, 2), 0.9, dtype=np.float32)
    out = S.schedule(conf, np.ones(5, dtype=np.float32), S.CAUSAL)
    assert out["K"] == 0 and out["theta"] == 0.0


def test_ties_are_admitted_strict_decrease_stops():
    # one request, a = 1, 1, 0.5: Theta_0 = 1*s1, Theta_1 = 2*s2, ...
    conf = np.array([[1.0, 1.0, 0.5]], dtype=np.float32)
    sps = np.array([1.0, 0.5, 1.0 / 3.0, 0.1], dtype=np.float32)
    out = S.schedule(conf, sps, S.CAUSAL)
    # Theta_1 = 2 * 0.5 = 1.0 == Theta_0 -> admitted (tie); Theta_2 = 3 * fl32(1/3) ~ 1
    th2 = 3.0 * float(np.float32(1.0 / 3.0))
    expect_K = 2 if th2 >= 1.0 else 1
    assert out["K"] == expect_K


@pytest.mark.parametrize("seed", range(5))
def test_lagged_equals_causal_when_lag_is_current_and_unimodal(seed):
    rng = np.random.default_rng(200 + seed)
    R, g = 6, 5
    conf = rng.uniform(0.3, 1.0, size=(R, g)).astype(np.float32)
    n = R * (g + 1)
    sps = (1.0 / (1.0 + 0.02 * np.arange(1, n + 1) + 0.004 * np.arange(1, n + 1) ** 2)
           ).astype(np.float32)
    c = S.schedule(conf, sps, S.CAUSAL)
    lg = S.schedule(conf, sps, S.LAGGED, conf_lagged=conf)
    # Theta along the descending order of a, from first principles:
    a = _a(conf)
    assert lg["K"] >= c["K"]
    a_sorted = sorted(a.reshape(-1), reverse=True)
    seq = []
    s = 0
    for i in range(min(R * g, n - R) + 1):
        if i:
            s += math.floor(float(a_sorted[i - 1]) * 2.0 ** 40 + 0.5)
        seq.append((R + s * 2.0 ** -40) * float(sps[R + i - 1]))
    if _unimodal(seq):
        assert lg["K"] == c["K"] and list(lg["L"]) == list(c["L"])


def test_lagged_uses_lagged_for_K_and_current_for_ranking():
    R, g = 2, 3
    cur = np.array([[0.1, 0.1, 0.1], [0.99, 0.99, 0.99]], dtype=np.float32)
    lag = np.array([[0.99, 0.99, 0.99], [0.1, 0.1, 0.1]], dtype=np.float32)
    sps = np.ones(R * (g + 1), dtype=np.float32)
    out = S.schedule(cur, sps, S.LAGGED, conf_lagged=lag)
    assert out["K"] == R * g
    sps2 = np.array([1, 1, 1, 1, 0.6, 0.5, 0.4, 0.3], dtype=np.float32)
    out2 = S.schedule(cur, sps2, S.LAGGED, conf_lagged=lag)
    # lagged a sorted: .99, .9801, .9703, .1, ...; B_i = 2 + i uses entry 1 + i:
    # Theta_0 = 2, Theta_1 = 2.99, Theta_2 = 3.9701, Theta_3 = 4.9404 * 0.6 -> K = 2
    assert out2["K"] == 2
    assert list(out2["L"]) == [0, 2]  # the top 2 by CURRENT confidence are request 1's


def test_all_mode_verifies_every_position():
    conf = np.full((3, 4), 0.5, dtype=np.float32)
    out = S.schedule(conf, np.ones(20, dtype=np.float32), S.ALL)
    assert list(out["L"]) == [4, 4, 4] and out["K"] == 12
