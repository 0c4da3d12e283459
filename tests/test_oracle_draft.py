"""Pins of the oracle's drafting stage (Markov head + tempered inverse-CDF sampler).

None of these re-types the oracle's formulas: each checks a special case the
pages or the mathematics fix independently.
"""
import numpy as np
import pytest

from oracle import draft, philox
from oracle.draft import DraftDist, draft_request, inverse_cdf


def test_inverse_cdf_hand_cases():
    w = np.array([1.0, 2.0, 3.0, 4.0])  # C = 1, 3, 6, 10
    assert inverse_cdf(w, 0.05)[0] == 0
    assert inverse_cdf(w, 0.1)[0] == 1      # u*Z == C_0 exactly: strict '<' moves on
    assert inverse_cdf(w, 0.2999)[0] == 1
    assert inverse_cdf(w, 0.3)[0] == 2
    assert inverse_cdf(w, 0.95)[0] == 3
    z = np.array([0.0, 1.0, 0.0, 1.0])
    assert inverse_cdf(z, 0.5)[0] == 3      # zero-weight entries are never drawn
    assert inverse_cdf(z, 0.25)[0] == 1
    x, margin, Z = inverse_cdf(w, 0.25)
    assert x == 1 and Z == 10.0 and margin == pytest.approx(0.05)


def test_bf16_decode_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x7F7F], dtype=np.uint16)
    vals = draft.decode(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[3] == 0.0
    assert vals[2] == np.float32(3.140625)
    assert vals[4] == np.float32(3.3895313892515355e38)


def test_zero_w2_reduces_to_parallel_drafter():
    """W2 = 0: no sequential bias, Q_k = softmax(base_k / T) ([GN] parallel stage)."""
    rng = np.random.default_rng(1)
    V, rank, T = 12, 4, 0.7
    base = rng.normal(0, 1.5, size=V).astype(np.float32)
    W1 = rng.normal(0, 1.0, size=(V, rank))
    W2 = np.zeros((rank, V))
    d = DraftDist(base, 5, W1, W2, T)
    e = np.exp(base.astype(np.float64) / T)
    np.testing.assert_allclose(d.prob(), e / e.sum(), rtol=1e-13)


def test_full_rank_identity_is_transition_table():
    """rank = V, W1 = I: the head reduces to a V x V transition table B[prev, :] = W2[prev, :]."""
    rng = np.random.default_rng(2)
    V = 7
    table = rng.normal(0, 2.0, size=(V, V))
    for prev in range(V):
        np.testing.assert_array_equal(draft.markov_bias(np.eye(V), table, prev), table[prev])
    base = np.zeros(V, dtype=np.float32)
    d = DraftDist(base, 3, np.eye(V), table, 1.0)
    e = np.exp(table[3])
    np.testing.assert_allclose(d.prob(), e / e.sum(), rtol=1e-13)


def test_low_rank_bias_is_outer_structure():
    """B = W1 W2 is rank <= r: bias vectors of all prev tokens span <= r dims."""
    rng = np.random.default_rng(3)
    V, rank = 20, 3
    W1 = rng.normal(size=(V, rank))
    W2 = rng.normal(size=(rank, V))
    Bm = np.stack([draft.markov_bias(W1, W2, p) for p in range(V)])
    s = np.linalg.svd(Bm, compute_uv=False)
    assert s[rank] < 1e-10 * s[0]
    # with one-hot rows in W1 the bias picks rows of W2
    W1h = np.zeros((V, rank)); W1h[4, 1] = 1.0
    np.testing.assert_array_equal(draft.markov_bias(W1h, W2, 4), W2[1])


def test_chain_conditions_on_previous_sampled_token():
    """A transition table forcing next = (prev + 3) mod V: the draft follows it
    from the anchor, i.e. position 1 uses the anchor and position k uses x_{k-1}
    ([GN] 'Etapa sequencial'; the anchor is the first prediction position)."""
    V, gamma = 11, 6
    table = np.full((V, V), -60.0)
    for p in range(V):
        table[p, (p + 3) % V] = 60.0
    base = np.zeros((gamma, V), dtype=np.float32)
    for T in (1.0, 0.0):
        out = draft_request(base, 4, np.eye(V), table, T, seed=0, r=0)
        expect = [(4 + 3 * k) % V for k in range(1, gamma + 1)]
        assert list(out["tokens"]) == expect
        np.testing.assert_allclose(out["q"], 1.0, atol=1e-40 if T else 0)


def test_greedy_ties_take_lowest_index():
    V = 9
    base = np.array([0, 2, 5, 1, 5, 5, 0, -1, 4], dtype=np.float32)
    d = DraftDist(base, 0, np.zeros((V, 2)), np.zeros((2, V)), 0.0)
    assert int(np.argmax(d.w)) == 2 and d.gap == 0.0


def test_small_temperature_converges_to_argmax():
    rng = np.random.default_rng(4)
    V = 16
    base = rng.normal(0, 1.0, size=V).astype(np.float32)
    W1 = rng.normal(0, 0.3, size=(V, 4)); W2 = rng.normal(0, 0.3, size=(4, V))
    l = base.astype(np.float64) + draft.markov_bias(W1, W2, 2)
    d = DraftDist(base, 2, W1, W2, 1e-4)
    assert int(np.argmax(d.prob())) == int(np.argmax(l))
    assert d.prob().max() > 1 - 1e-12
    d0 = DraftDist(base, 2, W1, W2, 0.0)
    assert int(np.argmax(d0.w)) == int(np.argmax(l))


def test_sampler_matches_softmax_chi_square():
    """Inverse-CDF draws with Philox uniforms follow softmax(l / T) (V = 16)."""
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(5)
    V, T, n = 16, 0.8, 6000
    base = rng.normal(0, 1.2, size=(1, V)).astype(np.float32)
    W1 = rng.normal(0, 0.5, size=(V, 3)); W2 = rng.normal(0, 0.5, size=(3, V))
    counts = np.zeros(V)
    for r in range(n):
        counts[draft_request(base, 6, W1, W2, T, seed=11, r=r)["tokens"][0]] += 1
    l = base[0].astype(np.float64) + W1[6] @ W2
    p = np.exp((l - l.max()) / T); p /= p.sum()
    _, pval = stats.chisquare(counts, p * n)
    assert pval > 1e-3


def test_draft_q_and_stats_consistent_with_distribution():
    rng = np.random.default_rng(6)
    V, gamma, T = 10, 3, 1.3
    base = rng.normal(0, 1, size=(gamma, V)).astype(np.float32)
    W1 = rng.normal(0, .4, size=(V, 2)); W2 = rng.normal(0, .4, size=(2, V))
    out = draft_request(base, 1, W1, W2, T, seed=2, r=9)
    prev = 1
    for k in range(gamma):
        l = base[k].astype(np.float64) + W1[prev] @ W2
        x = out["tokens"][k]
        # log-partition T*ln(sum exp(l/T)) from the recorded (m, Z)
        lse = out["m"][k] + T * np.log(out["Z"][k])
        assert lse == pytest.approx(T * np.log(np.sum(np.exp(l / T))), rel=1e-12)
        assert out["q"][k] == pytest.approx(np.exp((l[x] - lse) / T), rel=1e-12)
        u = philox.uniform(2, 9, k + 1, philox.DRAFT)
        cdf = np.cumsum(np.exp(l / T)) / np.sum(np.exp(l / T))
        assert (x == 0 or cdf[x - 1] <= u) and u < cdf[x]
        prev = x
