"""Pins of the oracle's recurrent (gated) sequential head ([GN] "Head RNN":
a recurrent state of the whole block prefix, updated through gates; the
Markov head is the special case that sees only the previous token)."""
import numpy as np
import pytest

from oracle import draft as D, gated as G
from oracle.verify import TargetDist
from oracle_law import law, lossless_violation

torch = pytest.importorskip("torch")


def _bf16_values(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def test_round_bf16_matches_torch_and_ties_go_to_even():
    rng = np.random.default_rng(0)
    x = (rng.normal(0, 1, 20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    assert np.array_equal(G.round_bf16(x), _bf16_values(x))
    # exact midpoints between two bf16 values: the kept last bit decides
    kept_even = np.array([0x3F800000 | 0x8000, 0x40000000 | 0x8000], dtype=np.uint32).view(np.float32)
    kept_odd = np.array([0x3F810000 | 0x8000, 0xC0010000 | 0x8000], dtype=np.uint32).view(np.float32)
    assert np.array_equal(G.round_bf16(kept_even).view(np.uint32), np.array([0x3F800000, 0x40000000], np.uint32))
    assert np.array_equal(G.round_bf16(kept_odd).view(np.uint32), np.array([0x3F820000, 0xC0020000], np.uint32))
    assert np.array_equal(G.round_bf16(kept_odd), _bf16_values(kept_odd))


def _case(seed, V, gamma, rank, w_sd=0.8):
    rng = np.random.default_rng(seed)
    base = rng.normal(0, 1.0, size=(gamma, V)).astype(np.float32)
    target = rng.normal(0, 1.0, size=(gamma + 1, V)).astype(np.float32)
    W1 = G.round_bf16(rng.normal(0, w_sd, size=(V, rank)).astype(np.float32))
    W2 = G.round_bf16(rng.normal(0, w_sd, size=(rank, V)).astype(np.float32)).astype(np.float64)
    Z = G.round_bf16(rng.uniform(0.25, 1.0, size=(V, rank)).astype(np.float32))
    return base, target, W1, W2, Z


@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_gate_one_is_the_markov_head(T):
    base, _, W1, W2, _ = _case(1, 50, 6, 8)
    ones = np.ones_like(W1)
    for r in range(20):
        g = G.draft_request_gated(base, 3 + r, W1, ones, W2, T, seed=9, r=r)
        m = D.draft_request(base, 3 + r, W1.astype(np.float64), W2, T, seed=9, r=r)
        for key in ("tokens", "q", "m", "Z", "margin", "gap"):
            assert np.array_equal(g[key], m[key]), key
        prevs = [3 + r] + [int(t) for t in m["tokens"][:-1]]
        assert np.array_equal(G.state_rows(3 + r, g["tokens"], W1, ones), W1[prevs])


def test_gate_zero_is_the_parallel_drafter():
    base, _, W1, W2, _ = _case(2, 40, 5, 8)
    zeros = np.zeros_like(W1)
    for r in range(10):
        g = G.draft_request_gated(base, r, W1, zeros, W2, 1.0, seed=3, r=r)
        p = D.draft_request(base, r, W1.astype(np.float64), np.zeros_like(W2), 1.0, seed=3, r=r)
        assert np.array_equal(g["tokens"], p["tokens"])
        assert np.array_equal(g["q"], p["q"])


@pytest.mark.parametrize("c", [0.5, 0.75, 0.3125])
def test_constant_gate_state_is_the_exponential_average(c):
    """s_k = sum_{j<=k} c (1 - c)^(k-j) W1[prev_j] (float64 closed form)."""
    rng = np.random.default_rng(int(c * 1000))
    V, rank, n = 30, 16, 12
    W1 = G.round_bf16(rng.normal(0, 1, size=(V, rank)).astype(np.float32))
    Z = np.full((V, rank), c, dtype=np.float32)
    anchor = 7
    tokens = rng.integers(0, V, size=n)
    prevs = [anchor] + [int(t) for t in tokens[:-1]]
    s = np.zeros(rank, dtype=np.float32)
    rows = G.state_rows(anchor, tokens, W1, Z)
    for k in range(1, n + 1):
        s = G.gated_update(s, Z[prevs[k - 1]], W1[prevs[k - 1]])
        closed = sum(c * (1 - c) ** (k - j) * W1[prevs[j - 1]].astype(np.float64) for j in range(1, k + 1))
        np.testing.assert_allclose(s, closed, rtol=2e-6 * k, atol=1e-6)
        # the operand row is the state rounded to bf16: within one bf16 step of the closed form
        assert np.all(np.abs(rows[k - 1] - closed) <= 2.0 ** -8 * np.abs(closed) + 1e-6)


def test_state_keeps_tokens_before_the_previous_one():
    """Two histories that end in the same previous token give different
    operand rows (the Markov head would give the same row)."""
    _, _, W1, _, Z = _case(3, 20, 4, 8)
    a = G.state_rows(2, [5, 9, 1], W1, Z)
    b = G.state_rows(11, [5, 9, 1], W1, Z)
    assert not np.array_equal(a[1], b[1])   # position 2: prev = 5 in both
    assert not np.array_equal(a[3 - 1], b[3 - 1])  # and still at position 3 (prev = 9)


@pytest.mark.parametrize("V,gamma,L,seed", [(3, 2, 1, 11), (3, 2, 2, 12), (2, 3, 3, 13)])
def test_gated_output_law_equals_target(monkeypatch, V, gamma, L, seed):
    """Lossless verification with the gated head, by exact enumeration: the
    residual at a rejection must use the same state the draft used there."""
    base, target, W1, W2, Z = _case(seed, V, gamma, 2)
    lw = law(monkeypatch, base, target, 1, W1, W2, 1.0, lambda toks: L, gate=Z)
    assert abs(sum(lw.values()) - 1.0) < 1e-9
    P = [TargetDist(target[k], 1.0).prob() for k in range(gamma + 1)]
    assert lossless_violation(lw, P, L) < 1e-9


def test_enumeration_catches_a_shifted_state(monkeypatch):
    """A planted mistake: verification recomputes Q_k from the state of
    position k + 1. The exact law then departs from the target."""
    V, gamma, L = 3, 2, 2
    base, target, W1, W2, Z = _case(12, V, gamma, 2)
    real = G.state_rows

    def shifted(anchor, tokens, W1_, Z_):
        rows = real(anchor, list(tokens) + [0], W1_, Z_)
        return rows[1:]

    monkeypatch.setattr(G, "state_rows", shifted)
    lw = law(monkeypatch, base, target, 1, W1, W2, 1.0, lambda toks: L, gate=Z)
    P = [TargetDist(target[k], 1.0).prob() for k in range(gamma + 1)]
    assert lossless_violation(lw, P, L) > 1e-4
