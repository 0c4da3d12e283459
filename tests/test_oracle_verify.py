"""Pins of the oracle's lossless verification ([GN] §Definição do problema:
rejection sampling keeps the longest prefix consistent with the target, so the
output follows the target distribution; [GN] decoding-cycle paragraph for the
worked round; [GN] "Confidence head" for acceptance = 1 - TV; [JD] and [GN]
"Hardware-Aware Prefix Scheduler" for the non-anticipation requirement)."""
import json
import os

import numpy as np
import pytest

from oracle import draft as D, verify as Vf, schedule as S, philox
from oracle.verify import TargetDist
from oracle_law import law, lossless_violation

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tiny_case(seed, V, gamma, T=1.0, rank=2):
    rng = np.random.default_rng(seed)
    base = rng.normal(0, 1.0, size=(gamma, V)).astype(np.float32)
    target = rng.normal(0, 1.0, size=(gamma + 1, V)).astype(np.float32)
    W1 = rng.normal(0, 0.8, size=(V, rank))
    W2 = rng.normal(0, 0.8, size=(rank, V))
    return base, target, W1, W2


@pytest.mark.parametrize("V,gamma,L,seed", [
    (3, 2, 0, 1), (3, 2, 1, 2), (3, 2, 2, 3), (2, 3, 3, 4), (4, 2, 2, 5), (4, 1, 1, 6),
])
def test_exact_output_law_equals_target(monkeypatch, V, gamma, L, seed):
    """Every emitted position i <= L+1 follows target row i-1 given the history,
    computed exactly over all draft sequences and accept/reject branches."""
    base, target, W1, W2 = _tiny_case(seed, V, gamma)
    lw = law(monkeypatch, base, target, 1, W1, W2, 1.0, lambda toks: L)
    assert abs(sum(lw.values()) - 1.0) < 1e-9
    P = [TargetDist(target[k], 1.0).prob() for k in range(gamma + 1)]
    assert lossless_violation(lw, P, L) < 1e-9


def test_anticipating_scheduler_breaks_losslessness(monkeypatch):
    """A scheduler that looks at the sampled token (verify x_1 only if it is
    token 0) biases the output: the counterexample shape of the pages (tokens
    A/B, the choice depends on the sampled token)."""
    V, gamma = 2, 2
    base = np.array([[1.5, 0.0], [0.0, 0.0]], dtype=np.float32)     # drafter prefers A
    target = np.array([[0.0, 0.0], [0.0, 0.0], [0.0, 0.0]], dtype=np.float32)
    W1 = np.zeros((V, 1)); W2 = np.zeros((1, V))
    P = [TargetDist(target[k], 1.0).prob() for k in range(gamma + 1)]
    causal = law(monkeypatch, base, target, 0, W1, W2, 1.0, lambda toks: 1)
    assert lossless_violation(causal, P, 1) < 1e-9
    peeking = law(monkeypatch, base, target, 0, W1, W2, 1.0,
                  lambda toks: 1 if int(toks[0]) == 0 else 0)
    assert lossless_violation(peeking, P, 0) > 0.05


def test_greedy_exact_law_is_target_argmax(monkeypatch):
    V, gamma = 4, 2
    base, target, W1, W2 = _tiny_case(8, V, gamma)
    target[1] = target[0]  # make the first draft token likely to match
    lw = law(monkeypatch, base, target, 2, W1, W2, 0.0, lambda toks: 2)
    assert len(lw) == 1
    (seq, p), = lw.items()
    assert p == 1.0
    assert seq[0] == int(np.argmax(target[0]))


def test_chi_square_first_two_positions():
    stats = pytest.importorskip("scipy.stats")
    V, gamma, n = 6, 3, 3000
    base, target, W1, W2 = _tiny_case(11, V, gamma)
    first = np.zeros(V)
    second = np.zeros(V)
    for r in range(n):
        d = D.draft_request(base, 0, W1, W2, 1.0, seed=5, r=r)
        v = Vf.verify_request(target, base, 0, W1, W2, d["tokens"], 3, 1.0, seed=5, r=r)
        first[v["out"][0]] += 1
        if v["A"] >= 1:
            second[v["out"][1]] += 1
    P0 = TargetDist(target[0], 1.0).prob()
    P1 = TargetDist(target[1], 1.0).prob()
    assert stats.chisquare(first, P0 * first.sum()).pvalue > 1e-3
    assert stats.chisquare(second, P1 * second.sum()).pvalue > 1e-3


def test_first_position_acceptance_is_one_minus_tv():
    """Acceptance of x_1 converges to sum_v min(P0, Q1) = 1 - TV(P0, Q1)."""
    V, gamma, n = 8, 1, 4000
    base, target, W1, W2 = _tiny_case(12, V, gamma)
    acc = 0
    for r in range(n):
        d = D.draft_request(base, 3, W1, W2, 1.0, seed=9, r=r)
        v = Vf.verify_request(target, base, 3, W1, W2, d["tokens"], 1, 1.0, seed=9, r=r)
        acc += v["A"]
    P0 = TargetDist(target[0], 1.0).prob()
    Q1 = D.DraftDist(base[0], 3, W1, W2, 1.0).prob()
    alpha = np.minimum(P0, Q1).sum()
    assert alpha == pytest.approx(1.0 - 0.5 * np.abs(P0 - Q1).sum(), abs=1e-12)
    sd = np.sqrt(alpha * (1 - alpha) / n)
    assert abs(acc / n - alpha) < 4.5 * sd


def _worked_round_inputs(T):
    g = json.load(open(os.path.join(GOLDEN, "worked_round.json")))
    ids = {c: i for i, c in enumerate(g["alphabet"])}
    V = len(ids)
    gamma = len(g["draft_rows"])
    off = g["off_logit"]
    base = np.full((gamma, V), off, dtype=np.float32)
    for k, c in enumerate(g["draft_rows"]):
        base[k, ids[c]] = 0.0
    target = np.full((gamma + 1, V), off, dtype=np.float32)
    for k, c in enumerate(g["target_rows"]):
        target[k, ids[c]] = 0.0
    return g, ids, base, target


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_worked_round_from_the_pages(T):
    g, ids, base, target = _worked_round_inputs(T)
    V = len(ids)
    conf = np.array([g["confidences"]], dtype=np.float32)
    sps = np.array(g["sps"], dtype=np.float32)
    W1 = np.zeros((V, 1)); W2 = np.zeros((1, V))
    sched = S.schedule(conf, sps, S.CAUSAL)
    assert sched["K"] == g["expected"]["K"] and sched["L"][0] == g["expected"]["L"]
    inv = {i: c for c, i in ids.items()}
    for seed in range(12):
        d = D.draft_request(base, ids[g["anchor"]], W1, W2, T, seed=seed, r=0)
        assert [inv[int(x)] for x in d["tokens"]] == g["expected"]["draft"]
        v = Vf.verify_request(target, base, ids[g["anchor"]], W1, W2, d["tokens"],
                              sched["L"][0], T, seed=seed, r=0)
        assert v["A"] == g["expected"]["A"]
        assert [inv[int(x)] for x in v["out"]] == g["expected"]["emitted"]


def test_forced_rejection_draws_from_residual(monkeypatch):
    """P = (1/2, 1/2, 0), Q = (1/2, 0, 1/2): drafting token 2 (P = 0) is always
    rejected and max(0, P - Q) = (0, 1/2, 0) leaves only token 1."""
    V = 3
    off = -10000.0
    base = np.array([[0.0, off, 0.0]], dtype=np.float32)
    target = np.array([[0.0, 0.0, off], [0.0, 0.0, 0.0]], dtype=np.float32)
    W1 = np.zeros((V, 1)); W2 = np.zeros((1, V))
    script = {philox.DRAFT: 0.9, philox.ACCEPT: 1e-9, philox.RESID: 0.999}
    monkeypatch.setattr(D, "uniform", lambda s_, r, k, p: script[p])
    monkeypatch.setattr(Vf, "uniform", lambda s_, r, k, p: script[p])
    d = D.draft_request(base, 0, W1, W2, 1.0, seed=0, r=0)
    assert int(d["tokens"][0]) == 2
    v = Vf.verify_request(target, base, 0, W1, W2, d["tokens"], 1, 1.0, seed=0, r=0)
    assert v["A"] == 0 and list(v["out"]) == [1]
    assert v["p"][0] == 0.0 and v["q"][0] == pytest.approx(0.5)


def _full_vocab_case(seed, V=129280, rank=256, gamma=2):
    rng = np.random.default_rng(seed)
    base = rng.normal(0, 1.5, size=(gamma, V)).astype(np.float32)
    W1 = rng.normal(0, 0.02, size=(V, rank))
    W2 = rng.normal(0, 0.02, size=(rank, V))
    return base, W1, W2


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_full_vocab_residual_is_the_boosted_token(T):
    """Closed form at the full DeepSeek-scale vocabulary (V = 129280, rank 256):
    if target row 0 equals the drafter's logits at position 1 except for one
    token v* raised by D, then P(v) < Q(v) for every v != v* and P(v*) > Q(v*),
    so normalize(max(0, P - Q)) is the point mass at v*; with D large, the
    drafted token (not v*) is rejected, and the corrected token must be v*
    whatever the uniform. Pins the residual construction and its sampler at
    full size, where no enumeration is possible."""
    V, gamma = 129280, 2
    base, W1, W2 = _full_vocab_case(11, V=V, gamma=gamma)
    anchor = 4242
    l1 = base[0].astype(np.float64) + W1[anchor] @ W2
    for vstar in (int(np.argmin(l1)), 77777):
        target = np.stack([l1, base[1], base[1]]).astype(np.float32)
        target[0, vstar] = np.float32(l1[vstar] + 60.0 * T)
        for seed in (0, 1, 2):
            d = D.draft_request(base, anchor, W1, W2, T, seed, 0)
            assert d["tokens"][0] != vstar
            v = Vf.verify_request(target, base, anchor, W1, W2, d["tokens"], 2, T, seed, 0)
            assert v["A"] == 0
            assert v["new_token"] == vstar


def test_full_vocab_bonus_is_the_dominant_token():
    """Closed form: when every scheduled token is accepted (target rows equal
    the drafter's logits exactly, so p = q and u < 1 accepts), the bonus token
    is drawn from the next target row; a row whose one logit exceeds the rest
    by 80/T puts all but ~e^-80 of its mass there, so the bonus is that token."""
    V, gamma, T = 129280, 2, 1.0
    base, W1, W2 = _full_vocab_case(12, V=V, gamma=gamma)
    anchor = 99
    d = D.draft_request(base, anchor, W1, W2, T, 3, 0)
    rows = []
    prev = anchor
    for k in range(gamma):
        rows.append(base[k].astype(np.float64) + W1[prev] @ W2)
        prev = int(d["tokens"][k])
    bonus_row = base[1].astype(np.float64).copy()
    vstar = 123456
    bonus_row[vstar] = bonus_row.max() + 80.0
    target = np.stack(rows + [bonus_row]).astype(np.float32)
    v = Vf.verify_request(target, base, anchor, W1, W2, d["tokens"], gamma, T, 3, 0)
    # p and q come from the same float32 logits up to the float32 rounding of
    # the drafter's float64 logits, so every ratio is 1 to ~1e-6 and u < 1
    assert v["A"] == gamma
    assert v["new_token"] == vstar


@pytest.mark.parametrize("T", [1.0, 0.8])
def test_full_vocab_residual_moves_mass_of_rejected_token(T):
    """Closed form at V = 129280 that tells the residual apart from P and Q:
    target row 0 = the drafter's logits at position 1, with the drafted token
    x1 pushed down by 60 T (its acceptance ratio is ~e^-60: rejected) and a
    second token v1 raised by b = T ln(1 + e^((l_x1 - l_v1)/T)(1 - e^-60)),
    which moves exactly x1's mass onto v1. Then P = Q off {x1, v1}, so
    max(0, P - Q) is the point mass at v1 and the corrected token is v1 for
    every uniform, while a draw from P or Q would give v1 only with
    probability about Q(x1)."""
    V = 129280
    base, W1, W2 = _full_vocab_case(13, V=V)
    anchor = 31337
    l1 = base[0].astype(np.float64) + W1[anchor] @ W2
    for seed in (0, 1, 2, 3):
        d = D.draft_request(base, anchor, W1, W2, T, seed, 0)
        x1 = int(d["tokens"][0])
        v1 = int(np.argsort(l1)[V // 2])  # a token of middling probability, != x1
        if v1 == x1:
            v1 = int(np.argsort(l1)[V // 2 + 1])
        b = T * np.log1p(np.exp((l1[x1] - l1[v1]) / T) * (1.0 - np.exp(-60.0)))
        row0 = l1.copy()
        row0[x1] -= 60.0 * T
        row0[v1] += b
        target = np.stack([row0, base[1], base[1]]).astype(np.float32)
        v = Vf.verify_request(target, base, anchor, W1, W2, d["tokens"], 2, T, seed, 0)
        assert v["A"] == 0
        assert v["new_token"] == v1
