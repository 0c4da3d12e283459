"""Pins of the oracle's acceptance labels ([GN] "Confidence head": the label of
draft position k is the probability that it passes verification, which under
the speculative-sampling rule is 1 - TV(P_{k-1}, Q_k))."""
import numpy as np
import pytest

from oracle import draft as D, verify as Vf, labels as Lb
from oracle.verify import TargetDist


def _case(seed, V, gamma, rank=3, sd=1.0):
    rng = np.random.default_rng(seed)
    base = rng.normal(0, sd, size=(gamma, V)).astype(np.float32)
    target = rng.normal(0, sd, size=(gamma + 1, V)).astype(np.float32)
    W1 = rng.normal(0, 0.7, size=(V, rank))
    W2 = rng.normal(0, 0.7, size=(rank, V))
    return base, target, W1, W2


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_labels_equal_sum_of_minima(T):
    """1 - (1/2)||Q - P||_1 = sum_v min(P, Q) for distributions (an identity,
    evaluated here through the other formula at every position)."""
    base, target, W1, W2 = _case(1, 50, 4)
    d = D.draft_request(base, 7, W1, W2, T, 3, 0)
    lab = Lb.position_labels(target, base, 7, W1, W2, d["tokens"], T)
    prev = 7
    for k in range(1, 5):
        Q = D.DraftDist(base[k - 1], prev, W1, W2, T).prob()
        P = TargetDist(target[k - 1], T).prob()
        assert lab[k - 1] == pytest.approx(np.minimum(P, Q).sum(), abs=1e-12)
        prev = int(d["tokens"][k - 1])
    assert np.all((lab >= 0) & (lab <= 1))


def test_labels_are_one_when_target_equals_drafter():
    """Target rows equal to the drafter's own logits: P = Q, every label is 1."""
    V, gamma, T = 40, 3, 1.0
    base, _, W1, W2 = _case(2, V, gamma)
    d = D.draft_request(base, 5, W1, W2, T, 1, 0)
    rows, prev = [], 5
    for k in range(gamma):
        rows.append(base[k].astype(np.float64) + W1[prev] @ W2)
        prev = int(d["tokens"][k])
    target = np.stack(rows + [rows[-1]])  # float64 rows: exactly the drafter's logits
    lab = Lb.position_labels(target, base, 5, W1, W2, d["tokens"], T)
    assert np.allclose(lab, 1.0, atol=1e-12)


def test_labels_are_zero_for_disjoint_supports():
    """The target puts (numerically) all its mass where the drafter puts none."""
    V, gamma, T = 6, 2, 1.0
    base = np.full((gamma, V), -1000.0, dtype=np.float32)
    base[:, :3] = 0.0            # drafter: tokens 0..2
    target = np.full((gamma + 1, V), -1000.0, dtype=np.float32)
    target[:, 3:] = 0.0          # target: tokens 3..5
    W1 = np.zeros((V, 1))
    W2 = np.zeros((1, V))
    d = D.draft_request(base, 0, W1, W2, T, 0, 0)
    lab = Lb.position_labels(target, base, 0, W1, W2, d["tokens"], T)
    assert np.allclose(lab, 0.0, atol=1e-12)


def test_label_is_the_empirical_acceptance_rate():
    """Over many requests with the same rows, the verifier accepts position 1
    with frequency c*_1 (binomial bound)."""
    V, gamma, n, T = 8, 1, 4000, 1.0
    base, target, W1, W2 = _case(5, V, gamma)
    acc = 0
    lab = None
    for r in range(n):
        d = D.draft_request(base, 2, W1, W2, T, 11, r)
        v = Vf.verify_request(target, base, 2, W1, W2, d["tokens"], 1, T, 11, r)
        acc += v["A"]
        if lab is None:
            lab = Lb.position_labels(target, base, 2, W1, W2, d["tokens"], T)[0]
    sd = np.sqrt(lab * (1 - lab) / n)
    assert abs(acc / n - lab) < 4.5 * sd


def test_greedy_labels_are_argmax_agreement():
    V, gamma = 30, 4
    base, target, W1, W2 = _case(7, V, gamma)
    d = D.draft_request(base, 1, W1, W2, 0.0, 0, 0)
    lab = Lb.position_labels(target, base, 1, W1, W2, d["tokens"], 0.0)
    prev = 1
    for k in range(1, gamma + 1):
        l32 = base[k - 1] + (W1[prev] @ W2).astype(np.float32)
        same = int(np.argmax(l32)) == int(np.argmax(target[k - 1]))
        assert lab[k - 1] == (1.0 if same else 0.0)
        prev = int(d["tokens"][k - 1])
