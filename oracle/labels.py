"""Acceptance labels of the confidence head -- oracle.

Test infrastructure: imported only by the tests, the smoke entry point and the
benchmark's CPU legs; never by the library.

What the pages define ([GN] "Confidence head", "Calibração posterior"): the
confidence head is trained to predict, for each draft position k, the
probability that token k passes verification given that all earlier tokens
did. Under speculative sampling that probability is
    c*_k = sum_v min(P_{k-1}(v), Q_k(v)) = 1 - (1/2) || Q_k - P_{k-1} ||_1,
Q_k the drafter's distribution at position k (conditioned on the drafted
tokens before it) and P_{k-1} the target's distribution after the anchor and
k - 1 drafted tokens (the same rows the verifier uses). The page prints the
formula garbled; the reading taken is one minus the total variation distance,
which is the acceptance probability of the rule in oracle/verify.py.

Readings where the pages are silent:
  * The label is computed for every draft position k = 1..gamma of every
    request, whatever the scheduler admitted (it is a training signal, not a
    decision).
  * Greedy (T = 0): both distributions are one-hot at their argmax (lowest
    index on ties), so c*_k is 1 when the argmaxes agree and 0 otherwise.

Pins (tests/test_oracle_labels.py): the identity with sum_v min(P, Q); c* = 1
when the target rows equal the drafter's logits; c* = 0 for disjoint
supports; the empirical acceptance frequency of the verifier at position 1
over many requests; greedy agreement.
"""

import numpy as np

from .draft import DraftDist
from .verify import TargetDist


def position_labels(target_r, base_r, anchor, W1f, W2f, tokens, T):
    """c*_k for k = 1..gamma of one request (float64 [gamma]).

    target_r [gamma+1, V] and base_r [gamma, V] float32 rows, tokens [gamma]
    the drafted tokens (position k's distribution is conditioned on them)."""
    gamma = base_r.shape[0]
    out = np.zeros(gamma)
    prev = int(anchor)
    for k in range(1, gamma + 1):
        Q = DraftDist(base_r[k - 1], prev, W1f, W2f, T)  # one-hot at the argmax for T = 0
        P = TargetDist(target_r[k - 1], T)
        out[k - 1] = 1.0 - 0.5 * float(np.abs(Q.prob() - P.prob()).sum())
        prev = int(tokens[k - 1])
    return out
