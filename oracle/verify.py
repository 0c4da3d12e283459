"""Lossless speculative-sampling verification -- oracle.

What the pages define ([GN] §Definição do problema and the decoding-cycle
paragraph of §Arquitetura; [AI] "El cuello de botella de la inferencia"):
the target scores the anchor plus the scheduled draft tokens in one forward
pass; rejection sampling keeps the longest prefix consistent with the target
distribution, so the output distribution equals the target's; after the first
rejected token a corrected token is emitted (the worked round: prompt ABC,
anchor D, draft EFGH, H dropped by the scheduler, E and F accepted, G
rejected and replaced by a corrected G*).

The acceptance rule is the standard speculative-sampling rule the pages refer
to (Leviathan et al. 2022, cited on the GeekNews page): accept x_k with
probability min(1, P(x_k) / Q(x_k)); at the first rejection j resample from
normalize(max(0, P - Q)); if every scheduled token is accepted, draw one bonus
token from the next target row. Per-step acceptance probability is then
sum_v min(P, Q) = 1 - (1/2)||P - Q||_1, the quantity the pages use as the
confidence label ([GN] "Confidence head", c*_k).

Readings where the pages are silent (each listed in the design notes):
  * Target row k of request r is the target distribution after the anchor and
    k draft tokens: P_k = softmax(t[r, k, :] / T), k = 0..gamma.
  * The target uses the same temperature T as the draft; T = 0 is greedy
    (one-hot at the argmax of the bf16/fp32 target row, lowest index on ties).
  * Ratio test is strict: accept iff u < P_{k-1}(x_k) / Q_k(x_k).
  * Q_k is recomputed exactly as the draft defined it (prev = x_{k-1}, or the
    anchor at k = 1).
  * If the residual has zero mass under rounding, sample from P_{j-1}.
  * Uniforms: ACCEPT at (r, k), RESID at (r, j), BONUS at (r, L_r + 1).

Pins (tests/test_oracle_verify.py): exact enumeration of the output law at
V <= 4, gamma <= 3 over every draft sequence and accept/reject branch equals
the target rows; chi-square of emitted tokens at V <= 16 over many requests;
empirical position-1 acceptance equals sum_v min(P, Q); the worked round of
the pages; an anticipating scheduler fails the same enumeration. At the full
vocabulary (V = 129280, rank 256), closed forms: a target row equal to the
drafter's logits with the drafted token pushed down and exactly its mass moved
onto a second token makes the residual a point mass there (a draw from P or Q
would not be); a boosted token is the residual's point mass; a dominant token
is the bonus.
"""

import numpy as np

from .draft import DraftDist, inverse_cdf
from .philox import uniform, ACCEPT, RESID, BONUS


class TargetDist:
    """P_k = softmax(t / T) (float64), or one-hot at the argmax for T = 0."""

    def __init__(self, t_row_f32, T):
        V = t_row_f32.shape[0]
        if T == 0.0:
            x = int(np.argmax(t_row_f32))
            self.w = np.zeros(V, dtype=np.float64)
            self.w[x] = 1.0
            self.m = float(t_row_f32[x])
        else:
            t = t_row_f32.astype(np.float64) / T
            self.m = float(t.max())
            self.w = np.exp(t - self.m)
        self.Z = float(np.cumsum(self.w)[-1])

    def prob(self):
        return self.w / self.Z


def verify_request(target_r, base_r, anchor, W1f, W2f, tokens, L, T, seed, r, a_rows=None):
    """Verify the first L draft tokens of request r.

    target_r [gamma+1, V] float32, base_r [gamma, V] float32, tokens [gamma].
    a_rows [gamma, rank]: the head's operand rows when the head is not the
    Markov head (oracle/gated.py state_rows); Q_k is then recomputed from
    a_rows[k-1] . W2.
    Returns dict(A, out [A+1] tokens emitted, p [L] = P_{k-1}(x_k),
    q [L] = Q_k(x_k), margins list of (kind, k, distance), new_token).
    """
    L = int(L)
    p = np.zeros(L)
    q = np.zeros(L)
    margins = []
    P = [TargetDist(target_r[k], T) for k in range(L + 1)]
    Qs = []
    prev = int(anchor)
    for k in range(1, L + 1):
        Qs.append(DraftDist(base_r[k - 1], prev, W1f, W2f, T,
                            a_row=None if a_rows is None else a_rows[k - 1]))
        prev = int(tokens[k - 1])
    for k in range(1, L + 1):
        x = int(tokens[k - 1])
        p[k - 1] = P[k - 1].w[x] / P[k - 1].Z
        q[k - 1] = Qs[k - 1].w[x] / Qs[k - 1].Z
    A = L
    for k in range(1, L + 1):
        u = uniform(seed, r, k, ACCEPT)
        ratio = p[k - 1] / q[k - 1] if q[k - 1] > 0 else float("inf")
        if T > 0:
            margins.append(("accept", k, abs(u - ratio)))
        if not (u < ratio):
            A = k - 1
            break
    if A < L:
        j = A + 1
        res = np.maximum(0.0, P[j - 1].prob() - Qs[j - 1].prob())
        u = uniform(seed, r, j, RESID)
        if np.cumsum(res)[-1] > 0.0:
            new, margin, _ = inverse_cdf(res, u)
        else:
            new, margin, _ = inverse_cdf(P[j - 1].w, u)
        if T > 0:
            margins.append(("resid", j, margin))
    else:
        u = uniform(seed, r, L + 1, BONUS)
        new, margin, _ = inverse_cdf(P[L].w, u)
        if T > 0:
            margins.append(("bonus", L + 1, margin))
    out = [int(t) for t in tokens[:A]] + [int(new)]
    return dict(A=A, out=np.array(out, dtype=np.int64), p=p, q=q,
                margins=margins, new_token=int(new))
