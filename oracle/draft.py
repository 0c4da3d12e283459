"""Sequential (semi-autoregressive) drafting stage with the Markov head -- oracle.

What the pages define ([GN] §Arquitetura, "Geração semiautorregressiva"):
  * Parallel stage: one backbone pass yields base logits for all gamma block
    positions; the anchor token (the target's last sampled token) is treated as
    the first prediction position ([GN] "Etapa paralela"; [JD] the section on
    the two-stage split). The base logits are an INPUT here: base[k-1, :] are
    the base logits of block position k.
  * Sequential stage: a prefix-dependent transition bias B_k is added to the
    base logits so that position k is conditioned on the tokens actually
    sampled before it ([GN] "Etapa sequencial").
  * Markov head: a first-order transition that depends only on the previous
    token; the V x V matrix is approximated by the low-rank product B = W1 W2
    (default rank 256) ([GN] "Head de Markov"; [JD] Markov head paragraph).

Readings where the pages are silent (each listed in the design notes):
  * The bias is added unscaled, and the temperature T divides the sum:
    l = base + W1[prev] . W2, distribution softmax(l / T).
  * prev at position 1 is the anchor; at position k > 1 it is x_{k-1}.
  * Sampling is inverse-CDF in vocabulary order with one uniform per decision:
    x = smallest v with u * Z < C_v, C_v = sum_{i<=v} w_i, Z = C_{V-1}; if
    rounding leaves no such v, the last v with w_v > 0.
  * T = 0 is greedy: argmax of l with the lowest index on ties. Because an
    argmax is an integer decided by floating point, it is taken in the
    precision the kernel computes l in: l32 = fl32(base + fl32(bias)).

Arithmetic: float64 throughout for T > 0 (bias by a float64 matrix-vector
product, exp, prefix sums); float32 only for the greedy l32 above.

Pins (tests/test_oracle_draft.py): the bias equals an independent float64
matmul; W2 = 0 reduces the draft to the plain parallel drafter; rank = V with
W1 = I reduces the head to a full V x V transition-table lookup; the sampler
matches softmax by chi-square at V <= 16; small T converges to the argmax;
hand-built CDFs land on the expected index.
"""

import numpy as np

from .philox import uniform, DRAFT


def decode(x):
    """Inputs to float32, exactly: bf16 bit patterns (uint16) or float32."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32)
    if x.dtype == np.float32:
        return x
    raise TypeError(f"unsupported input dtype {x.dtype}")


def markov_bias(W1f, W2f, prev):
    """B[prev, :] = W1[prev, :] . W2 in float64 ([GN] "Head de Markov")."""
    return np.asarray(W1f[prev], dtype=np.float64) @ np.asarray(W2f, dtype=np.float64)


def inverse_cdf(w, u):
    """Inverse-CDF draw from unnormalised non-negative weights w with uniform u.

    Returns (index, margin, Z): margin is the distance from u to the nearest
    boundary C_{x-1}/Z or C_x/Z of the chosen interval (0 when the rounding
    fallback fired). Prefix sums run in index order in float64.
    """
    C = np.cumsum(np.asarray(w, dtype=np.float64))
    Z = float(C[-1])
    t = u * Z
    x = int(np.searchsorted(C, t, side="right"))  # smallest v with C_v > t
    if x >= len(C):
        x = int(np.flatnonzero(np.asarray(w) > 0)[-1])
        return x, 0.0, Z
    lo = float(C[x - 1]) / Z if x > 0 else 0.0
    hi = float(C[x]) / Z
    return x, min(u - lo, hi - u), Z


class DraftDist:
    """Draft distribution Q_k at one block position.

    w: unnormalised weights (float64); Z = sum in index order; m: the max of
    the (tempered) logits the weights are relative to; for T = 0, w is one-hot
    at the fp32 argmax, m is that fp32 max and Z = 1; gap is the fp32 top-2
    gap (infinite for T > 0) so a flipped argmax can be attributed.
    """

    def __init__(self, base_row_f32, prev, W1f, W2f, T, a_row=None):
        # a_row: the head's operand row when it is not W1[prev] (the gated
        # head's rounded state, oracle/gated.py); the bias is a_row . W2
        if a_row is None:
            bias = markov_bias(W1f, W2f, prev)
        else:
            bias = np.asarray(a_row, dtype=np.float64) @ np.asarray(W2f, dtype=np.float64)
        V = base_row_f32.shape[0]
        if T == 0.0:
            l32 = base_row_f32 + bias.astype(np.float32)  # fl32(base + fl32(bias))
            x = int(np.argmax(l32))  # first occurrence = lowest index on ties
            self.w = np.zeros(V, dtype=np.float64)
            self.w[x] = 1.0
            self.m = float(l32[x])
            if V > 1:
                rest = np.delete(l32, x)
                self.gap = float(l32[x]) - float(rest.max())
            else:
                self.gap = float("inf")
        else:
            l = base_row_f32.astype(np.float64) + bias
            self.m = float(l.max())
            self.w = np.exp((l - self.m) / T)
            self.gap = float("inf")
        self.Z = float(np.cumsum(self.w)[-1])

    def prob(self):
        """Normalised probabilities Q(v) in float64."""
        return self.w / self.Z


def draft_request(base_r, anchor, W1f, W2f, T, seed, r):
    """Draft gamma tokens for request r ([GN] "Etapa sequencial").

    base_r: [gamma, V] float32 base logits of request r; anchor: int token id;
    W1f [V, rank], W2f [rank, V] decoded weights (float32 or float64). Returns dict with tokens [gamma]
    int64, q [gamma] (Q_k(x_k)), m [gamma], Z [gamma], margin [gamma]
    (inverse-CDF boundary distance, inf for T = 0), gap [gamma].
    """
    gamma = base_r.shape[0]
    out = {k: np.zeros(gamma) for k in ("q", "m", "Z", "margin", "gap")}
    out["tokens"] = np.zeros(gamma, dtype=np.int64)
    prev = int(anchor)
    for k in range(1, gamma + 1):
        dist = DraftDist(base_r[k - 1], prev, W1f, W2f, T)
        u = uniform(seed, r, k, DRAFT)
        x, margin, _ = inverse_cdf(dist.w, u)
        out["tokens"][k - 1] = x
        out["q"][k - 1] = dist.w[x] / dist.Z
        out["m"][k - 1] = dist.m
        out["Z"][k - 1] = dist.Z
        out["margin"][k - 1] = margin if T > 0 else float("inf")
        out["gap"][k - 1] = dist.gap
        prev = x
    return out
