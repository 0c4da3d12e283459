"""Recurrent (gated) sequential head -- oracle.

Test infrastructure: imported only by the tests, the smoke entry point and the
benchmark's CPU legs; never by the library.

What the pages define ([GN] "Geração semiautorregressiva", "Head RNN"; [AI]
the two variants of the sequential module; [JD] the RNN head paragraph): a
second form of the sequential head keeps a recurrent state s_k that gathers
the whole prefix drafted so far inside the block, updated through gates, so
that position k can use tokens before x_{k-1}; the Markov head (the default)
sees x_{k-1} only. The pages give no equations for it.

Reading taken (the plainest gated recurrence over the head's own input, the
previous token; listed in the design notes):
  * the input at position k is the previous token prev_k (the anchor at
    k = 1, else x_{k-1}), one-hot, as for the Markov head; a linear map of a
    one-hot input is a row lookup, so the candidate state is W1[prev_k] and
    the update gate is a per-token row z[prev_k] in [0, 1] (the sigmoid of the
    gate's linear map, which depends on the token only and is therefore
    tabulated once: the head's parameter here is the table of gate values);
  * s_0 = 0 and s_k = (1 - z[prev_k]) * s_{k-1} + z[prev_k] * W1[prev_k]
    (elementwise: a minimal gated unit with its gate driven by the input);
  * the bias of position k is a_k . W2 with a_k = bf16(s_k), the state in the
    precision of the weights it is multiplied with (W1's rows are bf16 too).
With every gate value 1 the state is W1[prev_k] and the head is the Markov
head exactly; with every gate value 0 the bias is 0 (the parallel drafter).

Precision: the state rounds to bf16 before it enters the bias, so the
rounding decides the operand of every later product; that decision is taken
in the precision the state is carried in, float32, with the operations in the
order written above, each rounded once: t = fl32((1 - z) * s),
s' = fl32(t + z * w) (z * w of two bf16 values is exact in float32). The
bias itself, the softmax and the draw are float64 as in oracle/draft.py.

Pins (tests/test_oracle_gated.py): bf16 rounding against torch's conversion
and hand-made ties; gate values 1 reproduce the Markov draft and
verification exactly; gate values 0 reproduce the draft with W2 = 0; with a
constant gate c the state equals the closed form sum_j c (1 - c)^(k-j)
W1[prev_j] (float64) within float32 rounding; the output law of a gated
round by exact enumeration at V = 3, gamma = 2 equals the target rows.
"""

import numpy as np

from .draft import DraftDist, inverse_cdf
from .philox import uniform, DRAFT


def round_bf16(x):
    """float32 -> nearest bf16 value (ties to the even significand), as float32.

    Written from the definition: keep the upper 16 bits of the float32
    pattern, adding half an ulp of bf16 plus the kept last bit (so that a tie
    rounds to even). Finite inputs only."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def gated_update(s, z, w):
    """One state update in float32: fl32(fl32((1 - z) * s) + z * w)."""
    s = np.asarray(s, dtype=np.float32)
    z = np.asarray(z, dtype=np.float32)
    w = np.asarray(w, dtype=np.float32)
    t = (np.float32(1.0) - z) * s
    return (t + z * w).astype(np.float32)


def state_rows(anchor, tokens, W1_32, Z_32):
    """A-operand rows a_k = bf16(s_k) for k = 1..len(tokens) (float32 [n, rank]).

    Position k's state uses prev_1 = anchor and prev_k = tokens[k-2]; only
    tokens[0..n-2] are read (the last drafted token feeds no position of
    this block)."""
    n = len(tokens)
    rank = W1_32.shape[1]
    s = np.zeros(rank, dtype=np.float32)
    rows = np.zeros((n, rank), dtype=np.float32)
    prev = int(anchor)
    for k in range(1, n + 1):
        s = gated_update(s, Z_32[prev], W1_32[prev])
        rows[k - 1] = round_bf16(s)
        if k < n:
            prev = int(tokens[k - 1])
    return rows


def draft_request_gated(base_r, anchor, W1_32, Z_32, W2f, T, seed, r):
    """Draft gamma tokens of request r with the gated head; same outputs as
    oracle.draft.draft_request (tokens, q, m, Z, margin, gap) plus the A rows
    used (a [gamma, rank])."""
    gamma = base_r.shape[0]
    rank = W1_32.shape[1]
    out = {k: np.zeros(gamma) for k in ("q", "m", "Z", "margin", "gap")}
    out["tokens"] = np.zeros(gamma, dtype=np.int64)
    out["a"] = np.zeros((gamma, rank), dtype=np.float32)
    s = np.zeros(rank, dtype=np.float32)
    prev = int(anchor)
    for k in range(1, gamma + 1):
        s = gated_update(s, Z_32[prev], W1_32[prev])
        a = round_bf16(s)
        out["a"][k - 1] = a
        dist = DraftDist(base_r[k - 1], None, None, W2f, T, a_row=a)
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
