"""Exact output law of the oracle's per-request pipeline, found by treating it
as a black box over its uniforms.

Each random decision of a round consumes one uniform, and every decision is a
monotone step function of its own uniform (inverse-CDF draws are non-decreasing
in u; a ratio test accepts exactly for u below a threshold). So the outcome
partition of (0, 1) at each decision can be found by bisection on the observed
outcome alone, without re-computing any probability the oracle computes. A
depth-first walk over decisions then yields every possible emitted sequence
with its exact probability (to the bisection width, 1e-14).
"""
from oracle import draft as D, verify as Vf, gated as G, philox

EPS = 1e-15


def run(monkeypatch, base_r, target_r, anchor, W1, W2, T, L_of, script, gate=None):
    """One request through the oracle's draft and verification with scripted
    uniforms; `gate` (float32 gate values [V, rank]) selects the gated head,
    whose W1 must then hold float32 (bf16-valued) rows."""
    calls = []

    def stub(seed, r, k, purpose):
        i = len(calls)
        calls.append((k, purpose))
        return script[i] if i < len(script) else 0.5

    monkeypatch.setattr(D, "uniform", stub)
    monkeypatch.setattr(Vf, "uniform", stub)
    monkeypatch.setattr(G, "uniform", stub)
    if gate is None:
        d = D.draft_request(base_r, anchor, W1, W2, T, seed=0, r=0)
        a_rows = None
    else:
        d = G.draft_request_gated(base_r, anchor, W1, gate, W2, T, seed=0, r=0)
        a_rows = G.state_rows(anchor, d["tokens"], W1, gate)
    L = L_of(d["tokens"])
    v = Vf.verify_request(target_r, base_r, anchor, W1, W2, d["tokens"], L, T, seed=0, r=0, a_rows=a_rows)
    return calls, d["tokens"], v


def _observe(call, tokens, v):
    k, purpose = call
    if purpose == philox.DRAFT:
        return int(tokens[k - 1])
    if purpose == philox.ACCEPT:
        return bool(v["A"] >= k)
    return int(v["new_token"])


def law(monkeypatch, base_r, target_r, anchor, W1, W2, T, L_of, gate=None):
    """dict: emitted tuple -> probability, plus dict: draft tuple -> probability."""
    out = {}

    def obs(script, n):
        calls, tokens, v = run(monkeypatch, base_r, target_r, anchor, W1, W2, T, L_of, script, gate)
        return _observe(calls[n], tokens, v)

    def segments(script, n):
        f = lambda u: obs(script + [u], n)
        pts = []

        def rec(lo, hi, flo, fhi):
            if flo == fhi:
                return
            if hi - lo < 1e-14:
                pts.append(0.5 * (lo + hi))
                return
            mid = 0.5 * (lo + hi)
            fm = f(mid)
            rec(lo, mid, flo, fm)
            rec(mid, hi, fm, fhi)

        lo, hi = EPS, 1.0 - EPS
        rec(lo, hi, f(lo), f(hi))
        edges = [0.0] + pts + [1.0]
        return [(edges[i], edges[i + 1]) for i in range(len(edges) - 1)]

    def dfs(script, weight):
        calls, tokens, v = run(monkeypatch, base_r, target_r, anchor, W1, W2, T, L_of, script, gate)
        n = len(script)
        if len(calls) == n:
            key = tuple(int(x) for x in v["out"])
            out[key] = out.get(key, 0.0) + weight
            return
        for a, b in segments(script, n):
            if b > a:
                dfs(script + [0.5 * (a + b)], weight * (b - a))

    dfs([], 1.0)
    return out


def lossless_violation(emitted_law, P_rows, L):
    """max |P(reach i, h, y_i = v) - P(reach i, h) P_{i-1}(v)| over i <= L+1.

    "reach i with history h": the first i-1 emitted tokens are h and were all
    accepted draft tokens (the round emitted more than i-1 tokens).
    """
    worst = 0.0
    for i in range(1, L + 2):
        joint, reach = {}, {}
        for seq, p in emitted_law.items():
            if len(seq) >= i:  # tokens before position i were accepted drafts
                h = seq[:i - 1]
                reach[h] = reach.get(h, 0.0) + p
                joint[(h, seq[i - 1])] = joint.get((h, seq[i - 1]), 0.0) + p
        V = len(P_rows[i - 1])
        for h, ph in reach.items():
            for v in range(V):
                worst = max(worst, abs(joint.get((h, v), 0.0) - ph * P_rows[i - 1][v]))
    return worst
