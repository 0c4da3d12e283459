"""One DSpark round, draft -> schedule -> verify, one request at a time (oracle).

The decoding cycle of the pages ([GN] §Arquitetura, decoding-cycle paragraph):
the target's last token is the anchor; the drafter proposes gamma tokens with
per-position confidences; the scheduler picks each request's verification
length; the target verifies the kept prefix and emits the accepted tokens plus
one corrected or bonus token.

The scheduler is global (it sees every request's confidences), while drafting
and verification are independent per request, so `requests` may select a
subset to draft and verify (used for sampled checks at full size and for the
bounded CPU baseline); the scheduled lengths always come from all requests.
"""

import numpy as np

from .draft import decode, draft_request
from .gated import draft_request_gated, state_rows
from .schedule import schedule
from .verify import verify_request


def run_round(inp, requests=None, mode=None):
    """inp: dict with base [R,g,V], target [R,g+1,V] (uint16 bf16 bits or float32),
    anchor [R], W1 [V,rank], W2 [rank,V], conf [R,g], conf_lag [R,g] or None,
    sps [n], T, seed, mode, and optionally gate [V,rank] (the gated head's
    gate values, oracle/gated.py). Returns dict of per-request results."""
    R = inp["anchor"].shape[0]
    mode = inp["mode"] if mode is None else mode
    T = float(inp["T"])
    seed = int(inp["seed"])
    W1f = decode(inp["W1"]).astype(np.float64)
    W2f = decode(inp["W2"]).astype(np.float64)
    gate = inp.get("gate")
    if gate is not None:
        W1_32, Z_32 = decode(inp["W1"]), decode(gate)
    sched = schedule(inp["conf"], inp["sps"], mode, inp.get("conf_lag"))
    reqs = range(R) if requests is None else requests
    res = {"sched": sched, "req": {}}
    for r in reqs:
        base_r = decode(inp["base"][r])
        target_r = decode(inp["target"][r])
        if gate is None:
            d = draft_request(base_r, int(inp["anchor"][r]), W1f, W2f, T, seed, r)
            a_rows = None
        else:
            d = draft_request_gated(base_r, int(inp["anchor"][r]), W1_32, Z_32, W2f, T, seed, r)
            a_rows = state_rows(int(inp["anchor"][r]), d["tokens"], W1_32, Z_32)
        v = verify_request(target_r, base_r, int(inp["anchor"][r]), W1f, W2f,
                           d["tokens"], sched["L"][r], T, seed, r, a_rows=a_rows)
        res["req"][r] = {"draft": d, "verify": v}
    return res
