"""The parallel oracle used by the full-size parity tests returns exactly what
the oracle returns when called directly, request by request (host-side, no
GPU)."""
import numpy as np

import oracle_pool
import workloads as W
from oracle import labels as Lb
from oracle.draft import decode
from oracle.round import run_round


def _same(a, b):
    if isinstance(a, dict):
        assert a.keys() == b.keys()
        for k in a:
            _same(a[k], b[k])
    elif isinstance(a, (list, tuple)):
        assert len(a) == len(b)
        for x, y in zip(a, b):
            _same(x, y)
    else:
        np.testing.assert_array_equal(a, b)


def test_pooled_round_and_labels_equal_the_direct_oracle():
    cfg = W.with_(W.CONFIGS["small"], R=10, V=640, rank=64)
    reqs = [0, 3, 4, 9]
    direct = run_round(W.oracle_inputs(cfg, reqs), requests=reqs)
    pooled = oracle_pool.oracle_round(cfg, reqs, chunk=3)
    _same(direct["sched"], pooled["sched"])
    _same(direct["req"], pooled["req"])
    tokens = np.stack([direct["req"][r]["draft"]["tokens"] if r in reqs else np.zeros(cfg.gamma, np.int64)
                       for r in range(cfg.R)])
    inp = W.oracle_inputs(cfg, reqs)
    W1f, W2f = decode(inp["W1"]).astype(np.float64), decode(inp["W2"]).astype(np.float64)
    lab = oracle_pool.oracle_labels(cfg, tokens, reqs, chunk=2)
    for r in reqs:
        ref = Lb.position_labels(decode(inp["target"][r]), decode(inp["base"][r]), int(inp["anchor"][r]), W1f, W2f,
                                 tokens[r], cfg.T)
        np.testing.assert_array_equal(lab[r], ref)
