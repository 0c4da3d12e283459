"""The oracle evaluated for many requests at once, for the full-size parity
tests: drafting and verification are independent per request, so the oracle's
per-request work is spread over host processes; the schedule (global over all
requests) is computed once in the calling process.

Test infrastructure only. The workers are started with the `spawn` method (a
fresh interpreter each, safe next to the calling process's CUDA context) and
import numpy, the seeded generators and the oracle, nothing else. Each worker
builds a workload's weights once and keeps them while it serves that
workload.
"""
import multiprocessing as mp
import os

import numpy as np

import workloads as W
from oracle import labels as Lb
from oracle.draft import decode
from oracle.round import run_round
from oracle.schedule import schedule

_POOL = None
_CACHE = {}  # in a worker: the inputs of one workload without its logit rows


def _procs():
    n = os.cpu_count() or 2
    return max(1, min(16, n - 1))


def pool():
    global _POOL
    if _POOL is None:
        _POOL = mp.get_context("spawn").Pool(_procs())
    return _POOL


def _inputs(cfg, reqs):
    if cfg not in _CACHE:  # everything but the logit rows (as oracle_inputs builds it)
        _CACHE.clear()
        d = W.host_inputs(cfg)
        d["W1"], d["W2"] = W.weights_np(cfg)
        if cfg.gated:
            d["gate"] = W.gate_np(cfg)
        _CACHE[cfg] = d
    inp = dict(_CACHE[cfg])
    base, tgt = W.logits_rows_np(cfg, reqs)
    inp["base"] = {r: base[i] for i, r in enumerate(reqs)}
    inp["target"] = {r: tgt[i] for i, r in enumerate(reqs)}
    return inp


def _round_chunk(args):
    cfg, reqs = args
    return run_round(_inputs(cfg, reqs), requests=reqs)["req"]


def _labels_chunk(args):
    cfg, reqs, tokens = args
    inp = _inputs(cfg, reqs)
    W1f, W2f = decode(inp["W1"]).astype(np.float64), decode(inp["W2"]).astype(np.float64)
    return {r: Lb.position_labels(decode(inp["target"][r]), decode(inp["base"][r]), int(inp["anchor"][r]), W1f,
                                  W2f, tokens[i], cfg.T) for i, r in enumerate(reqs)}


def _chunks(requests, size):
    requests = list(requests)
    return [requests[i:i + size] for i in range(0, len(requests), size)]


def oracle_round(cfg, requests, chunk=4):
    """The oracle's round for `requests` (same structure as oracle.round.run_round)."""
    h = W.host_inputs(cfg)
    res = {"sched": schedule(h["conf"], h["sps"], cfg.mode, h["conf_lag"]), "req": {}}
    for part in pool().map(_round_chunk, [(cfg, c) for c in _chunks(requests, chunk)]):
        res["req"].update(part)
    return res


def oracle_labels(cfg, tokens, requests, chunk=4):
    """The oracle's acceptance labels c*_k for `requests`, given the drafted tokens [R, gamma]."""
    jobs = [(cfg, c, [np.asarray(tokens[r]) for r in c]) for c in _chunks(requests, chunk)]
    out = {}
    for part in pool().map(_labels_chunk, jobs):
        out.update(part)
    return out
