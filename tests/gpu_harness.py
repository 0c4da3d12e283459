"""Shared helpers of the GPU parity tests: device inputs from the seeded
generators, one library round through the C ABI, and the comparison with the
oracle under the parity contract:

  * token ids, accepted lengths, scheduled lengths: bit-exact, except a
    sampling decision whose uniform lies within 1e-6 of the oracle's boundary
    (a CDF edge C_{x-1}/Z, C_x/Z, or the ratio p/q); such decisions are counted,
    and later positions of that request are excluded (they are conditioned on
    a different token);
  * probabilities (q_tok, p_tok): within 2e-3 relative;
  * greedy (temperature 0): fully bit-exact, the recorded maximum logit
    fl32(base + fl32(bias)) of every drafted position included.

The report counts, besides the boundary cases, how many requests had their
residual draw (a rejection before the scheduled length) and their bonus draw
compared with the oracle.
"""
import numpy as np
import torch

import workloads as W
from oracle.round import run_round
from speculative_decoding_draft_seq_gb300 import dspark

BOUNDARY = 1e-6
PROB_RTOL = 2e-3


device_inputs = W.device_inputs


def gpu_round(cfg, inp=None, device="cuda"):
    inp = device_inputs(cfg, device) if inp is None else inp
    R, gamma, V = inp["base"].shape
    rank = inp["W1"].shape[1]
    dt = dspark.BF16 if inp["base"].dtype == torch.bfloat16 else dspark.FP32
    ws = dspark.new_workspace(R, gamma, V, rank, dt, inp["sps"].numel(), device)
    out = dspark.RoundOutputs(R, gamma, device)
    if inp.get("gate") is not None:  # the recurrent (gated) head
        dspark.round_gated(inp["base"], inp["target"], inp["anchor"], inp["W1"], inp["gate"], inp["W2"],
                           inp["conf"], inp["conf_lag"], inp["sps"], inp["mode"], inp["T"], inp["seed"], out, ws)
    else:
        dspark.round_(inp["base"], inp["target"], inp["anchor"], inp["W1"], inp["W2"], inp["conf"],
                      inp["conf_lag"], inp["sps"], inp["mode"], inp["T"], inp["seed"], out, ws)
    status = dspark.device_status(ws)
    res = out.host()
    res["status"] = status
    res["launches"] = dspark.last_launch_count()
    return res


def oracle_round(cfg, requests):
    return run_round(W.oracle_inputs(cfg, requests), requests=requests)


def _rel(a, b):
    a, b = float(a), float(b)
    return abs(a - b) / max(abs(b), 1e-30)


def compare(cfg, g, o, requests, check_schedule=True):
    """Asserts the parity contract; returns a report of counted cases."""
    rep = dict(requests=len(requests), draft_boundary=0, accept_boundary=0, sample_boundary=0,
               verify_excluded=0, positions=0, max_rel_q=0.0, max_rel_p=0.0, min_greedy_gap=np.inf,
               resid_compared=0, bonus_compared=0)
    T = cfg.T
    gamma = cfg.gamma
    assert g["status"] == dspark.OK, dspark.status_string(g["status"])
    if check_schedule:
        s = o["sched"]
        assert np.array_equal(g["sched_len"], s["L"].astype(np.int32)), "scheduled lengths differ"
        assert int(g["K"][0]) == s["K"]
        assert g["tau_theta"][0] == s["tau"] and g["tau_theta"][1] == s["theta"]
    for r in requests:
        d = o["req"][r]["draft"]
        v = o["req"][r]["verify"]
        gt = g["tokens"][r]
        mis = next((k for k in range(gamma) if gt[k] != d["tokens"][k]), None)
        if T == 0:
            rep["min_greedy_gap"] = min(rep["min_greedy_gap"], float(np.min(d["gap"])))
        if mis is not None:
            assert T > 0 and d["margin"][mis] < BOUNDARY, (
                f"request {r}: draft token {mis + 1} differs ({gt[mis]} vs {d['tokens'][mis]}), "
                f"oracle margin {d['margin'][mis]:.3g}, gap {d['gap'][mis]:.3g}")
            rep["draft_boundary"] += 1
        upto = gamma if mis is None else mis
        rep["positions"] += upto
        for k in range(upto):
            e = _rel(g["q_tok"][r, k], d["q"][k])
            rep["max_rel_q"] = max(rep["max_rel_q"], e)
            assert e < PROB_RTOL, f"request {r} q_tok[{k}] {g['q_tok'][r, k]} vs {d['q'][k]}"
            if T > 0:
                lse_g = g["q_stats"][r, k, 0] + T * np.log(g["q_stats"][r, k, 1])
                lse_o = d["m"][k] + T * np.log(d["Z"][k])
                assert abs(lse_g - lse_o) < PROB_RTOL * T, f"request {r} q_stats[{k}]"
            else:  # greedy: the recorded maximum logit fl32(base + fl32(bias)) and Z = 1, bit for bit
                assert np.float32(g["q_stats"][r, k, 0]) == np.float32(d["m"][k]), (
                    f"request {r} greedy max logit[{k}] {g['q_stats'][r, k, 0]!r} vs {d['m'][k]!r}")
                assert g["q_stats"][r, k, 1] == 1.0
        L = int(o["sched"]["L"][r])
        if mis is not None and mis < L:
            rep["verify_excluded"] += 1
            continue
        for k in range(L):
            e = _rel(g["p_tok"][r, k], v["p"][k]) if v["p"][k] > 1e-30 else abs(float(g["p_tok"][r, k]))
            rep["max_rel_p"] = max(rep["max_rel_p"], e)
            assert e < PROB_RTOL, f"request {r} p_tok[{k}] {g['p_tok'][r, k]} vs {v['p'][k]}"
        assert np.all(g["p_tok"][r, L:] == 0)
        gA = int(g["accepted_len"][r])
        if gA != v["A"]:
            k = min(gA, v["A"]) + 1
            m = [x for kind, kk, x in v["margins"] if kind == "accept" and kk == k]
            assert T > 0 and m and m[0] < BOUNDARY, (
                f"request {r}: accepted {gA} vs {v['A']}, margin {m}")
            rep["accept_boundary"] += 1
            continue
        A = gA
        assert np.array_equal(g["out_tokens"][r, :A], v["out"][:A])
        assert np.all(g["out_tokens"][r, A + 1:] == -1)
        # the emitted token: the residual draw after the first rejection (A < L), else the bonus draw
        rep["resid_compared" if A < L else "bonus_compared"] += 1
        if g["out_tokens"][r, A] != v["new_token"]:
            m = [x for kind, kk, x in v["margins"] if kind in ("resid", "bonus")]
            assert T > 0 and m and m[0] < BOUNDARY, (
                f"request {r}: emitted {g['out_tokens'][r, A]} vs {v['new_token']}, margin {m}")
            rep["sample_boundary"] += 1
    return rep
