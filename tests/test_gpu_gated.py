"""GPU parity of the recurrent (gated) sequential head ([GN] "Head RNN")
against the oracle, through the C ABI: the same parity contract as the Markov
head (tokens and lengths bit-exact but for counted boundary decisions,
probabilities within 2e-3 relative, greedy fully bit-exact)."""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import oracle_pool
    from gpu_harness import compare, device_inputs, gpu_round, oracle_round
    from speculative_decoding_draft_seq_gb300 import dspark

GATED = [
    # (R, gamma, V, rank): several chunks per CTA, a vocabulary tail, two M tiles
    (1, 1, 64, 64),       # the smallest tensor-core shape: one request, one step, one chunk
    (33, 6, 640, 256),
    (150, 4, 3000, 64),
    (200, 3, 2056, 128),
    (64, 5, 4104, 192),
]


def _cfg(R, gamma, V, rank, T, **kw):
    return W.Workload(f"gated_{R}_{gamma}_{V}_{rank}", R=R, gamma=gamma, V=V, rank=rank, dtype="bf16", T=T,
                      mode=W.CAUSAL, seed=5000 + R + gamma + rank, base_sd=1.5, w_sd=0.05,
                      target_sd=(0.45,), conf_law="decreasing", table="concave", n_table=R * (gamma + 1),
                      gated=True, **kw)


@pytest.mark.parametrize("R,gamma,V,rank", GATED)
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_gated_round_parity(R, gamma, V, rank, T):
    cfg = _cfg(R, gamma, V, rank, T)
    g = gpu_round(cfg)
    o = oracle_round(cfg, list(range(R)))
    rep = compare(cfg, g, o, list(range(R)))
    assert rep["positions"] > 0
    # the drafting launch (with the round's schedule, the row statistics and the chains) and, sampled, the
    # state staging and the residual sweep
    assert g["launches"] == (3 if T > 0 else 1), g["launches"]


def test_gated_uses_the_prefix():
    """With gates well below 1 the drafted tokens differ from the Markov
    head's on the same inputs (the state carries earlier tokens)."""
    cfg = _cfg(64, 6, 2048, 128, 1.0, gate_lo=0.1)
    inp = device_inputs(cfg)
    g = gpu_round(cfg, inp)
    m = gpu_round(cfg, dict(inp, gate=None))
    assert not np.array_equal(g["tokens"], m["tokens"])


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_gate_one_equals_the_markov_round(T):
    """Gate values 1: the gated path on the device gives the Markov head's
    round bit for bit (every output)."""
    cfg = _cfg(96, 5, 3000, 128, T)
    inp = device_inputs(cfg)
    ones = torch.ones_like(inp["W1"])
    g = gpu_round(cfg, dict(inp, gate=ones))
    m = gpu_round(cfg, dict(inp, gate=None))
    for key in ("tokens", "q_tok", "q_stats", "sched_len", "out_tokens", "accepted_len", "p_tok"):
        assert np.array_equal(g[key], m[key]), key


def test_gated_full_size_every_request():
    """The DeepSeek-scale round with the gated head, every request against the
    oracle."""
    cfg = W.with_(W.CONFIGS["ds"], gated=True)
    requests = list(range(cfg.R))
    g = gpu_round(cfg)
    rep = compare(cfg, g, oracle_pool.oracle_round(cfg, requests), requests)
    rep = {k: (float(v) if isinstance(v, (float, np.floating)) else v) for k, v in rep.items()}
    out_dir = os.environ.get("DSPARK_OUT_DIR", "runs")
    os.makedirs(out_dir, exist_ok=True)
    with open(os.path.join(out_dir, "parity_reports.jsonl"), "a") as f:
        f.write(json.dumps({"workload": "ds_gated", "T": cfg.T, "n_requests": len(requests), **rep}) + "\n")
    assert rep["resid_compared"] >= 30, rep


def test_gated_refuses_shapes_off_the_tensor_core_path():
    cfg = W.Workload("gated_fp32", R=4, gamma=3, V=130, rank=5, dtype="fp32", T=1.0, mode=W.CAUSAL, seed=7,
                     zipf=0.0, w_sd=0.4, n_table=16, gated=True)
    inp = device_inputs(cfg)
    with pytest.raises(dspark.DSparkError) as e:
        gpu_round(cfg, inp)
    assert e.value.status == dspark.ERR_INVALID_ARG


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_gated_mixed_domain(T):
    """The mixed-domain workload (256 requests: two M tiles, two CTAs' worth of
    draws per step on some SMs) with the gated head, sampled and greedy: 64
    requests, 32 in each M tile (both domains)."""
    cfg = W.with_(W.CONFIGS["mixed"], T=T, gated=True)
    requests = list(range(0, cfg.R, 4))
    g = gpu_round(cfg)
    compare(cfg, g, oracle_pool.oracle_round(cfg, requests), requests)


def _separate_calls(cfg, inp):
    """The round as three separate C-ABI calls: dspark_draft_sequential_gated,
    dspark_schedule and dspark_verify_gated, on one workspace and stream."""
    R, gamma, V = inp["base"].shape
    ws = dspark.new_workspace(R, gamma, V, cfg.rank, dspark.BF16, inp["sps"].numel())
    out = dspark.RoundOutputs(R, gamma)
    dspark.draft_sequential_gated(inp["base"], inp["anchor"], inp["W1"], inp["gate"], inp["W2"], inp["T"],
                                  inp["seed"], out.tokens, out.q_tok, out.q_stats, ws)
    dspark.schedule(inp["conf"], inp["conf_lag"], inp["sps"], inp["mode"], out.sched_len, out.K, out.tau_theta, ws)
    dspark.verify_gated(inp["target"], inp["base"], inp["anchor"], inp["W1"], inp["gate"], inp["W2"], out.tokens,
                        out.q_tok, out.q_stats, out.sched_len, inp["T"], inp["seed"], out.out_tokens,
                        out.accepted_len, out.p_tok, ws)
    res = out.host()
    res["status"] = dspark.device_status(ws)
    return res


# (R, gamma, V, rank, mode, T): two M tiles with a vocabulary tail, both admission modes, greedy, full rank
SEPARATE = [(150, 4, 3000, 64, W.CAUSAL, 1.0), (150, 4, 3000, 64, W.LAGGED, 1.0), (150, 4, 3000, 64, W.CAUSAL, 0.0),
            (64, 5, 4104, 256, W.CAUSAL, 1.0)]


@pytest.mark.parametrize("R,gamma,V,rank,mode,T", SEPARATE)
def test_gated_separate_calls_equal_the_round(R, gamma, V, rank, mode, T):
    """The stages called one by one (the gated drafting, the scheduler, the
    gated verification with its state replay for the residual draws) give
    every output of dspark_round_gated bit for bit, and match the oracle."""
    cfg = W.with_(_cfg(R, gamma, V, rank, T), mode=mode)
    inp = device_inputs(cfg)
    s = _separate_calls(cfg, inp)
    assert s["status"] == dspark.OK, dspark.status_string(s["status"])
    g = gpu_round(cfg, inp)
    for k in ("tokens", "q_tok", "q_stats", "sched_len", "K", "tau_theta", "out_tokens", "accepted_len", "p_tok"):
        assert np.array_equal(s[k], g[k]), k
    requests = list(range(R))
    rep = compare(cfg, s, oracle_pool.oracle_round(cfg, requests), requests)
    assert rep["positions"] > 0


def test_gated_separate_calls_full_size():
    """The same equality at DeepSeek scale (R = 128, gamma = 16, V = 129,280,
    rank 256), where the round verifies inside its drafting launch."""
    cfg = W.with_(W.CONFIGS["ds"], gated=True)
    inp = device_inputs(cfg)
    s = _separate_calls(cfg, inp)
    assert s["status"] == dspark.OK, dspark.status_string(s["status"])
    g = gpu_round(cfg, inp)
    for k in ("tokens", "q_tok", "q_stats", "sched_len", "K", "tau_theta", "out_tokens", "accepted_len", "p_tok"):
        assert np.array_equal(s[k], g[k]), k
