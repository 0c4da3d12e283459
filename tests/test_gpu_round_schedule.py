"""The round's schedule as the drafting launch computes it on the tensor-core
path: one extra CTA of that launch runs the whole prefix scheduler (survival
keys, a stable radix sort, the exact fixed-point scan and the mode's
admission rule) while the other CTAs sweep the vocabulary.

The confidences are drawn from a few values, 0 and 1 included, so that many
prefix survivals tie and the order of equal keys decides which candidates are
admitted; the cost tables are concave, a step or a cliff, from longer than
every candidate needs down to shorter than R. Each case checks the round's
schedule against the oracle's scheduler and against the library's standalone
scheduler (dspark_schedule), bit for bit; some also run the whole round
against the oracle. Then the edge cases: a non-finite confidence, a
non-finite cost-table entry, and more candidates than the scheduler CTA keeps
in shared memory (8,192: its sort then runs through the workspace).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import schedule as S
from oracle.round import run_round

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import compare, device_inputs, gpu_round
    from speculative_decoding_draft_seq_gb300 import dspark


def _table(kind, n_table, rng):
    b = np.arange(1, n_table + 1, dtype=np.float64)
    if kind == "concave":
        t = 100.0 / (1.0 + 0.002 * b) + rng.uniform(0.0, 0.01, n_table)
    elif kind == "step":
        t = np.where(b <= n_table // 2, 100.0, 60.0)
    else:  # flat with a cliff at 3/4
        t = np.where(b <= (3 * n_table) // 4, 80.0, 10.0)
    return t.astype(np.float32)


def _conf(R, gamma, rng):
    vals = np.array([0.0, 0.25, 0.5, 0.75, 1.0, 0.9, 0.9], dtype=np.float32)
    return vals[rng.integers(0, vals.size, size=(R, gamma))]


def _cfg(R, gamma, V, mode, n_table, gated=False, T=1.0):
    return W.Workload(f"round_sched_{R}_{gamma}", R=R, gamma=gamma, V=V, rank=64, dtype="bf16", T=T, mode=mode,
                      seed=4700 + R + gamma, base_sd=1.5, w_sd=0.05, target_sd=(0.45,), conf_law="decreasing",
                      table="concave", n_table=n_table, gated=gated)


def _tie_inputs(cfg, table):
    """Device inputs of `cfg` with tie-heavy confidences and a `table`-shaped
    cost table in place of the workload's own; also returns them on the host."""
    rng = np.random.default_rng(7100 + cfg.R * 13 + cfg.gamma * 5 + cfg.mode + cfg.n_table)
    conf, lag = _conf(cfg.R, cfg.gamma, rng), _conf(cfg.R, cfg.gamma, rng)
    sps = _table(table, cfg.n_table, rng)
    inp = device_inputs(cfg)
    dev = inp["base"].device
    inp["conf"] = torch.from_numpy(conf).to(dev)
    inp["conf_lag"] = torch.from_numpy(lag).to(dev) if cfg.mode == W.LAGGED else None
    inp["sps"] = torch.from_numpy(sps).to(dev)
    return inp, conf, (lag if cfg.mode == W.LAGGED else None), sps


def _standalone(inp, cfg):
    dev = inp["conf"].device
    L = torch.full((cfg.R,), -7, dtype=torch.int32, device=dev)
    K = torch.full((1,), -7, dtype=torch.int32, device=dev)
    tt = torch.full((2,), -7.0, dtype=torch.float64, device=dev)
    ws = dspark.new_workspace(cfg.R, cfg.gamma, 1, 1, dspark.FP32, cfg.n_table, dev)
    dspark.schedule(inp["conf"], inp["conf_lag"], inp["sps"], cfg.mode, L, K, tt, ws)
    assert dspark.device_status(ws) == dspark.OK
    return L.cpu().numpy(), int(K.item()), tt.cpu().numpy()


def _check_schedule(g, want, alone):
    np.testing.assert_array_equal(g["sched_len"], want["L"].astype(np.int32))
    assert int(g["K"][0]) == want["K"]
    assert g["tau_theta"][0] == want["tau"] and g["tau_theta"][1] == want["theta"]
    L, K, tt = alone
    np.testing.assert_array_equal(g["sched_len"], L)
    assert int(g["K"][0]) == K
    assert g["tau_theta"].tobytes() == tt.tobytes()


def _check_verified(g, gamma):
    L, A = g["sched_len"], g["accepted_len"]
    assert np.all((0 <= A) & (A <= L)) and np.all(L <= gamma)
    for r in range(L.size):
        assert np.array_equal(g["out_tokens"][r, :A[r]], g["tokens"][r, :A[r]])
        assert np.all(g["out_tokens"][r, A[r] + 1:] == -1)


MODES = [W.CAUSAL, W.LAGGED, W.ALL]
MODE_IDS = ["causal", "lagged", "all"]
# (R, gamma, V, n_table, table): 600 candidates with tables from longer than needed down to shorter than R,
# and 4,096 candidates
CASES = [(150, 4, 640, 760, "concave"), (150, 4, 640, 420, "step"), (150, 4, 640, 155, "cliff"),
         (150, 4, 640, 150, "step"), (150, 4, 640, 149, "concave"), (256, 16, 128, 4400, "step"),
         (256, 16, 128, 1800, "cliff")]


@pytest.mark.parametrize("R,gamma,V,n_table,table", CASES)
@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_round_schedule_with_ties(R, gamma, V, n_table, table, mode):
    cfg = _cfg(R, gamma, V, mode, n_table)
    inp, conf, lag, sps = _tie_inputs(cfg, table)
    g = gpu_round(cfg, inp)
    assert g["status"] == dspark.OK, dspark.status_string(g["status"])
    # drafting (with the schedule, the row statistics and the chains), residual sweep; in ALL mode the row
    # statistics and chains have their own launch
    assert g["launches"] == (3 if mode == W.ALL else 2), g["launches"]
    _check_schedule(g, S.schedule(conf, sps, mode=mode, conf_lagged=lag), _standalone(inp, cfg))
    _check_verified(g, gamma)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("gated", [False, True], ids=["markov", "gated"])
def test_round_with_tie_schedule_matches_oracle(mode, gated):
    """The whole round against the oracle when the schedule comes from the
    drafting launch and is full of ties: every request's drafted tokens,
    verification and bonus draw."""
    cfg = _cfg(150, 4, 640, mode, 420, gated=gated)
    inp, conf, lag, sps = _tie_inputs(cfg, "step")
    g = gpu_round(cfg, inp)
    assert g["launches"] == (3 if gated else 2) + (mode == W.ALL), g["launches"]
    o_in = W.oracle_inputs(cfg)
    o_in.update(conf=conf, conf_lag=lag, sps=sps)
    requests = list(range(cfg.R))
    rep = compare(cfg, g, run_round(o_in, requests=requests), requests)
    assert rep["positions"] > 0 and rep["bonus_compared"] > 0, rep


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_round_schedule_greedy(mode):
    cfg = _cfg(150, 4, 640, mode, 420, T=0.0)
    inp, conf, lag, sps = _tie_inputs(cfg, "concave")
    g = gpu_round(cfg, inp)
    assert g["status"] == dspark.OK and g["launches"] == (2 if mode == W.ALL else 1), (g["status"], g["launches"])
    _check_schedule(g, S.schedule(conf, sps, mode=mode, conf_lagged=lag), _standalone(inp, cfg))
    _check_verified(g, cfg.gamma)


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_round_schedule_nonfinite_confidence(mode):
    cfg = _cfg(150, 4, 640, mode, 420)
    inp, *_ = _tie_inputs(cfg, "step")
    inp["conf"][77, 2] = float("nan")
    assert gpu_round(cfg, inp)["status"] == dspark.ERR_NONFINITE
    if mode == W.LAGGED:  # the lagged confidences are checked as well
        inp, *_ = _tie_inputs(cfg, "step")
        inp["conf_lag"][3, 0] = float("inf")
        assert gpu_round(cfg, inp)["status"] == dspark.ERR_NONFINITE


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("where", [0, 151, 419], ids=["first", "middle", "last"])
def test_round_schedule_nonfinite_table(mode, where):
    """Any non-finite cost-table entry is an error, read or not (the
    scheduler checks the whole table)."""
    cfg = _cfg(150, 4, 640, mode, 420)
    inp, *_ = _tie_inputs(cfg, "step")
    inp["sps"][where] = float("nan") if where != 151 else float("-inf")
    assert gpu_round(cfg, inp)["status"] == dspark.ERR_NONFINITE


@pytest.mark.parametrize("R,gamma,n_table,table", [(600, 14, 8800, "concave"), (4096, 16, 69632, "step")],
                         ids=["8400", "65536"])
@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
def test_round_schedule_sort_in_workspace(mode, R, gamma, n_table, table):
    """8,400 candidates, more than the scheduler CTA's shared memory holds:
    its radix sort runs through the workspace's buffers, still inside the
    drafting launch; and the largest round the scheduler takes (65,536
    candidates, 4,096 requests in 32 M tiles)."""
    cfg = _cfg(R, gamma, 128, mode, n_table)
    inp, conf, lag, sps = _tie_inputs(cfg, table)
    g = gpu_round(cfg, inp)
    assert g["status"] == dspark.OK, dspark.status_string(g["status"])
    assert g["launches"] == (3 if mode == W.ALL else 2), g["launches"]
    _check_schedule(g, S.schedule(conf, sps, mode=mode, conf_lagged=lag), _standalone(inp, cfg))
    _check_verified(g, cfg.gamma)
