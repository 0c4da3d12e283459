"""GPU parity of the scheduler alone, against the oracle, on inputs with many
exact ties in the prefix survivals (confidences drawn from a few values,
including 0 and 1) -- the case where the order of equal keys decides which
candidates are admitted. Covers both device forms: the rank-and-admit pair
(R * gamma <= 4096) and the single-CTA radix sort (larger problems, up to the
entry point's maximum of 65,536 candidates).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import schedule as S

pytestmark = pytest.mark.gpu


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


CASES = [(40, 5, 260, "concave"), (128, 16, 2200, "step"), (256, 16, 4400, "cliff"),
         (300, 20, 6400, "concave"), (1, 1, 4, "step"), (7, 3, 9, "cliff"),
         # more than 8192 keys: the radix sort runs through the workspace (scheduler-stress size)
         (1024, 16, 17408, "step"), (1024, 16, 16384, "cliff"),
         # the largest problem the entry point takes, R * gamma = 65,536, in three shapes
         (4096, 16, 69632, "step"), (2048, 32, 65536, "cliff"), (65536, 1, 98304, "cliff")]


@pytest.mark.parametrize("R,gamma,n_table,table", CASES)
@pytest.mark.parametrize("mode", [S.CAUSAL, S.LAGGED, S.ALL])
def test_schedule_with_ties(R, gamma, n_table, table, mode):
    from speculative_decoding_draft_seq_gb300 import dspark
    rng = np.random.default_rng(7000 + R * 31 + gamma * 7 + mode)
    conf = _conf(R, gamma, rng)
    lag = _conf(R, gamma, rng)
    sps = _table(table, n_table, rng)
    want = S.schedule(conf, sps, mode=mode, conf_lagged=lag if mode == S.LAGGED else None)

    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    L = torch.full((R,), -7, dtype=torch.int32, device=dev)
    K = torch.full((1,), -7, dtype=torch.int32, device=dev)
    tt = torch.full((2,), -7.0, dtype=torch.float64, device=dev)
    ws = dspark.new_workspace(R, gamma, 1, 1, dspark.FP32, n_table, dev)
    dspark.schedule(t(conf), t(lag) if mode == S.LAGGED else None, t(sps), mode, L, K, tt, ws)
    assert dspark.device_status(ws) == dspark.OK
    np.testing.assert_array_equal(L.cpu().numpy(), want["L"].astype(np.int32))
    assert int(K.item()) == want["K"]
    got = tt.cpu().numpy()
    assert got[0] == want["tau"] and got[1] == want["theta"]
