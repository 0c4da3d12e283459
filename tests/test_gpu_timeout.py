"""Failure detection on the device without a fault: a bounded wait of each
kind the kernels use (the grid barrier, an mbarrier wait, the poll on a
counter another CTA advances) is made to run out
on a condition nothing meets; it records DSPARK_ERR_TIMEOUT in the status
word, the kernel returns, and the context keeps working (a round afterwards
is correct)."""
import time

import pytest

torch = pytest.importorskip("torch")

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import compare, gpu_round, oracle_round
    from speculative_decoding_draft_seq_gb300 import dspark


@pytest.mark.parametrize("which", [0, 1, 2], ids=["grid_barrier", "mbarrier", "counter_poll"])
def test_bounded_wait_times_out_and_the_context_stays_usable(which):
    ws = dspark.new_workspace(4, 4, 64, 8, dspark.FP32, 16, "cuda")
    t0 = time.time()
    dspark.wait_selftest(which, ws)
    st = dspark.device_status(ws)
    elapsed = time.time() - t0
    assert st == dspark.ERR_TIMEOUT, dspark.status_string(st)
    assert elapsed < 60
    cfg = W.CONFIGS["tiny"]
    g = gpu_round(cfg)
    assert g["status"] == dspark.OK
    compare(cfg, g, oracle_round(cfg, list(range(cfg.R))), list(range(cfg.R)))
