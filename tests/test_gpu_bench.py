"""The benchmark on the GPU at the small-vocabulary workload: one JSON line
with every field of the contract, and round statistics that are those of the
timed round (equal to a round of the library on the same inputs, which the
parity tests hold to the oracle)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads as W
from gpu_harness import gpu_round

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_and_round_stats_small():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--config", "small", "--steps", "20",
                          "--warmup", "3", "--no-cpu-baseline"], capture_output=True, text=True, cwd=ROOT,
                         timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches", "round_stats"):
        assert k in d, k
    assert d["steps"] == 20 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["value"] > 0
    assert d["gpu_launches"] > 0
    assert d["roofline"]["bound"] == "hbm" and 0 < d["roofline"]["frac"] < 1.5
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0

    g = gpu_round(W.CONFIGS["small"])
    L, A = np.asarray(g["sched_len"]), np.asarray(g["accepted_len"])
    rs = d["round_stats"]
    assert rs["scheduled_positions"] == int(L.sum())
    assert rs["accepted"] == int(A.sum())
    assert rs["emitted"] == int((A + 1).sum())
