"""The request-sharded round (speculative_decoding_draft_seq_gb300/shard.py)
on one GPU: a process group of one rank (NCCL), so the all-gather of the
confidences, the global schedule on the library's scheduler and the local
verification all run through their real code path. The result must equal the
oracle's round and, bit for bit, the single-GPU dspark_round."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_harness import compare, device_inputs, gpu_round, oracle_round
    from speculative_decoding_draft_seq_gb300 import dspark, shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


SHARD_CFG = W.Workload("shard_tc", R=150, gamma=4, V=3000, rank=64, dtype="bf16", T=1.0, mode=W.CAUSAL, seed=2103,
                       base_sd=1.5, w_sd=0.05, target_sd=(0.45,), conf_law="decreasing", table="concave",
                       n_table=150 * 5)


@pytest.fixture(scope="module")
def one_rank_group():
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    yield
    dist.destroy_process_group()


@pytest.mark.parametrize("cfg", [SHARD_CFG, W.with_(SHARD_CFG, mode=W.LAGGED, conf_law="beta_mixed"),
                                 W.with_(SHARD_CFG, T=0.0)], ids=["causal", "lagged", "greedy"])
def test_sharded_round_world1(one_rank_group, cfg):
    inp = device_inputs(cfg)
    assert shard.request_range(cfg.R, 1, 0) == (0, cfg.R)
    sr = shard.ShardedRound(dspark, cfg.R, cfg.gamma, cfg.V, cfg.rank, dspark.BF16, cfg.n_table, "cuda")
    out = dspark.RoundOutputs(cfg.R, cfg.gamma)
    sr(inp, out)
    g = out.host()
    g["status"] = max(dspark.device_status(sr.ws), dspark.device_status(sr.ws_sched))
    requests = list(range(cfg.R))
    compare(cfg, g, oracle_round(cfg, requests), requests)
    ref = gpu_round(cfg, inp)
    for k in ("tokens", "q_tok", "q_stats", "sched_len", "K", "tau_theta", "out_tokens", "accepted_len", "p_tok"):
        assert np.array_equal(g[k], ref[k]), k
