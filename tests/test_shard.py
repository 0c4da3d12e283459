"""The request-sharded round's host logic on CPU with `gloo`, world size 2:
request ranges, the all-gather of confidences, and the global schedule each
rank computes (the oracle's scheduler stands in for the library's, which
needs a GPU): every rank's lengths equal the single-process schedule of the
whole batch restricted to its requests, and K agrees across ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _conf(seed, R, gamma):
    rng = np.random.default_rng(seed)
    return rng.beta(8, 2, size=(R, gamma)).astype(np.float32)


def _worker(rank, world, port, R_local, gamma, mode, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from oracle.schedule import schedule as oracle_schedule
    from speculative_decoding_draft_seq_gb300 import shard
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        R_total = R_local * world
        full = _conf(11, R_total, gamma)
        lag_full = _conf(12, R_total, gamma) if mode == 1 else None
        start, stop = shard.request_range(R_total, world, rank)
        local = torch.from_numpy(full[start:stop])
        lag_local = None if lag_full is None else torch.from_numpy(lag_full[start:stop])
        sps = (1.0 / (1.0 + 2e-3 * np.arange(1, R_total * (gamma + 1) + 1))).astype(np.float32)

        def fn(conf, lag):
            s = oracle_schedule(conf.numpy(), sps, mode, None if lag is None else lag.numpy())
            return torch.from_numpy(np.asarray(s["L"], dtype=np.int32)), int(s["K"]), (s["tau"], s["theta"])

        L_local, K, tt = shard.sharded_schedule(local, lag_local, fn)
        ref = oracle_schedule(full, sps, mode, lag_full)
        ok = np.array_equal(L_local.numpy(), np.asarray(ref["L"], dtype=np.int32)[start:stop]) and K == ref["K"]
        Ks = [None] * world
        dist.all_gather_object(Ks, K)
        q.put((rank, ok, len(set(Ks)) == 1, (start, stop)))
    finally:
        dist.destroy_process_group()


def test_request_range_covers_every_request_once():
    from speculative_decoding_draft_seq_gb300 import shard
    for R in (1, 7, 128, 1000):
        for world in (1, 2, 3, 8):
            spans = [shard.request_range(R, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == R
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("mode", [0, 1])
def test_sharded_schedule_gloo_world2(mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, 24, 5, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] for r in res), res
    assert all(r[2] for r in res)
    assert res[0][3] == (0, 24) and res[1][3] == (24, 48)
