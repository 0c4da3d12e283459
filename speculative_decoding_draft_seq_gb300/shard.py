"""Request-sharded rounds over several GPUs, one process per GPU.

Drafting and verification are independent per request, so each rank keeps
its own requests and runs them on its own GPU. The scheduler is global: it
ranks every request's candidates by prefix survival against one cost table
("DSpark: Aceleração da inferência de LLM com speculative decoding [pdf]"
(GeekNews), "Hardware-Aware Prefix Scheduler"), so its input -- the
confidences, R_local x gamma floats per rank -- is all-gathered, and every
rank runs the same deterministic schedule over the whole batch and keeps the
lengths of its own requests. That all-gather is the only exchange of a round.

Host-side logic only; the schedule itself is a callable (the library's
scheduler on the GPU, `round_step` below).
"""

import torch
import torch.distributed as dist


def request_range(R_total, world, rank):
    """[start, stop) of rank's contiguous share of R_total requests (sizes
    differ by at most one, lower ranks first)."""
    base, extra = divmod(R_total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def gather_rows(t_local, group=None):
    """All-gather equal-sized row blocks of every rank, in rank order."""
    world = dist.get_world_size(group)
    parts = [torch.empty_like(t_local) for _ in range(world)]
    dist.all_gather(parts, t_local.contiguous(), group=group)
    return torch.cat(parts, 0)


def sharded_schedule(conf_local, conf_lagged_local, schedule_fn, group=None):
    """Global schedule over every rank's requests; returns (local lengths, K,
    tau_theta). `schedule_fn(conf, conf_lagged) -> (L [R_total], K, tau_theta)`
    must be deterministic, so every rank computes the same result. Each rank
    holds the same number of requests."""
    rank = dist.get_rank(group)
    conf = gather_rows(conf_local, group)
    lag = None if conf_lagged_local is None else gather_rows(conf_lagged_local, group)
    L, K, tau_theta = schedule_fn(conf, lag)
    n = conf_local.shape[0]
    return L[rank * n:(rank + 1) * n], K, tau_theta


class ShardedRound:
    """One round of this rank's requests with the global schedule: draft on
    the local GPU, all-gather of the confidences, the library's scheduler over
    the whole batch (every rank the same), verification of the local requests
    with their scheduled lengths."""

    def __init__(self, dspark, R_local, gamma, V, rank_dim, dtype, n_table_global, device, group=None):
        self.dspark = dspark
        self.group = group
        world = dist.get_world_size(group)
        self.R_total = R_local * world
        self.ws = dspark.new_workspace(R_local, gamma, V, rank_dim, dtype, 1, device)
        self.ws_sched = dspark.new_workspace(self.R_total, gamma, 1, rank_dim, dtype, n_table_global, device)
        self.L_all = torch.empty(self.R_total, dtype=torch.int32, device=device)
        self.K = torch.empty(1, dtype=torch.int32, device=device)
        self.tau_theta = torch.empty(2, dtype=torch.float64, device=device)

    def _schedule(self, sps, mode):
        def fn(conf, lag):
            self.dspark.schedule(conf, lag, sps, mode, self.L_all, self.K, self.tau_theta, self.ws_sched)
            return self.L_all, self.K, self.tau_theta
        return fn

    def __call__(self, inp, out):
        d = self.dspark
        d.draft_sequential(inp["base"], inp["anchor"], inp["W1"], inp["W2"], inp["T"], inp["seed"], out.tokens,
                           out.q_tok, out.q_stats, self.ws)
        L, K, tt = sharded_schedule(inp["conf"], inp["conf_lag"], self._schedule(inp["sps"], inp["mode"]), self.group)
        out.sched_len.copy_(L)
        out.K.copy_(K)
        out.tau_theta.copy_(tt)
        d.verify(inp["target"], inp["base"], inp["anchor"], inp["W1"], inp["W2"], out.tokens, out.q_tok, out.q_stats,
                 out.sched_len, inp["T"], inp["seed"], out.out_tokens, out.accepted_len, out.p_tok, self.ws)
