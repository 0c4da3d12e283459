"""Seeded synthetic inputs for one DSpark round, shared by the tests, the
benchmark and the smoke entry point.

This module holds random numbers only -- none of the method's arithmetic. The
pages' workloads (Qwen3 / DeepSeek-V4 drafters and targets on math, code and
chat suites) are not available, so these tensors stand in for them with the
shapes, value distributions and structure the pages describe:

  * base logits of the parallel backbone ([GN] "Etapa paralela"), Zipf(1.1)
    rank-shaped per request plus Gaussian noise;
  * low-rank Markov factors W1 [V, rank], W2 [rank, V] ([GN] "Head de Markov");
  * target logits = base + Gaussian noise whose scale sets the acceptance
    length (the pages report 5.1-5.6 accepted tokens on math/code and 3.1-3.6
    on chat at a 7-token window, [JD] and [GN] §"Resultados principais");
  * per-position confidences, and a steps-per-second cost table SPS(B)
    ([GN] "Hardware-Aware Prefix Scheduler", §"Aplicação prática").

Bit-identical on CPU (numpy) and GPU (torch): the large logit tensors are
built from a counter-based 32-bit integer hash of each element's flat index,
mapped through a 65536-entry Gaussian quantile table and a Zipf rank table that
are computed once per process; the remaining float steps are single float32
multiplies and adds, and bf16 rounding is done with integer operations. So the
oracle can regenerate just the requests it checks while the device builds the
full tensors directly in HBM. Small tensors (anchors, confidences, tables,
rank permutations) come from numpy PCG64 streams and are copied to the device.
"""

from dataclasses import dataclass, replace
import math
import statistics

import numpy as np

M32 = 0xFFFFFFFF
_MUL_A = 0x7FEB352D  # odd multipliers below 2**31: products stay below 2**63
_MUL_B = 0x2C1B3C6D

# Tensor stream salts.
S_BASE, S_EXTRA, S_TARGET, S_W1, S_W2 = 0x1B873593, 0x5BD1E995, 0x27D4EB2F, 0x165667B1, 0x61C88647
S_GATE = 0x3C6EF372
S_HIDDEN, S_LMHEAD = 0x7A4E2B19, 0x1F83D9AB

CAUSAL, LAGGED, ALL = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    gamma: int
    V: int
    rank: int
    dtype: str                  # "bf16" or "fp32"
    T: float
    mode: int
    seed: int                   # seed of every generator stream of this workload
    philox_seed: int = 0        # seed of the round's uniforms
    base_sd: float = 1.5
    zipf: float = 1.1           # 0 disables the rank-shaped term
    w_sd: float = 0.02
    target_sd: tuple = (0.5,)   # per request group (cycled over equal halves)
    conf_law: str = "decreasing"
    table: str = "concave"
    n_table: int = 0
    gated: bool = False         # the recurrent (gated) head: gate values [V, rank] in [gate_lo, 1]
    gate_lo: float = 0.25
    notes: str = ""

    @property
    def positions(self):
        return self.R * self.gamma


# Target-noise scales, chosen by bisection with oracle/calibrate_sigma.py so
# that the mean accepted length per round (accepted draft tokens + 1) at a
# 7-token block, scheduler off, temperature 1, is about 5.0 (DeepSeek-scale),
# 5.5 (structured half of the mixed workload) and 3.3 (chat half).
DS_TARGET_SD = 0.429
STRUCTURED_TARGET_SD = 0.341
CHAT_TARGET_SD = 0.802

CONFIGS = {
    "tiny": Workload("tiny", R=4, gamma=4, V=64, rank=8, dtype="fp32", T=1.0, mode=CAUSAL,
                     seed=1001, base_sd=1.5, zipf=0.0, w_sd=0.3, target_sd=(0.5,),
                     conf_law="uniform", table="linear", n_table=16),
    "small": Workload("small", R=32, gamma=8, V=32000, rank=256, dtype="bf16", T=0.8,
                      mode=CAUSAL, seed=1002, base_sd=2.0, w_sd=0.02, target_sd=(0.7,),
                      conf_law="beta82", table="concave", n_table=512),
    "ds": Workload("ds", R=128, gamma=16, V=129280, rank=256, dtype="bf16", T=1.0,
                   mode=CAUSAL, seed=1003, base_sd=1.5, w_sd=0.02, target_sd=(DS_TARGET_SD,),
                   conf_law="decreasing", table="concave", n_table=128 * 17),
    "stress": Workload("stress", R=1024, gamma=16, V=129280, rank=256, dtype="bf16", T=1.0,
                       mode=LAGGED, seed=1004, base_sd=1.5, w_sd=0.02,
                       target_sd=(DS_TARGET_SD,), conf_law="beta_mixed", table="step",
                       n_table=16384),
    "mixed": Workload("mixed", R=256, gamma=16, V=129280, rank=256, dtype="bf16", T=1.0,
                      mode=CAUSAL, seed=1005, base_sd=1.5, w_sd=0.02,
                      target_sd=(STRUCTURED_TARGET_SD, CHAT_TARGET_SD),
                      conf_law="two_domain", table="concave", n_table=256 * 17),
}


def with_(cfg, **kw):
    """Copy of a workload with some fields replaced (e.g. T=0.0, R=8)."""
    return replace(cfg, **kw)


# ----------------------------------------------------------------------------
# tables computed once per process (identical for the numpy and torch paths)

_NORM = None
_ZIPF = {}


def norm_table():
    """Gaussian quantiles at (i + 1/2) / 65536, float32 [65536]."""
    global _NORM
    if _NORM is None:
        nd = statistics.NormalDist()
        _NORM = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)],
                         dtype=np.float32)
    return _NORM


def zipf_table(V, s):
    """-s * ln(1 + rank) for rank 0..V-1, float32 (the rank-shaped log-prob)."""
    key = (V, s)
    if key not in _ZIPF:
        _ZIPF[key] = (-s * np.log1p(np.arange(V, dtype=np.float64))).astype(np.float32)
    return _ZIPF[key]


def _salt(cfg, stream):
    return (stream * 0x9E3779B1 + cfg.seed * 0x85EBCA6B) & M32


def _mix32_np(x):
    x = x ^ (x >> 16)
    x = (x * _MUL_A) & M32
    x = x ^ (x >> 15)
    x = (x * _MUL_B) & M32
    x = x ^ (x >> 16)
    return x


def _hash_np(idx, salt):
    """32-bit hash of flat indices (numpy uint64 arrays holding 32-bit values)."""
    return _mix32_np(_mix32_np((idx & M32) ^ salt) ^ ((salt * 0x2545F491) & M32))


def _bf16_bits_np(f32):
    b = f32.view(np.uint32).astype(np.uint64)
    return (((b + 0x7FFF + ((b >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def _bf16_value_np(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def rank_permutation(cfg, r):
    """pi_r: a random rank (Zipf position) for every token id of request r."""
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 7, r]))
    return rng.permutation(cfg.V).astype(np.int64)


def target_sd_of(cfg, r):
    groups = len(cfg.target_sd)
    return cfg.target_sd[min(groups - 1, r * groups // cfg.R)]


# ----------------------------------------------------------------------------
# numpy path: rows of chosen requests (used by the oracle side and small tests)

def _noise_np(cfg, stream, flat_idx, sd):
    h = _hash_np(flat_idx.astype(np.uint64), _salt(cfg, stream))
    return np.float32(sd) * norm_table()[(h >> 16).astype(np.int64)]


def _finish_np(cfg, f32):
    if cfg.dtype == "bf16":
        bits = _bf16_bits_np(f32)
        return bits, _bf16_value_np(bits)
    return f32, f32


def logits_rows_np(cfg, requests):
    """base [n, gamma, V] and target [n, gamma+1, V] for the given requests.

    Returned as stored on the device: uint16 bf16 bit patterns for bf16
    workloads, float32 otherwise.
    """
    g, V = cfg.gamma, cfg.V
    zt = zipf_table(V, cfg.zipf) if cfg.zipf else None
    v = np.arange(V, dtype=np.uint64)
    base_out, tgt_out = [], []
    for r in requests:
        shape = zt[rank_permutation(cfg, r)] if zt is not None else np.zeros(V, np.float32)
        sd_t = target_sd_of(cfg, r)
        b_rows, t_rows = [], []
        base_vals = []
        for k in range(g + 1):
            if k < g:
                idx = np.uint64((r * g + k) * V) + v
                raw = shape + _noise_np(cfg, S_BASE, idx, cfg.base_sd)
            else:
                idx = np.uint64(r * V) + v
                raw = shape + _noise_np(cfg, S_EXTRA, idx, cfg.base_sd)
            stored, value = _finish_np(cfg, raw.astype(np.float32))
            if k < g:
                b_rows.append(stored)
            base_vals.append(value)
        for k in range(g + 1):
            idx = np.uint64((r * (g + 1) + k) * V) + v
            raw = base_vals[k] + _noise_np(cfg, S_TARGET, idx, sd_t)
            t_rows.append(_finish_np(cfg, raw.astype(np.float32))[0])
        base_out.append(np.stack(b_rows))
        tgt_out.append(np.stack(t_rows))
    return np.stack(base_out), np.stack(tgt_out)


def weights_np(cfg):
    """W1 [V, rank], W2 [rank, V] as stored (bf16 bits or float32)."""
    n = cfg.V * cfg.rank
    idx = np.arange(n, dtype=np.uint64)
    w1 = _noise_np(cfg, S_W1, idx, cfg.w_sd).reshape(cfg.V, cfg.rank)
    w2 = _noise_np(cfg, S_W2, idx, cfg.w_sd).reshape(cfg.rank, cfg.V)
    return _finish_np(cfg, w1)[0], _finish_np(cfg, w2)[0]


def _gate_f32_np(cfg):
    """Gate values lo + (1 - lo) u, u = 24 hash bits * 2^-24 (exact in float32),
    one float32 multiply and one add."""
    idx = np.arange(cfg.V * cfg.rank, dtype=np.uint64)
    h = _hash_np(idx, _salt(cfg, S_GATE))
    u = (h >> 8).astype(np.float32) * np.float32(2.0 ** -24)
    return (np.float32(cfg.gate_lo) + np.float32(1.0 - cfg.gate_lo) * u).astype(np.float32).reshape(cfg.V, cfg.rank)


def gate_np(cfg):
    """Gate values [V, rank] of the gated head, as stored (bf16 bits or float32)."""
    return _finish_np(cfg, _gate_f32_np(cfg))[0]


# ----------------------------------------------------------------------------
# small host tensors (PCG64)

def anchors(cfg):
    rng = np.random.Generator(np.random.PCG64([cfg.seed, 1]))
    return rng.integers(0, cfg.V, size=cfg.R).astype(np.int32)


def _conf_draw(cfg, stream):
    rng = np.random.Generator(np.random.PCG64([cfg.seed, stream]))
    R, g = cfg.R, cfg.gamma
    if cfg.conf_law == "uniform":
        c = rng.uniform(0.5, 1.0, size=(R, g))
    elif cfg.conf_law == "beta82":
        c = rng.beta(8.0, 2.0, size=(R, g))
    elif cfg.conf_law in ("decreasing", "two_domain"):
        if cfg.conf_law == "two_domain":
            start = np.where(np.arange(R) < R // 2, 0.95, 0.80)[:, None]
        else:
            start = np.full((R, 1), 0.92)
        logit0 = np.log(start / (1.0 - start))
        z = logit0 - 0.15 * np.arange(g)[None, :] + rng.normal(0.0, 0.3, size=(R, g))
        c = 1.0 / (1.0 + np.exp(-z))
    elif cfg.conf_law == "beta_mixed":
        mu = rng.uniform(0.4, 0.95, size=(R, 1))
        c = rng.beta(mu * 10.0, (1.0 - mu) * 10.0, size=(R, g))
    else:
        raise ValueError(cfg.conf_law)
    return c.astype(np.float32)


def confidences(cfg):
    """Current confidences c [R, gamma] float32."""
    return _conf_draw(cfg, 2)


def lagged_confidences(cfg):
    """Confidences 'from two rounds earlier': an independent draw of the same law."""
    return _conf_draw(cfg, 3)


def sps_table(cfg):
    """SPS(B) for B = 1..n_table, float32 (entry i <-> B = i + 1)."""
    n = cfg.n_table
    B = np.arange(1, n + 1, dtype=np.float64)
    if cfg.table == "linear":
        s = 1.0 - (B - 1.0) / 32.0
    elif cfg.table == "concave":
        s = 1.0 / (1.0 + 2e-3 * B + 4e-6 * B * B)
    elif cfg.table == "step":
        s = 1.0 / (1.0 + 2e-3 * 64.0 * np.ceil(B / 64.0))
        s = np.where(B > 8192, 0.8 * s, s)
    else:
        raise ValueError(cfg.table)
    return s.astype(np.float32)


def host_inputs(cfg):
    """Everything except the large logit/weight tensors, as numpy arrays."""
    return dict(anchor=anchors(cfg), conf=confidences(cfg),
                conf_lag=lagged_confidences(cfg) if cfg.mode == LAGGED else None,
                sps=sps_table(cfg), T=cfg.T, seed=cfg.philox_seed, mode=cfg.mode)


def oracle_inputs(cfg, requests=None):
    """Full numpy input dict for the oracle; logits only for `requests`
    (all requests when None; rows of other requests are left absent)."""
    reqs = list(range(cfg.R)) if requests is None else list(requests)
    base, tgt = logits_rows_np(cfg, reqs)
    W1, W2 = weights_np(cfg)
    d = host_inputs(cfg)
    d.update(W1=W1, W2=W2)
    if cfg.gated:
        d["gate"] = gate_np(cfg)
    d["base"] = {r: base[i] for i, r in enumerate(reqs)}
    d["target"] = {r: tgt[i] for i, r in enumerate(reqs)}
    return d


# ----------------------------------------------------------------------------
# torch path: the same tensors built directly on a device

def _torch():
    import torch
    return torch


def _mix32_t(x):
    x = x ^ (x >> 16)
    x = (x * _MUL_A) & M32
    x = x ^ (x >> 15)
    x = (x * _MUL_B) & M32
    x = x ^ (x >> 16)
    return x


def _hash_t(idx, salt):
    return _mix32_t(_mix32_t((idx & M32) ^ salt) ^ ((salt * 0x2545F491) & M32))


def _bf16_t(f32):
    torch = _torch()
    b = f32.view(torch.int32).to(torch.int64) & M32
    bits = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) & 0xFFFF
    signed = torch.where(bits >= 32768, bits - 65536, bits).to(torch.int16)
    return signed.view(torch.bfloat16)


def _noise_t(cfg, stream, flat_idx, sd, table):
    torch = _torch()
    h = _hash_t(flat_idx, _salt(cfg, stream))
    return table[h >> 16] * torch.tensor(sd, dtype=torch.float32, device=flat_idx.device)


def _finish_t(cfg, f32):
    if cfg.dtype == "bf16":
        return _bf16_t(f32)
    return f32


def logits_device(cfg, device, requests_per_chunk=8):
    """base [R, gamma, V] and target [R, gamma+1, V] on `device`
    (torch.bfloat16 for bf16 workloads, torch.float32 otherwise)."""
    torch = _torch()
    g, V, R = cfg.gamma, cfg.V, cfg.R
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    base = torch.empty((R, g, V), dtype=dt, device=device)
    tgt = torch.empty((R, g + 1, V), dtype=dt, device=device)
    table = torch.from_numpy(norm_table()).to(device)
    zt = torch.from_numpy(zipf_table(V, cfg.zipf)).to(device) if cfg.zipf else None
    v = torch.arange(V, dtype=torch.int64, device=device)
    for r0 in range(0, R, requests_per_chunk):
        rs = list(range(r0, min(R, r0 + requests_per_chunk)))
        for r in rs:
            if zt is not None:
                perm = torch.from_numpy(rank_permutation(cfg, r)).to(device)
                shape = zt[perm]
            else:
                shape = torch.zeros(V, dtype=torch.float32, device=device)
            kk = torch.arange(g, dtype=torch.int64, device=device)[:, None]
            idx = (r * g + kk) * V + v[None, :]
            raw = shape[None, :] + _noise_t(cfg, S_BASE, idx, cfg.base_sd, table)
            b = _finish_t(cfg, raw)
            base[r] = b
            raw_x = shape + _noise_t(cfg, S_EXTRA, r * V + v, cfg.base_sd, table)
            bx = _finish_t(cfg, raw_x)
            bvals = torch.cat([b.float(), bx.float()[None, :]], 0)
            kt = torch.arange(g + 1, dtype=torch.int64, device=device)[:, None]
            idx_t = (r * (g + 1) + kt) * V + v[None, :]
            raw_t = bvals + _noise_t(cfg, S_TARGET, idx_t, target_sd_of(cfg, r), table)
            tgt[r] = _finish_t(cfg, raw_t)
    return base, tgt


def weights_device(cfg, device):
    torch = _torch()
    table = torch.from_numpy(norm_table()).to(device)
    n = cfg.V * cfg.rank
    idx = torch.arange(n, dtype=torch.int64, device=device)
    w1 = _finish_t(cfg, _noise_t(cfg, S_W1, idx, cfg.w_sd, table)).reshape(cfg.V, cfg.rank)
    w2 = _finish_t(cfg, _noise_t(cfg, S_W2, idx, cfg.w_sd, table)).reshape(cfg.rank, cfg.V)
    return w1.contiguous(), w2.contiguous()


def hidden_np(cfg, d, rows):
    """Final hidden states of block positions `rows` (flat r * gamma + k), [len(rows), d]
    bf16 bits: N(0, 1)."""
    rows = np.asarray(rows, dtype=np.uint64)
    idx = rows[:, None] * np.uint64(d) + np.arange(d, dtype=np.uint64)[None, :]
    return _bf16_bits_np(_noise_np(cfg, S_HIDDEN, idx, 1.0))


def lm_head_np(cfg, d, cols=None):
    """LM head [d, V] (or its columns `cols`) as bf16 bits: N(0, (1.5 / sqrt(d))^2), so
    that the logits have the spread of the base logits."""
    cols = np.arange(cfg.V, dtype=np.uint64) if cols is None else np.asarray(cols, dtype=np.uint64)
    idx = np.arange(d, dtype=np.uint64)[:, None] * np.uint64(cfg.V) + cols[None, :]
    return _bf16_bits_np(_noise_np(cfg, S_LMHEAD, idx, 1.5 / math.sqrt(d)))


def hidden_device(cfg, d, device):
    torch = _torch()
    table = torch.from_numpy(norm_table()).to(device)
    idx = torch.arange(cfg.R * cfg.gamma * d, dtype=torch.int64, device=device)
    return _bf16_t(_noise_t(cfg, S_HIDDEN, idx, 1.0, table)).reshape(cfg.R, cfg.gamma, d).contiguous()


def lm_head_device(cfg, d, device, rows_per_chunk=512):
    torch = _torch()
    table = torch.from_numpy(norm_table()).to(device)
    out = torch.empty((d, cfg.V), dtype=torch.bfloat16, device=device)
    for i0 in range(0, d, rows_per_chunk):
        i1 = min(d, i0 + rows_per_chunk)
        idx = (torch.arange(i0, i1, dtype=torch.int64, device=device)[:, None] * cfg.V +
               torch.arange(cfg.V, dtype=torch.int64, device=device)[None, :])
        out[i0:i1] = _bf16_t(_noise_t(cfg, S_LMHEAD, idx, 1.5 / math.sqrt(d), table))
    return out


def gate_device(cfg, device):
    torch = _torch()
    idx = torch.arange(cfg.V * cfg.rank, dtype=torch.int64, device=device)
    h = _hash_t(idx, _salt(cfg, S_GATE))
    u = (h >> 8).to(torch.float32) * torch.tensor(2.0 ** -24, dtype=torch.float32, device=device)
    lo = torch.tensor(cfg.gate_lo, dtype=torch.float32, device=device)
    one_m = torch.tensor(1.0 - cfg.gate_lo, dtype=torch.float32, device=device)
    return _finish_t(cfg, lo + one_m * u).reshape(cfg.V, cfg.rank).contiguous()


def device_inputs(cfg, device="cuda"):
    """Every input of one round as device tensors (torch), for the library."""
    torch = _torch()
    base, target = logits_device(cfg, device)
    W1, W2 = weights_device(cfg, device)
    h = host_inputs(cfg)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return dict(base=base, target=target, W1=W1, W2=W2, anchor=t(h["anchor"]), conf=t(h["conf"]),
                conf_lag=t(h["conf_lag"]), sps=t(h["sps"]), T=cfg.T, seed=cfg.philox_seed,
                mode=cfg.mode, gate=gate_device(cfg, device) if cfg.gated else None)


def device_inputs_from_host(cfg, device="cuda"):
    """The same inputs as device_inputs, generated with numpy on the host and
    copied to the device with one copy per tensor (no generator kernels run on
    the device). Meant for small workloads: every request's rows are built on
    the host."""
    torch = _torch()
    base, tgt = logits_rows_np(cfg, range(cfg.R))
    W1, W2 = weights_np(cfg)
    h = host_inputs(cfg)

    def dev(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:  # bf16 bit patterns
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(a).to(device)

    return dict(base=dev(base), target=dev(tgt), W1=dev(W1), W2=dev(W2), anchor=dev(h["anchor"]),
                conf=dev(h["conf"]), conf_lag=dev(h["conf_lag"]), sps=dev(h["sps"]), T=cfg.T,
                seed=cfg.philox_seed, mode=cfg.mode, gate=dev(gate_np(cfg)) if cfg.gated else None)
