"""GPU parity of the base logits from hidden states (dspark_lm_head) against
the oracle ([GN] "Etapa paralela", "Comunicação de estados ocultos").

The device accumulates the d products in float32 on the tensor cores and
rounds once to bf16; the oracle rounds the float64 sum (exact to far below a
bf16 step). The float32 sum's error grows like a random walk over the
accumulation steps, so every element must satisfy
    |gpu - exact| <= half a bf16 step + sqrt(d) * 2^-24 * sum_i |h_i lm_i|
(a wrong index, operand layout or tile offset gives errors of the order of
the logits themselves). Where that slack is below a quarter of half a bf16
step (most logits of magnitude 0.5 and more), the rounded values must equal
the oracle's except for the rare sums that fall within float32 error of a
rounding midpoint: fewer than 1 in 100 such elements may differ, and only by
one bf16 step."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads as W
from oracle import lm_head as LH
from oracle.draft import decode, draft_request

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from speculative_decoding_draft_seq_gb300 import dspark


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _ulp_half(x):
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 0.5 * 2.0 ** (np.floor(np.log2(a)) - 7)


def check_logits(g_bits, H_bits, LM_bits):
    d = H_bits.shape[1]
    exact = LH.lm_head_exact(H_bits, LM_bits)
    ref = LH.round_bf16_bits(exact)
    slack = np.sqrt(d) * 2.0 ** -24 * LH.abs_products(H_bits, LM_bits)
    g = LH.decode_bf16(g_bits)
    assert np.all(np.abs(g - exact) <= _ulp_half(exact) * (1 + 1e-12) + slack)
    mis = g_bits != ref
    big = slack < 0.25 * _ulp_half(exact)  # the well-conditioned elements
    assert big.sum() >= exact.size // 4
    mb = mis & big
    assert mb.sum() <= max(1, big.sum() // 100), (int(mb.sum()), int(big.sum()))
    if mb.any():  # one bf16 step apart
        gm, r = g[mb], LH.decode_bf16(ref[mb])
        assert np.all(np.abs(gm - r) <= 2 * _ulp_half(np.maximum(np.abs(gm), np.abs(r))) * (1 + 1e-12))
    return int(mis.sum())


def _run(cfg, d, dev="cuda"):
    H = W.hidden_device(cfg, d, dev)
    LM = W.lm_head_device(cfg, d, dev)
    out = torch.empty((cfg.R, cfg.gamma, cfg.V), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    dspark.lm_head(H, LM, out, ws)
    assert dspark.device_status(ws) == dspark.OK
    return H, LM, out


@pytest.mark.parametrize("M,d,V", [
    (1, 64, 64),        # one row, one K step, one column box
    (256, 64, 64),      # one full 256-row tile (both 128-row halves), one column box
    (129, 128, 128),    # the second half of the tile holds a single row
    (200, 512, 1000),   # a partial row tile and a partial last column box
    (5, 64, 72),        # fewer rows than a tile, two column boxes
    (128, 136, 256),    # a K tail of 8
    (520, 192, 320),    # three row tiles, the last with an empty second half
    (300, 7168, 512),   # the DeepSeek hidden size; the second row tile is partial
])
def test_lm_head_matches_oracle(M, d, V):
    cfg = W.Workload(f"lm_{M}_{d}_{V}", R=M, gamma=1, V=V, rank=64, dtype="bf16", T=1.0, mode=W.CAUSAL,
                     seed=6000 + M + d + V)
    H, LM, out = _run(cfg, d)
    H_bits = W.hidden_np(cfg, d, range(M))
    LM_bits = W.lm_head_np(cfg, d)
    assert np.array_equal(_bits(H).reshape(M, d), H_bits)  # the generator agrees with itself
    check_logits(_bits(out).reshape(M, V), H_bits, LM_bits)


def test_lm_head_full_size_sampled():
    """DeepSeek scale: M = 128 x 16 positions, d = 7168, V = 129,280; rows and
    columns sampled across every tile position."""
    cfg = W.with_(W.CONFIGS["ds"])
    d = 7168
    H, LM, out = _run(cfg, d)
    rows = np.array([0, 127, 128, 1000, 2047])
    rng = np.random.default_rng(0)
    cols = np.unique(np.concatenate([rng.choice(cfg.V, 3000, replace=False), np.arange(cfg.V - 300, cfg.V),
                                     np.arange(0, 300)]))
    H_bits = W.hidden_np(cfg, d, rows)
    LM_bits = W.lm_head_np(cfg, d, cols)
    g = _bits(out).reshape(-1, cfg.V)[rows][:, cols]
    check_logits(g, H_bits, LM_bits)


def test_lm_head_argument_errors():
    dev = "cuda"
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    H = torch.zeros((4, 32), dtype=torch.bfloat16, device=dev)
    LM = torch.zeros((32, 64), dtype=torch.bfloat16, device=dev)
    out = torch.empty((4, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(dspark.DSparkError) as e:  # d below one K box
        dspark.lm_head(H, LM, out, ws)
    assert e.value.status == dspark.ERR_INVALID_ARG


def test_draft_from_hidden_states():
    """The hidden-state path end to end on the device: base logits from the
    LM head, then the sequential draft. A base row can differ from the
    oracle's by one bf16 step in rare elements (float32 accumulation next to a
    rounding midpoint); the requests whose base rows equal the oracle's bit for
    bit (most of them at this size) must draft the oracle's tokens."""
    cfg = W.Workload("hidden_draft", R=32, gamma=2, V=512, rank=64, dtype="bf16", T=1.0, mode=W.CAUSAL,
                     seed=6100, w_sd=0.05)
    d = 512
    _, _, base = _run(cfg, d)
    inp = W.device_inputs(cfg)
    ws = dspark.new_workspace(cfg.R, cfg.gamma, cfg.V, cfg.rank, dspark.BF16, 1, "cuda")
    tok = torch.empty((cfg.R, cfg.gamma), dtype=torch.int32, device="cuda")
    q = torch.empty((cfg.R, cfg.gamma), dtype=torch.float32, device="cuda")
    qs = torch.empty((cfg.R, cfg.gamma, 2), dtype=torch.float32, device="cuda")
    dspark.draft_sequential(base, inp["anchor"], inp["W1"], inp["W2"], cfg.T, cfg.philox_seed, tok, q, qs, ws)
    assert dspark.device_status(ws) == dspark.OK
    tok, q = tok.cpu().numpy(), q.cpu().numpy()
    H_bits = W.hidden_np(cfg, d, range(cfg.R * cfg.gamma))
    ref_base = LH.lm_head_logits(H_bits, W.lm_head_np(cfg, d)).reshape(cfg.R, cfg.gamma, cfg.V)
    g_base = _bits(base)
    oi = W.oracle_inputs(cfg, [0])
    W1f, W2f = decode(oi["W1"]).astype(np.float64), decode(oi["W2"]).astype(np.float64)
    compared = 0
    for r in range(cfg.R):
        if not np.array_equal(g_base[r], ref_base[r]):
            continue
        o = draft_request(decode(ref_base[r]), int(oi["anchor"][r]), W1f, W2f, cfg.T, cfg.philox_seed, r)
        mis = next((k for k in range(cfg.gamma) if tok[r, k] != o["tokens"][k]), None)
        if mis is not None:
            assert o["margin"][mis] < 1e-6
        for k in range(cfg.gamma if mis is None else mis):
            assert abs(q[r, k] - o["q"][k]) <= 2e-3 * o["q"][k]
        compared += 1
    assert compared >= cfg.R // 2


def test_lm_head_qwen_shape_sampled():
    """A second model shape: Qwen3-4B's hidden size (2560) and vocabulary
    (151,936, not a multiple of 256: a partial last column tile), a 7-token
    block over 32 requests (224 rows: one row tile, its second half partial)."""
    cfg = W.Workload("lm_qwen", R=32, gamma=7, V=151936, rank=64, dtype="bf16", T=1.0, mode=W.CAUSAL, seed=6200)
    d = 2560
    H, LM, out = _run(cfg, d)
    rows = np.array([0, 100, 127, 128, 223])
    rng = np.random.default_rng(1)
    cols = np.unique(np.concatenate([rng.choice(cfg.V, 2000, replace=False), np.arange(cfg.V - 300, cfg.V)]))
    check_logits(_bits(out).reshape(-1, cfg.V)[rows][:, cols], W.hidden_np(cfg, d, rows), W.lm_head_np(cfg, d, cols))


def test_lm_head_repeats_bit_for_bit():
    """The GEMM run repeatedly on the same inputs (L2 flushed between runs)
    gives the same bits: the staging rings and the accumulator handover leave
    no room for a read of a buffer that is being refilled."""
    cfg = W.Workload("lm_rep", R=32, gamma=7, V=151936, rank=64, dtype="bf16", T=1.0, mode=W.CAUSAL, seed=6201)
    d = 2560
    H, LM, out = _run(cfg, d)
    first = out.clone()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(10):
        flush.zero_()
        dspark.lm_head(H, LM, out, ws)
        assert torch.equal(out, first)
    assert dspark.device_status(ws) == dspark.OK
