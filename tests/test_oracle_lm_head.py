"""Pins of the oracle's base logits from hidden states ([GN] "Etapa
paralela": hidden states and base logits of the parallel backbone; [GN]
"Comunicação de estados ocultos": the LM head applied to the hidden state)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import lm_head as LH

torch = pytest.importorskip("torch")


def _bits(x32):
    return (np.asarray(x32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_frac(bits):
    v = float(LH.decode_bf16(np.array([bits], dtype=np.uint16))[0])
    return Fraction(v)


def _nearest_bf16_exact(q):
    """Nearest bf16 to the rational q, ties to even, by exact search over
    the two neighbours of q's float32 truncation."""
    x = float(q)
    b = int(np.array([x], dtype=np.float32).view(np.uint32)[0]) >> 16
    cands = []
    for c in (b - 1, b, b + 1, b + 2):
        c &= 0xFFFF
        if (c & 0x7F80) == 0x7F80:
            continue
        cands.append(c)
    best = min(cands, key=lambda c: (abs(_bf16_frac(c) - q), c & 1))
    return best


def test_round_bf16_bits_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x32 = (rng.normal(0, 1, 50000) * np.exp(rng.uniform(-30, 30, 50000))).astype(np.float32)
    # exact midpoints between bf16 neighbours, both parities of the kept bit
    mids = (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3F000000 + 0x8000).view(np.float32)
    x32 = np.concatenate([x32, mids, -mids])
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(LH.round_bf16_bits(x32.astype(np.float64)), ref)


def test_round_bf16_bits_is_the_nearest_with_ties_to_even():
    rng = np.random.default_rng(1)
    xs = list(rng.normal(0, 3, 300))
    # float64 values just off a bf16 midpoint (a float32 detour would land on it)
    for b in (0x3F80, 0x3F81, 0xC0A3, 0x4123):
        mid = (_bf16_frac(b) + _bf16_frac(b + 1)) / 2
        for eps in (Fraction(1, 2 ** 40), -Fraction(1, 2 ** 40), 0):
            xs.append(float(mid + eps * abs(mid)))
    for x in xs:
        got = int(LH.round_bf16_bits(np.array([x]))[0])
        assert got == _nearest_bf16_exact(Fraction(x)), (x, hex(got))


@pytest.mark.parametrize("d", [8, 64, 7168])
def test_logits_equal_exact_rational_sums(d):
    rng = np.random.default_rng(d)
    M, V = 3, 5
    H = _bits(rng.normal(0, 1, (M, d)).astype(np.float32))
    LM = _bits(rng.normal(0, 1.5 / np.sqrt(d), (d, V)).astype(np.float32))
    got = LH.lm_head_logits(H, LM)
    Hf, LMf = LH.decode_bf16(H), LH.decode_bf16(LM)
    for i in range(M):
        for v in range(V):
            q = sum(Fraction(float(Hf[i, j])) * Fraction(float(LMf[j, v])) for j in range(d))
            assert int(got[i, v]) == _nearest_bf16_exact(q)


def test_one_hot_columns_select_hidden_entries():
    rng = np.random.default_rng(3)
    M, d, V = 6, 64, 40
    H = _bits(rng.normal(0, 1, (M, d)).astype(np.float32))
    LMf = np.zeros((d, V), dtype=np.float32)
    sel = rng.integers(0, d, V)
    LMf[sel, np.arange(V)] = 0.5
    got = LH.decode_bf16(LH.lm_head_logits(H, _bits(LMf)))
    assert np.array_equal(got, 0.5 * LH.decode_bf16(H)[:, sel])
