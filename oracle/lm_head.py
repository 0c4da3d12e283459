"""Base logits from the parallel backbone's hidden states -- oracle.

Test infrastructure: imported only by the tests, the smoke entry point and the
benchmark's CPU legs; never by the library.

What the pages define ([GN] "Etapa paralela": one forward pass of the
parallel backbone over the block yields hidden states and the base logits;
[GN] "Comunicação de estados ocultos": only the hidden state before the LM
head needs to travel, and the LM head is applied where the logits are used):
the base logits of a position are its final hidden state h [d] times the LM
head [d, V], logits = h . LM.

Readings where the pages are silent (listed in the design notes):
  * hidden states and the LM head are bf16 (the weights' precision); the
    logits the drafting stage consumes are bf16 too, the product rounded once
    to the nearest bf16 (ties to even) -- the form the base logits have in
    the rest of this library;
  * the product itself is the exact real-number sum; the oracle forms it in
    float64 (bf16 x bf16 products are exact there; the float64 sum is within
    d * 2^-53 of exact, far inside one bf16 step), then rounds.

Pins (tests/test_oracle_lm_head.py): the float64 -> bf16 rounding against
torch's float32 -> bf16 conversion on float32-representable values and
against the nearest neighbour found with exact fractions (ties to even); the
logits against exact rational arithmetic (Python fractions) element by
element; one-hot LM-head columns select and scale hidden-state entries.
"""

import numpy as np


def decode_bf16(bits):
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16_bits(x):
    """float64 -> bf16 bit patterns, to nearest with ties to even.

    Rounds the 52-bit float64 significand at its 45th bit (keeping 7 stored
    bits, as bf16 does): add half a step minus one plus the kept last bit,
    then clear the 45 low bits; the result has at most 8 significant bits and
    converts to float32 exactly, whose upper half is the bf16 pattern.
    Normal-range values (and zero) only."""
    b = np.asarray(x, dtype=np.float64).view(np.uint64)
    keep = (b >> np.uint64(45)) & np.uint64(1)
    r = ((b + np.uint64((1 << 44) - 1) + keep) >> np.uint64(45)) << np.uint64(45)
    y = r.view(np.float64).astype(np.float32)
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def lm_head_exact(H_bits, LM_bits):
    """h . LM in float64 for hidden states [M, d] and LM head [d, V] (bf16 bits)."""
    return decode_bf16(H_bits) @ decode_bf16(LM_bits)


def lm_head_logits(H_bits, LM_bits):
    """Base logits [M, V] as bf16 bit patterns: the product rounded once."""
    return round_bf16_bits(lm_head_exact(H_bits, LM_bits))


def abs_products(H_bits, LM_bits):
    """sum_i |h_i * lm_iv| [M, V] (float64): the scale of a float32 sum's error."""
    return np.abs(decode_bf16(H_bits)) @ np.abs(decode_bf16(LM_bits))
