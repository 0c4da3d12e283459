"""Philox4x64-10 and the uniform draws of one DSpark round (oracle side).

The pages fix no random-number generator; they only require that the rejection
sampler be lossless ([GN] §Definição do problema: the target verifies the block
in one pass and rejection sampling keeps the longest prefix consistent with the
target distribution). Reading taken here: every random decision of a round
consumes exactly one uniform u = U(seed, r, k, purpose) from a counter-based
generator, so that each decision is reproducible and independent of launch
order.

Generator: Philox4x64 with 10 rounds, as published by Salmon, Moraes, Dror and
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11). One block maps a
128-bit key and a 256-bit counter to four 64-bit words. Pinned against
numpy.random.Philox (an independent implementation of the same generator) in
tests/test_oracle_philox.py.

Mapping used by the round:
  key     = (seed, 0x44535041524B0000)          ("DSPARK" in ASCII, zero padded)
  counter = (r, k, purpose, 0)
  u       = (2 * (w0 >> 12) + 1) * 2**-53       (w0 = first output word)
u is an exact double in (0, 1): 2*(w0>>12)+1 is an odd integer below 2**53.
"""

MASK64 = (1 << 64) - 1

# Round multipliers and Weyl key increments of Philox4x64 (published constants
# of the generator).
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15
PHILOX_W1 = 0xBB67AE8584CAA73B

KEY_HI = 0x44535041524B0000

DRAFT, ACCEPT, RESID, BONUS = 0, 1, 2, 3


def philox4x64_10(counter, key):
    """One Philox4x64-10 block: 4x64-bit counter, 2x64-bit key -> 4 words."""
    c0, c1, c2, c3 = (int(x) & MASK64 for x in counter)
    k0, k1 = (int(x) & MASK64 for x in key)
    for _ in range(10):
        prod0 = PHILOX_M0 * c0
        prod1 = PHILOX_M1 * c2
        hi0, lo0 = prod0 >> 64, prod0 & MASK64
        hi1, lo1 = prod1 >> 64, prod1 & MASK64
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + PHILOX_W0) & MASK64
        k1 = (k1 + PHILOX_W1) & MASK64
    return c0, c1, c2, c3


def uniform(seed, r, k, purpose):
    """U(seed, r, k, purpose) in (0, 1) as an exact double."""
    w0 = philox4x64_10((r, k, purpose, 0), (seed, KEY_HI))[0]
    return float(2 * (w0 >> 12) + 1) * 2.0 ** -53
