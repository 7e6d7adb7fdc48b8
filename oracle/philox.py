"""Philox4x64-10 counter-based generator, written from its published definition.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle (see ``oracle/__init__.py``).

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random
Numbers: As Easy as 1, 2, 3", SC'11 -- the Philox-4xW S-box (two wide
multiplies per round, their high halves xored with the other counter words and
the round key) and the Weyl-sequence key schedule (golden ratio and sqrt(3)-1
increments).  Plain Python integers are used so every 64x64->128 product is
exact; nothing here is tuned.

The verify round draws its uniforms from this generator keyed by the caller's
seed and counted by (position, lane) so that every implementation of the round
sees the same numbers (the strata2signal guide, "Guess, then check": the
acceptance rule is a random test per draft; mashbox docs, "What it does for you":
a sampled request draws each token "with the same settings and seed").
"""

MASK64 = (1 << 64) - 1

# Round multipliers and key increments of Philox4x64 (SC'11, section 5).
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15  # golden ratio
PHILOX_W1 = 0xBB67AE8584CAA73B  # sqrt(3) - 1

ROUNDS = 10

# Uniforms are the top 24 bits of a 64-bit word scaled by 2^-24: exactly
# representable in float32 and float64, so every implementation holds the
# same value, in [0, 1).
UNIFORM_BITS = 24


def philox4x64_10(counter, key):
    """One Philox4x64-10 block: four 64-bit words from a 256-bit counter.

    ``counter`` is four ints, ``key`` two ints (all taken mod 2^64).
    """
    c0, c1, c2, c3 = (int(w) & MASK64 for w in counter)
    k0, k1 = (int(w) & MASK64 for w in key)
    for _ in range(ROUNDS):
        prod0 = PHILOX_M0 * c0
        prod1 = PHILOX_M1 * c2
        hi0, lo0 = prod0 >> 64, prod0 & MASK64
        hi1, lo1 = prod1 >> 64, prod1 & MASK64
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + PHILOX_W0) & MASK64
        k1 = (k1 + PHILOX_W1) & MASK64
    return c0, c1, c2, c3


def word_to_uniform(word):
    """Top 24 bits of a 64-bit word as a float in [0, 1)."""
    return float((int(word) & MASK64) >> (64 - UNIFORM_BITS)) * 2.0 ** -UNIFORM_BITS


def round_uniforms(seed, lane, position):
    """The two uniforms of (seed, lane, position).

    Counter = (position, lane, 0, 0), key = (seed, 0).  Word 0 is the
    acceptance uniform u of the draft at this position; word 1 is the uniform
    u' of an inverse-CDF draw made at this position (residual or bonus).
    """
    w = philox4x64_10((position, lane, 0, 0), (seed, 0))
    return word_to_uniform(w[0]), word_to_uniform(w[1])
