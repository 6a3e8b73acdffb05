"""Philox4x32-10 and the random quantities the verification rule draws (oracle side).

Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3" (SC'11): a 4 x 32-bit counter and
a 2 x 32-bit key go through ten rounds; each round multiplies counter words 0
and 2 by two fixed odd constants, takes the high and low halves of the 64-bit
products, xors the high halves with the other counter words and the key, and
permutes; the key is bumped by two Weyl constants between rounds.

The pages leave the randomness of the rule unspecified; the key tuple below is
the one both the oracle and the CUDA path implement, each from this definition:

  key                      = (seed mod 2^32, seed >> 32)
  accept uniform (b, i)    = word 0 of Philox(counter = (0, i, b, 0))
  Gumbel uniform (b, j, v) = word (v mod 4) of Philox(counter = (v >> 2, j, b, 1))
  U(w)                     = ((w >> 9) + 0.5) * 2^-23, in (0, 1); the numerator
                             2 (w >> 9) + 1 has at most 24 bits, so U is exact in fp32
  G(U)                     = -ln(-ln U)                (standard Gumbel)
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
# Multipliers and Weyl key increments of Philox4x32 (SC'11, Table 2 / Section 4).
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten rounds of Philox4x32 on broadcastable arrays of 32-bit words.

    Returns the four output words as uint32 arrays.
    """
    c0, c1, c2, c3, k0, k1 = (np.asarray(x, dtype=np.uint64) & MASK32 for x in (c0, c1, c2, c3, k0, k1))
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(c0, c1, c2, c3, k0, k1)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & MASK32
            k1 = (k1 + PHILOX_W1) & MASK32
        prod0 = PHILOX_M0 * c0            # < 2^64: both factors < 2^32
        prod1 = PHILOX_M1 * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & MASK32
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def key_of(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def uniform_from_word(w) -> np.ndarray:
    """Top 23 bits of a word, centred in their cell: ((w >> 9) + 0.5) / 2^23.

    Lies in [2^-24, 1 - 2^-24] and is exactly representable in fp32.
    """
    w = np.asarray(w, dtype=np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def accept_uniform(seed: int, b: int, i: int) -> float:
    """The uniform that decides draft position i of sequence b."""
    k0, k1 = key_of(seed)
    w = philox4x32_10(0, i, b, 0, k0, k1)[0]
    return float(uniform_from_word(w))


def gumbel_uniforms(seed: int, b: int, j: int, V: int) -> np.ndarray:
    """Uniforms U(seed, b, j, v) for v = 0..V-1 (row j of sequence b)."""
    k0, k1 = key_of(seed)
    v = np.arange(V, dtype=np.uint64)
    words = philox4x32_10(v >> np.uint64(2), j, b, 1, k0, k1)
    lane = (v & np.uint64(3)).astype(np.int64)
    w = np.choose(lane, words)
    return uniform_from_word(w)


def gumbel(u: np.ndarray) -> np.ndarray:
    """Standard Gumbel noise -ln(-ln U) in fp64."""
    return -np.log(-np.log(np.asarray(u, dtype=np.float64)))
