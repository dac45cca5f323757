"""Philox4x32-10 and the uniform/Gumbel mapping used by the sampler (oracle side).

Definition (Salmon et al., SC'11, section on Philox): the state is four 32-bit
words (c0, c1, c2, c3) and a two-word key (k0, k1).  One round multiplies c0 by
M0 = 0xD2511F53 and c2 by M1 = 0xCD9E8D57 as 32x32->64-bit products and
produces

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)).

Between rounds the key is bumped by the Weyl constants (0x9E3779B9,
0xBB67AE85) modulo 2**32.  Philox4x32-10 applies ten rounds.

Stream layout of the sampler (one reading of "the same counter-based Philox
stream"): for sequence row ``row`` at decode step ``step`` with 64-bit seed
``seed``, token ``t`` uses word ``t & 3`` of
Philox(ctr = (t >> 2, row, step, 0), key = (seed mod 2**32, seed >> 32)).
The word r maps to u = (2 * (r >> 9) + 1) * 2**-24, an odd multiple of 2**-24
in (0, 1), exactly representable in binary32 and binary64.
"""

from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(ctr: tuple[int, int, int, int], key: tuple[int, int]) -> tuple[int, int, int, int]:
    """Scalar Philox4x32-10 on Python integers."""
    c0, c1, c2, c3 = (int(v) & MASK32 for v in ctr)
    k0, k1 = (int(v) & MASK32 for v in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = M0 * c0
        p1 = M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0, p1 & MASK32, (p0 >> 32) ^ c3 ^ k1, p0 & MASK32)
    return c0, c1, c2, c3


def philox4x32_10_np(c0, c1, c2, c3, k0: int, k1: int):
    """The same function, elementwise over numpy arrays (uint64 lanes hold 32-bit words)."""
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) & np.uint64(MASK32) for v in (c0, c1, c2, c3))
    k0 = np.uint64(k0 & MASK32)
    k1 = np.uint64(k1 & MASK32)
    m32 = np.uint64(MASK32)
    for rnd in range(10):
        if rnd:
            k0 = np.uint64((int(k0) + W0) & MASK32)
            k1 = np.uint64((int(k1) + W1) & MASK32)
        p0 = np.uint64(M0) * c0
        p1 = np.uint64(M1) * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & m32,
                          (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & m32)
    return c0, c1, c2, c3


def sampler_words(tokens, row: int, step: int, seed: int) -> np.ndarray:
    """Raw 32-bit word of the sampler stream for each token id (uint64 array)."""
    t = np.asarray(tokens, dtype=np.uint64)
    n = t.shape[0]
    words = philox4x32_10_np(t >> np.uint64(2), np.full(n, row, np.uint64),
                             np.full(n, step, np.uint64), np.zeros(n, np.uint64),
                             seed & MASK32, (seed >> 32) & MASK32)
    lane = (t & np.uint64(3)).astype(np.int64)
    stacked = np.stack(words, axis=0)
    return stacked[lane, np.arange(n)]


def uniform_from_word(r) -> np.ndarray:
    """u = (2 * (r >> 9) + 1) * 2**-24, in float64 (exact)."""
    r = np.asarray(r, dtype=np.uint64)
    return ((r >> np.uint64(9)).astype(np.float64) * 2.0 + 1.0) * 2.0 ** -24


def gumbel(u) -> np.ndarray:
    """Standard Gumbel variate g = -log(-log u), float64."""
    u = np.asarray(u, dtype=np.float64)
    return -np.log(-np.log(u))
