"""Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
as 1, 2, 3", SC'11) — oracle copy, written from the published definition.

One round maps counter (c0,c1,c2,c3) under key (k0,k1) to

    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57; the key is bumped by the Weyl
constants (0x9E3779B9, 0xBB67AE85) between rounds; ten rounds.

The sampling verifier draws every uniform from this generator with the
counter (step, offset, test, purpose) and the key (seed low, seed high), so a
second implementation of the same definition draws the same numbers.
"""
from __future__ import annotations

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF

# purposes of a draw
ACCEPT, RESIDUAL, PLAIN = 0, 1, 2


def philox4x32_10(ctr, key):
    c0, c1, c2, c3 = (int(v) & MASK for v in ctr)
    k0, k1 = (int(v) & MASK for v in key)
    for r in range(10):
        if r:
            k0 = (k0 + W0) & MASK
            k1 = (k1 + W1) & MASK
        p0 = M0 * c0
        p1 = M1 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & MASK, p1 & MASK, ((p0 >> 32) ^ c3 ^ k1) & MASK, p0 & MASK
    return c0, c1, c2, c3


def uniform(seed: int, step: int, offset: int, test: int, purpose: int) -> float:
    """A uniform in [0, 1) with 24 bits: (word0 >> 8) * 2**-24 (exact in fp32)."""
    w = philox4x32_10((step, offset, test, purpose), (seed & MASK, (seed >> 32) & MASK))[0]
    return (w >> 8) * (1.0 / 16777216.0)


def philox4x32_10_np(c0, c1, c2, c3, k0: int, k1: int):
    """Vectorised copy of ``philox4x32_10`` over numpy counter arrays (same definition)."""
    import numpy as np
    m = np.uint64(MASK)
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) & m for v in (c0, c1, c2, c3))
    k0, k1 = np.uint64(k0 & MASK), np.uint64(k1 & MASK)
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(W0)) & m
            k1 = (k1 + np.uint64(W1)) & m
        p0 = np.uint64(M0) * c0
        p1 = np.uint64(M1) * c2
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ k0) & m, p1 & m, ((p0 >> np.uint64(32)) ^ c3 ^ k1) & m, p0 & m
    return c0, c1, c2, c3
