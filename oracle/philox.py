"""Philox4x32-10 counter-based generator, written from its published
definition (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy
as 1, 2, 3", SC 2011): a 128-bit counter (four 32-bit words) and a 64-bit key
(two words) go through 10 rounds.  One round multiplies counter words 0 and 2
by the constants M0 = 0xD2511F53 and M1 = 0xCD9E8D57 into 64-bit products and
rearranges:  (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); between rounds the key is advanced by the
Weyl constants (0x9E3779B9, 0xBB67AE85).

TEST INFRASTRUCTURE ONLY (part of the oracle): never on the product path.
"""
from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Vectorised Philox4x32-10.  Counter words are arrays (or scalars) of
    unsigned 32-bit values; the key is two Python ints.  Returns the four
    output words as uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint64) for x in (c0, c1, c2, c3))
    for _ in range(10):
        p0 = M0 * c0
        p1 = M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + W0) & 0xFFFFFFFF
        k1 = (k1 + W1) & 0xFFFFFFFF
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))
