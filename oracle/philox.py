"""Philox4x32-10 counter-based random number generator.

Test infrastructure (see ``oracle/__init__``).

Written from the published definition: J. K. Salmon, M. A. Moraes,
R. O. Dror, D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11,
section 4 (Philox).  One round maps counter (x0, x1, x2, x3) with key (k0, k1) to

    (hi(M1*x2) ^ x1 ^ k0,  lo(M1*x2),  hi(M0*x0) ^ x3 ^ k1,  lo(M0*x0))

with M0 = 0xD2511F53, M1 = 0xCD9E8D57; the key is bumped by the Weyl
constants (0x9E3779B9, 0xBB67AE85) between rounds; ten rounds.

The pages ask for stochastic rounding of gradients in NVFP4 and name no
generator ("How to Optimize Transformer-Based Models for Low-Precision
Training", section "実モデルにおける結果の解釈", list of NVFP4 overheads); a
counter-based generator is the plainest reading that lets any element's random
word be recomputed independently.  Parity: pinned (known-answer vectors and
uniformity statistics, tests/test_oracle_philox).
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
_MASK = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Vectorised Philox4x32-10 over counter arrays; returns four uint32 arrays."""
    x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) & np.uint64(_MASK) for c in (c0, c1, c2, c3))
    x0, x1, x2, x3 = np.broadcast_arrays(x0, x1, x2, x3)
    key0, key1 = int(k0) & _MASK, int(k1) & _MASK
    mask = np.uint64(_MASK)
    for rnd in range(10):
        if rnd > 0:
            key0 = (key0 + W0) & _MASK
            key1 = (key1 + W1) & _MASK
        p0 = np.uint64(M0) * x0
        p1 = np.uint64(M1) * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        x0, x1, x2, x3 = hi1 ^ x1 ^ np.uint64(key0), lo1, hi0 ^ x3 ^ np.uint64(key1), lo0
    return tuple(v.astype(np.uint32) for v in (x0, x1, x2, x3))


def element_words(n_elems: int, first: int, seed: int, copy_id: int, offset: int) -> np.ndarray:
    """32-bit random word of elements ``first .. first + n_elems - 1`` of a tensor copy.

    Elements are taken in groups of four consecutive indices; one Philox4x32-10
    output (128 bits) serves four groups (16 elements): element g (row-major index
    within the quantized copy) reads word (g // 4) % 4 of Philox4x32-10 with
    counter (g // 16, copy_id, offset_lo, offset_hi) and key (seed_lo, seed_hi).
    The four elements of a group see the same word; how they split it is part of
    the rounding rule (oracle.quantize.sr_rand16).
    """
    g = np.arange(first, first + n_elems, dtype=np.int64)
    grp = g >> 4
    uniq = np.unique(grp)
    w = philox4x32_10(uniq & _MASK, np.uint64(copy_id), np.uint64(offset & _MASK),
                      np.uint64((offset >> 32) & _MASK), seed & _MASK, (seed >> 32) & _MASK)
    table = np.stack(w, axis=1)  # [n_groups, 4]
    return table[grp - uniq[0], (g >> 2) & 3].astype(np.uint32)
