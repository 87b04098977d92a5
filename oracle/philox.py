"""Philox4x32-10, written from its published definition.

Reference: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11, section 4 (the Philox S-box): a 4x32
counter, a 2x32 key, ten rounds; each round multiplies counter words 0 and 2 by
two fixed odd constants, keeps both halves of the 64-bit products, swaps the
pairs and XORs the high halves with the other counter words and the round key;
between rounds the key is bumped by the two Weyl constants (golden ratio and
sqrt(3) - 1, as 32-bit fixed point).

Use in FORGE: the explainer's Technical Summary §2 ("Precision and Fidelity")
asks for stochastic rounding of the BF16 weight write-back but names no random
source.  The reading used here: 16 random bits per element from Philox keyed by
the 64-bit seed, counter = (g_lo, g_hi, step_lo, step_hi) with g = idx >> 3, and
element j = idx & 7 taking 16-bit half (j & 1) of output word (j >> 1).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""

import numpy as np

# Multipliers of the two 32x32 -> 64-bit products in each round.
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
# Weyl sequence key increments.
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85

_MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(a: int, b: np.ndarray):
    """Full 64-bit product of the 32-bit constant a and the uint32 array b."""
    p = np.uint64(a) * b.astype(np.uint64)
    return (p >> np.uint64(32)).astype(np.uint32), (p & _MASK32).astype(np.uint32)


def philox4x32_10(counter: np.ndarray, key0, key1) -> np.ndarray:
    """Philox4x32 with 10 rounds.

    counter: uint32 array of shape (..., 4).  key0, key1: uint32 scalars or arrays
    broadcastable to counter[..., 0].  Returns a uint32 array of shape (..., 4).
    """
    c = np.asarray(counter, dtype=np.uint32)
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0 = np.asarray(key0, dtype=np.uint64) & _MASK32
    k1 = np.asarray(key1, dtype=np.uint64) & _MASK32
    for rnd in range(10):
        if rnd > 0:  # key schedule: bump before every round after the first
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        n0 = hi1 ^ c1 ^ k0.astype(np.uint32)
        n1 = lo1
        n2 = hi0 ^ c3 ^ k1.astype(np.uint32)
        n3 = lo0
        c0, c1, c2, c3 = n0, n1, n2, n3
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def sr_random16(idx: np.ndarray, seed: int, step: int) -> np.ndarray:
    """16 random bits (as uint32 in [0, 65535]) for each global element index.

    idx: int64 array of element indices n*K + k inside one weight matrix.
    seed: 64-bit key; step: the optimizer step (1-based) the rounding belongs to.
    """
    idx = np.asarray(idx, dtype=np.int64)
    g = (idx >> 3).astype(np.uint64)
    j = (idx & 7).astype(np.int64)
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    ctr = np.empty(idx.shape + (4,), dtype=np.uint32)
    ctr[..., 0] = (g & _MASK32).astype(np.uint32)
    ctr[..., 1] = (g >> np.uint64(32)).astype(np.uint32)
    ctr[..., 2] = np.uint32(step & 0xFFFFFFFF)
    ctr[..., 3] = np.uint32(step >> 32)
    out = philox4x32_10(ctr, seed & 0xFFFFFFFF, seed >> 32)
    word = np.take_along_axis(out, (j >> 1)[..., None], axis=-1)[..., 0]
    half = (j & 1).astype(np.uint32)
    return ((word >> (np.uint32(16) * half)) & np.uint32(0xFFFF)).astype(np.uint32)
