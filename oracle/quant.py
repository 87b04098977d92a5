"""Block-wise INT8 optimizer-state quantiser, block size 64.

The explainer's Technical Summary §2 ("Precision and Fidelity", last bullet)
fixes only the granularity: INT8 optimizer states with blocks of 64 elements
(against 2048 in standard 8-bit optimizers).  Reading used for everything else
(the pages are silent): a linear absmax code per block of 64 contiguous
elements of a row,

    a = max |x_i|                       (stored as the block's fp32 scale)
    s = a / 127   (signed state, codes -127..127)
        a / 255   (unsigned state, codes 0..255)
    q_i = clamp(round_half_even(x_i / s))   (q_i = 0 when a == 0 or x_i / s is NaN)
    dequantised x_i = float(q_i) * s        (s recomputed from a by the same division)

Every operation is a single IEEE float32 operation.  The first moment (may be
negative) uses the signed code; the second moment / accumulated square (never
negative) uses the unsigned code.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""

import numpy as np

BLOCK = 64


def _levels(signed: bool) -> np.float32:
    return np.float32(127.0) if signed else np.float32(255.0)


def quantize_blocks(x, signed: bool, block: int = BLOCK):
    """x: float32 [rows, cols] with cols % block == 0 (block 64 is the method's;
    other sizes serve the block-size comparison).

    Returns (codes, absmax): codes int8 (signed) or uint8 (unsigned) [rows, cols],
    absmax float32 [rows, cols // block]."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % block == 0
    xb = x.reshape(rows, cols // block, block)
    ax = np.abs(xb)
    # NaN never wins the maximum (it compares false), matching a running max
    # that only replaces on a strictly larger value.
    absmax = np.where(np.isnan(ax), np.float32(0), ax).max(axis=2).astype(np.float32)
    s = (absmax / _levels(signed)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (xb / s[..., None]).astype(np.float32)
    q = np.rint(r)
    lo = np.float32(-127.0) if signed else np.float32(0.0)
    hi = _levels(signed)
    q = np.minimum(np.maximum(q, lo), hi)
    q = np.where(np.isnan(r) | (absmax[..., None] == 0), np.float32(0), q)
    codes = q.astype(np.int8 if signed else np.uint8).reshape(rows, cols)
    return codes, absmax


def dequantize_blocks(codes, absmax, signed: bool, block: int = BLOCK) -> np.ndarray:
    codes = np.asarray(codes)
    rows, cols = codes.shape
    absmax = np.asarray(absmax, dtype=np.float32).reshape(rows, cols // block)
    s = (absmax / _levels(signed)).astype(np.float32)
    qf = codes.astype(np.float32).reshape(rows, cols // block, block)
    return (qf * s[..., None]).astype(np.float32).reshape(rows, cols)
