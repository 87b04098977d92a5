"""bfloat16 conversions: round-to-nearest-even and stochastic rounding.

bfloat16 is the upper half of an IEEE binary32.  Values are carried here as
uint16 bit patterns (numpy has no bfloat16).

Stochastic rounding follows the explainer's Technical Summary §2 ("Precision and
Fidelity", dead-zone bullet): the BF16 weight write-back must round so that the
expected stored value equals the FP32 result, letting sub-ULP updates
accumulate.  Reading used: add 16 uniform random bits to the FP32 bit pattern
(unsigned 32-bit arithmetic) and keep the top 16 bits.  On the magnitude this
rounds away from zero with probability (dropped bits) / 2^16, so the rounding is
unbiased for every finite input.  NaN becomes the canonical 0x7FC0; +-Inf is
kept; a finite value within one BF16 ULP of the largest finite magnitude may
round to Inf (it is where the carry leads).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""

import numpy as np


def f32_bits(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _is_nan_bits(u):
    return (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)


def bf16_bits_rne(x) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest, ties to even; NaN -> 0x7FC0."""
    u = f32_bits(x).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint32)
    r = np.where(_is_nan_bits(u.astype(np.uint32)), np.uint32(0x7FC0), r)
    return (r & np.uint32(0xFFFF)).astype(np.uint16)


def bf16_bits_stochastic(x, r16) -> np.ndarray:
    """float32 -> bf16 bits by stochastic rounding with the given 16 random bits."""
    u = f32_bits(x)
    r16 = np.asarray(r16, dtype=np.uint32) & np.uint32(0xFFFF)
    mag = u & np.uint32(0x7FFFFFFF)
    is_nan = mag > np.uint32(0x7F800000)
    is_inf = mag == np.uint32(0x7F800000)
    # uint32 wrap-around cannot happen: the largest finite pattern 0xFF7FFFFF
    # plus 0xFFFF stays below 2^32.
    rounded = (u.astype(np.uint64) + r16.astype(np.uint64)) >> np.uint64(16)
    out = np.where(is_inf, u >> np.uint32(16), rounded.astype(np.uint32))
    out = np.where(is_nan, np.uint32(0x7FC0), out)
    return (out & np.uint32(0xFFFF)).astype(np.uint16)


def bf16_ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Distance in representable bf16 steps between two bf16 bit patterns.

    Uses the standard monotone mapping of sign-magnitude patterns onto integers
    (+0 and -0 map to the same point)."""
    def ordinal(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordinal(a_bits) - ordinal(b_bits))
