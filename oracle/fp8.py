"""FP8 (E4M3) operands of the FORGE step: decoding and the weight gradient.

The explainer (Technical Summary §4, "Composability") says FORGE composes with
FP8 quantisation; it gives no format or scale recipe.  Reading used: X and dY
arrive as E4M3 codes (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits; exponent 15 with mantissa 7 is NaN, there is no infinity; largest
finite 448) with one float32 scale per tensor, value = decode(code) * scale,
laid out token-contiguous: X^T [K, T] and dY^T [N, T].  The gradient is
g[n, k] = RN32( RN32(S) * c ) with S = sum_t decode(dY[n, t]) decode(X[k, t])
(exact: every product of two E4M3 values fits float64 exactly, and so do sums
of up to 2^18 of them) and c = RN32(x_scale * dy_scale) formed in double.
The rest of the step is the float32 optimizer of optimizers.py.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""

import numpy as np


def e4m3_bits_to_f32(b) -> np.ndarray:
    """Exact decoding of E4M3 codes (uint8) to float32; NaN codes -> NaN."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return (sign * val).astype(np.float32)


def grad_scale(x_scale: float, dy_scale: float) -> np.float32:
    return np.float32(float(np.float32(x_scale)) * float(np.float32(dy_scale)))


def weight_gradient_fp8(xt_bits, dyt_bits, x_scale, dy_scale) -> np.ndarray:
    """g [N, K] from X^T [K, T] and dY^T [N, T] E4M3 codes and their scales."""
    X = e4m3_bits_to_f32(xt_bits).astype(np.float64)
    dY = e4m3_bits_to_f32(dyt_bits).astype(np.float64)
    S = (dY @ X.T).astype(np.float32)
    return (S * grad_scale(x_scale, dy_scale)).astype(np.float32)
