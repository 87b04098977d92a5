"""The FORGE backward step of one linear layer y = x W^T, on the CPU.

Written from the explainer "FORGE: Fused On-Register Gradient Elimination for
Memory-Efficient LLM Training" (gist.science), Technical Summary:

  §5 "Limitations": the input gradient dX = dY W is taken from the weights
      *before* the update;
  §2 "Core Mechanism": the weight gradient dW[n, k] = sum_t dY[t, n] X[t, k]
      is accumulated, the elementwise optimizer is applied, and only the
      updated weights and (optionally quantised) moments are written back;
  §2 "Exactness": the tiled update equals the update computed from the full
      gradient, up to the order of summation over tokens.  This oracle uses the
      full-gradient form: dW is formed for the whole matrix (or for any chosen
      set of elements: each element's update depends only on its own
      coordinate), accumulated in float64 and rounded once to float32;
  §2 "Precision and Fidelity": the gradient stays float32 (never truncated to
      bf16); bf16 weights are written back by stochastic rounding; INT8 states
      use blocks of 64.

Per element the order is: dequantise states -> rule (float32) -> requantise
states (new block absmax) and round the weight.

Layouts (row-major): X [T, K] bf16, dY [T, N] bf16, W [N, K] (float32 master or
bf16), states [N, K] (float32; int8/uint8 codes with float32 absmax
[N, K / 64]; or bf16 rounded to nearest even), dX [T, K] bf16.  bf16 tensors
are numpy uint16 bit patterns.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).
"""

import numpy as np

from . import optimizers as opt
from .philox import sr_random16
from .quant import quantize_blocks, dequantize_blocks
from .rounding import bf16_bits_to_f32, bf16_bits_rne, bf16_bits_stochastic


# ----------------------------------------------------------------------------
# Gradients
# ----------------------------------------------------------------------------

def weight_gradient(X_bits, dY_bits, rows=None, cols=None) -> np.ndarray:
    """g[n, k] = sum_t dY[t, n] * X[t, k]; float64 accumulation, one rounding to float32.

    rows=(n0, n1), cols=(k0, k1) restrict the result to a sub-block."""
    X = bf16_bits_to_f32(X_bits)
    dY = bf16_bits_to_f32(dY_bits)
    if rows is not None:
        dY = dY[:, rows[0]:rows[1]]
    if cols is not None:
        X = X[:, cols[0]:cols[1]]
    g64 = dY.astype(np.float64).T @ X.astype(np.float64)
    return g64.astype(np.float32)


def bf16_bits_rne_from_f64(x) -> np.ndarray:
    """float64 -> bf16 bits, correctly rounded (nearest, ties to even).

    Goes through float32 with round-to-odd, which keeps the second rounding to
    bf16 correct because float32 carries more than two extra bits."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    back = f.astype(np.float64)
    inexact = back != x
    overshoot = np.abs(back) > np.abs(x)
    f = np.where(inexact & overshoot, np.nextafter(f, np.float32(0)), f).astype(np.float32)
    bits = f.view(np.uint32) | np.where(inexact, np.uint32(1), np.uint32(0)).astype(np.uint32)
    return bf16_bits_rne(bits.view(np.float32))


def input_gradient(dY_bits, W_bf16_bits) -> np.ndarray:
    """dX[t, k] = sum_n dY[t, n] * W[n, k] with float64 accumulation, rounded to bf16."""
    dY = bf16_bits_to_f32(dY_bits).astype(np.float64)
    W = bf16_bits_to_f32(W_bf16_bits).astype(np.float64)
    return bf16_bits_rne_from_f64(dY @ W)


def weights_for_dx(W, w_dtype: str) -> np.ndarray:
    """The bf16 operand dX is formed from: the bf16 weights themselves, or the
    float32 master weights rounded to nearest-even (mixed-precision reading)."""
    if w_dtype == "bf16":
        return np.asarray(W, dtype=np.uint16)
    return bf16_bits_rne(W)


# ----------------------------------------------------------------------------
# Elementwise update of a block of W
# ----------------------------------------------------------------------------

def update_block(kind, hp, step, seed, g, W, w_dtype, s1=None, s2=None,
                 s1_scale=None, s2_scale=None, s_dtype="fp32", n0=0, k0=0, K=None,
                 block=64):
    """Apply one optimizer step to the block W[n0:n0+R, k0:k0+C] given its gradient g.

    K is the full row length of W (for the element index n*K + k that keys the
    stochastic rounding).  s_dtype: 'fp32', 'int8' (codes with an absmax per
    `block` row elements; 64 is the method's) or 'bf16' (moments stored as
    bf16, rounded to nearest even after the FP32 update).  Returns a dict with
    W, s1, s2, s1_scale, s2_scale for the block (None where unused)."""
    g = np.asarray(g, dtype=np.float32)
    R, C = g.shape
    if K is None:
        K = C
    uses1, uses2 = opt.USES_S1[kind], opt.USES_S2[kind]
    # current weight value in float32
    wf = bf16_bits_to_f32(W) if w_dtype == "bf16" else np.asarray(W, dtype=np.float32)
    # dequantise states
    if s_dtype == "int8":
        m = dequantize_blocks(s1, s1_scale, signed=True, block=block) if uses1 else None
        v = dequantize_blocks(s2, s2_scale, signed=False, block=block) if uses2 else None
    elif s_dtype == "bf16":
        m = bf16_bits_to_f32(s1) if uses1 else None
        v = bf16_bits_to_f32(s2) if uses2 else None
    else:
        m = np.asarray(s1, dtype=np.float32) if uses1 else None
        v = np.asarray(s2, dtype=np.float32) if uses2 else None
    sc = opt.step_scalars(kind, hp, step)
    w_new, m_new, v_new = opt.apply_rule(kind, sc, wf, g, m, v)
    out = {"W": None, "s1": None, "s2": None, "s1_scale": None, "s2_scale": None}
    if w_dtype == "bf16":
        n_idx = np.arange(n0, n0 + R, dtype=np.int64)[:, None]
        k_idx = np.arange(k0, k0 + C, dtype=np.int64)[None, :]
        r16 = sr_random16(n_idx * np.int64(K) + k_idx, seed, step)
        out["W"] = bf16_bits_stochastic(w_new, r16)
    else:
        out["W"] = w_new.astype(np.float32)
    if s_dtype == "int8":
        if uses1:
            out["s1"], out["s1_scale"] = quantize_blocks(m_new, signed=True, block=block)
        if uses2:
            out["s2"], out["s2_scale"] = quantize_blocks(v_new, signed=False, block=block)
    elif s_dtype == "bf16":
        out["s1"] = bf16_bits_rne(m_new) if uses1 else None
        out["s2"] = bf16_bits_rne(v_new) if uses2 else None
    else:
        out["s1"] = m_new.astype(np.float32) if uses1 else None
        out["s2"] = v_new.astype(np.float32) if uses2 else None
    return out


# ----------------------------------------------------------------------------
# Whole step
# ----------------------------------------------------------------------------

def linear_bwd_step(X_bits, dY_bits, state: dict, kind: int, hp, step: int, seed: int,
                    want_dx: bool = True) -> dict:
    """One full step on one layer.

    state: dict with W (float32 or uint16 bf16 bits), w_dtype ('fp32' | 'bf16'),
    s_dtype ('fp32' | 'int8' | 'bf16'), s1, s2, s1_scale, s2_scale.  Returns a new dict of
    the same form plus 'dX' (bf16 bits) when want_dx."""
    W = state["W"]
    w_dtype, s_dtype = state["w_dtype"], state["s_dtype"]
    N, K = W.shape
    out = {}
    if want_dx:
        out["dX"] = input_gradient(dY_bits, weights_for_dx(W, w_dtype))
    g = weight_gradient(X_bits, dY_bits)
    upd = update_block(kind, hp, step, seed, g, W, w_dtype, state.get("s1"), state.get("s2"),
                       state.get("s1_scale"), state.get("s2_scale"), s_dtype, 0, 0, K)
    out.update(upd)
    out["w_dtype"], out["s_dtype"] = w_dtype, s_dtype
    return out


def _tile(a, n0, k0, tn, tk, block=1):
    if a is None:
        return None
    return a[n0:n0 + tn, (k0 // block):(k0 + tk) // block]


def linear_bwd_step_tiles(X_bits, dY_bits, state: dict, kind: int, hp, step: int, seed: int,
                          tiles, tile=(128, 128)) -> dict:
    """The same step evaluated only on the listed W tiles [(n0, k0), ...].

    Every element's update depends only on its own coordinate (§2 "Exactness"),
    so a tile of the result is computed from the matching tile of the gradient
    and of the state.  Returns {(n0, k0): dict(W, s1, s2, s1_scale, s2_scale)}."""
    W = state["W"]
    N, K = W.shape
    tn, tk = tile
    res = {}
    for (n0, k0) in tiles:
        assert n0 % tn == 0 and k0 % tk == 0 and n0 + tn <= N and k0 + tk <= K
        g = weight_gradient(X_bits, dY_bits, rows=(n0, n0 + tn), cols=(k0, k0 + tk))
        res[(n0, k0)] = update_block(
            kind, hp, step, seed, g, _tile(W, n0, k0, tn, tk), state["w_dtype"],
            _tile(state.get("s1"), n0, k0, tn, tk), _tile(state.get("s2"), n0, k0, tn, tk),
            _tile(state.get("s1_scale"), n0, k0, tn, tk, 64),
            _tile(state.get("s2_scale"), n0, k0, tn, tk, 64),
            state["s_dtype"], n0, k0, K)
    return res
