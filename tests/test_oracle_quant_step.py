"""Pins for the oracle's INT8 block-64 quantiser and for the whole linear step.

Quantiser: a hand-worked fixture (tests/golden/quant_block64.json) plus the
invariants any absmax code must satisfy.  Linear step: brute-force exact sums
on tiny inputs, the explainer's exactness claim (Technical Summary §2: a tiled
update equals the full-gradient update) checked bit for bit on integer-grid
inputs, dX from the pre-update weights (§5 "Limitations"), the FP32 gradient
(§2 "Precision and Fidelity": never truncated to bf16), and the INT8 ordering
(the update consumes the new float32 moments; quantisation comes after).
"""

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import quant, rounding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ quantiser

def test_quant_golden_fixture():
    with open(os.path.join(GOLDEN, "quant_block64.json")) as f:
        blocks = json.load(f)["blocks"]
    for blk in blocks:
        x = np.zeros((1, 64), dtype=np.float32)
        want = np.zeros(64, dtype=np.int64)
        for i, v, code, _why in blk["entries"]:
            x[0, i] = np.float32(float.fromhex(v))
            want[i] = code
        codes, absmax = quant.quantize_blocks(x, signed=blk["signed"])
        assert codes.dtype == (np.int8 if blk["signed"] else np.uint8)
        assert codes[0].astype(np.int64).tolist() == want.tolist(), blk["name"]
        assert absmax[0, 0] == np.float32(float.fromhex(blk["absmax"])), blk["name"]
        deq = quant.dequantize_blocks(codes, absmax, signed=blk["signed"])
        s = np.float32(float.fromhex(blk["absmax"])) / np.float32(127 if blk["signed"] else 255)
        assert np.array_equal(deq[0], want.astype(np.float32) * s)


@pytest.mark.parametrize("signed", [True, False])
def test_quant_invariants(signed):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 64 * 8)).astype(np.float32) * np.float32(1e-3)
    if not signed:
        x = np.abs(x)
    x[3, 64:128] = 0.0  # one all-zero block
    codes, absmax = quant.quantize_blocks(x, signed)
    deq = quant.dequantize_blocks(codes, absmax, signed)
    xb = x.reshape(16, 8, 64)
    assert np.array_equal(absmax, np.abs(xb).max(axis=2))
    s = (absmax / np.float32(127 if signed else 255)).astype(np.float64)
    err = np.abs(deq.astype(np.float64) - x.astype(np.float64)).reshape(16, 8, 64)
    assert np.all(err <= s[..., None] * 0.5 * (1 + 1e-5) + 1e-30)
    top = 127 if signed else 255
    cb = codes.astype(np.int64).reshape(16, 8, 64)
    arg = np.abs(xb).argmax(axis=2)
    picked = np.take_along_axis(cb, arg[..., None], axis=2)[..., 0]
    nz = absmax > 0
    assert np.all(np.abs(picked[nz]) == top)
    assert np.all(cb[3, 1] == 0) and absmax[3, 1] == 0
    assert cb.min() >= (-127 if signed else 0) and cb.max() <= top


def test_quant_block_size_is_64():
    """Changing one element changes the scale of its own 64-block only."""
    x = np.full((1, 256), 0.5, dtype=np.float32)
    x[0, 70] = 4.0
    _, absmax = quant.quantize_blocks(x, signed=True)
    assert absmax[0].tolist() == [0.5, 4.0, 0.5, 0.5]


# ------------------------------------------------------------------ gradients

def _bits(a):
    return rounding.bf16_bits_rne(np.asarray(a, dtype=np.float32))


def test_weight_gradient_brute_force_tiny():
    rng = np.random.default_rng(4)
    T, N, K = 5, 3, 4
    X = _bits(rng.standard_normal((T, K)))
    dY = _bits(rng.standard_normal((T, N)) * 1e-2)
    g = ls.weight_gradient(X, dY)
    Xf, dYf = rounding.bf16_bits_to_f32(X), rounding.bf16_bits_to_f32(dY)
    for n, k in itertools.product(range(N), range(K)):
        exact = sum(Fraction(float(dYf[t, n])) * Fraction(float(Xf[t, k])) for t in range(T))
        assert g[n, k] == np.float32(float(exact)), (n, k)  # float() rounds correctly
    assert g.shape == (N, K)


def test_input_gradient_brute_force_exact():
    rng = np.random.default_rng(6)
    T, N, K = 4, 6, 3
    dY = _bits(rng.integers(-8, 9, size=(T, N)) * 2.0 ** -6)
    W = _bits(rng.integers(-8, 9, size=(N, K)) * 2.0 ** -5)
    dX = ls.input_gradient(dY, W)
    dYf, Wf = rounding.bf16_bits_to_f32(dY), rounding.bf16_bits_to_f32(W)
    for t, k in itertools.product(range(T), range(K)):
        exact = sum(Fraction(float(dYf[t, n])) * Fraction(float(Wf[n, k])) for n in range(N))
        assert rounding.bf16_bits_to_f32(dX[t:t + 1, k])[0] == float(exact)


def test_bf16_from_f64_is_correctly_rounded():
    # just above the tie between 1 and 1 + 2^-7: a float32 detour would land on
    # the tie and round down to even; the correct bf16 is 1 + 2^-7
    x = np.array([1.0 + 2 ** -8 + 2 ** -30, 1.0 + 2 ** -8, 1.0 + 2 ** -8 - 2 ** -30,
                  -(1.0 + 2 ** -8 + 2 ** -40)], dtype=np.float64)
    got = ls.bf16_bits_rne_from_f64(x).tolist()
    assert got == [0x3F81, 0x3F80, 0x3F80, 0xBF81]


# ------------------------------------------------------------------ whole step

def _grid_inputs(T, N, K, seed):
    rng = np.random.default_rng(seed)
    X = _bits(rng.integers(-4, 5, size=(T, K)).astype(np.float32))
    dY = _bits(rng.integers(-4, 5, size=(T, N)).astype(np.float32) * np.float32(2.0 ** -12))
    return X, dY


def _state(N, K, w_dtype, s_dtype, kind, seed=0):
    rng = np.random.default_rng(seed + 100)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    st = {"w_dtype": w_dtype, "s_dtype": s_dtype,
          "W": W if w_dtype == "fp32" else _bits(W)}
    m = (rng.standard_normal((N, K)) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal((N, K)) * 1e-6).astype(np.float32)
    for key, arr, signed, uses in (("s1", m, True, opt.USES_S1[kind]),
                                   ("s2", v, False, opt.USES_S2[kind])):
        if not uses:
            continue
        if s_dtype == "int8":
            st[key], st[key + "_scale"] = quant.quantize_blocks(arr, signed)
        elif s_dtype == "bf16":
            st[key] = rounding.bf16_bits_rne(arr)
        else:
            st[key] = arr
    return st


@pytest.mark.parametrize("kind", range(8), ids=opt.NAMES)
@pytest.mark.parametrize("w_dtype,s_dtype", [("fp32", "fp32"), ("bf16", "fp32"), ("bf16", "int8"),
                                             ("bf16", "bf16")])
def test_tiled_update_equals_full_gradient_update(kind, w_dtype, s_dtype):
    """§2 "Exactness": with integer-grid inputs every sum is exact, so the
    tile-by-tile step must equal the full-matrix step bit for bit."""
    T, N, K = 96, 256, 384
    X, dY = _grid_inputs(T, N, K, seed=kind)
    st = _state(N, K, w_dtype, s_dtype, kind)
    hp = opt.Hparams(lr=1e-3, weight_decay=0.01, momentum=0.9)
    full = ls.linear_bwd_step(X, dY, st, kind, hp, step=3, seed=77, want_dx=False)
    tiles = [(n0, k0) for n0 in range(0, N, 128) for k0 in range(0, K, 128)]
    parts = ls.linear_bwd_step_tiles(X, dY, st, kind, hp, 3, 77, tiles)
    for (n0, k0), r in parts.items():
        for key in ("W", "s1", "s2"):
            if full[key] is None:
                assert r[key] is None
                continue
            assert np.array_equal(full[key][n0:n0 + 128, k0:k0 + 128], r[key]), (key, n0, k0)
        for key in ("s1_scale", "s2_scale"):
            if full[key] is not None:
                assert np.array_equal(full[key][n0:n0 + 128, k0 // 64:(k0 + 128) // 64], r[key])


def test_gradient_is_consumed_in_fp32_not_bf16():
    """SGD with lr = 1 on an fp32 master weight exposes the gradient: bits below
    bf16 precision must survive (§2: never truncated to bf16)."""
    T, N, K = 3, 2, 64
    X = _bits(np.full((T, K), 1.0))
    dY = np.zeros((T, N), dtype=np.uint16)
    dY[:, 0] = _bits(np.array([1.0, 2.0 ** -9, 2.0 ** -9]))
    st = {"W": np.zeros((N, K), dtype=np.float32), "w_dtype": "fp32", "s_dtype": "fp32"}
    out = ls.linear_bwd_step(X, dY, st, opt.SGD, opt.Hparams(lr=1.0), 1, 0)
    assert np.all(out["W"][0] == np.float32(-(1.0 + 2.0 ** -8)))  # not representable in bf16
    assert rounding.bf16_bits_rne(np.float32(1.0 + 2.0 ** -8)) == 0x3F80


def test_dx_uses_pre_update_weights():
    T, N, K = 4, 3, 64
    rng = np.random.default_rng(8)
    X = _bits(rng.standard_normal((T, K)))
    dY = _bits(rng.standard_normal((T, N)))
    W = _bits(rng.standard_normal((N, K)) * 0.02)
    st = {"W": W, "w_dtype": "bf16", "s_dtype": "fp32"}
    out = ls.linear_bwd_step(X, dY, st, opt.SGD, opt.Hparams(lr=0.5), 1, 0)
    assert not np.array_equal(out["W"], W)
    assert np.array_equal(out["dX"], ls.input_gradient(dY, W))
    # an fp32 master weight feeds dX through its nearest bf16
    Wf = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    out = ls.linear_bwd_step(X, dY, {"W": Wf, "w_dtype": "fp32", "s_dtype": "fp32"},
                             opt.SGD, opt.Hparams(lr=0.5), 1, 0)
    assert np.array_equal(out["dX"], ls.input_gradient(dY, _bits(Wf)))


def test_int8_update_consumes_new_fp32_moments():
    """From zero INT8 state, step 1 of AdamW must move W exactly as with fp32
    states (the new moments are used before they are quantised), while the
    stored moments are the quantised ones."""
    T, N, K = 64, 128, 128
    rng = np.random.default_rng(12)
    X = _bits(rng.standard_normal((T, K)))
    dY = _bits(rng.standard_normal((T, N)) * 1e-3)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    hp = opt.Hparams(lr=1e-3, weight_decay=0.01)
    z8 = np.zeros((N, K), dtype=np.int8)
    zs = np.zeros((N, K // 64), dtype=np.float32)
    q = ls.linear_bwd_step(X, dY, {"W": W, "w_dtype": "fp32", "s_dtype": "int8", "s1": z8,
                                   "s2": z8.view(np.uint8), "s1_scale": zs, "s2_scale": zs},
                           opt.ADAMW, hp, 1, 0, want_dx=False)
    zf = np.zeros((N, K), dtype=np.float32)
    f = ls.linear_bwd_step(X, dY, {"W": W, "w_dtype": "fp32", "s_dtype": "fp32", "s1": zf,
                                   "s2": zf}, opt.ADAMW, hp, 1, 0, want_dx=False)
    assert np.array_equal(q["W"], f["W"])
    c, s = quant.quantize_blocks(f["s1"], signed=True)
    assert np.array_equal(q["s1"], c) and np.array_equal(q["s1_scale"], s)
    c, s = quant.quantize_blocks(f["s2"], signed=False)
    assert np.array_equal(q["s2"], c) and np.array_equal(q["s2_scale"], s)


def test_sr_keys_on_global_element_index():
    """Two tiles of one matrix draw different random bits; the same element in
    a tile and in the full matrix draws the same bits."""
    T, N, K = 8, 128, 256
    X, dY = _grid_inputs(T, N, K, seed=1)
    st = _state(N, K, "bf16", "fp32", opt.SGD)
    hp = opt.Hparams(lr=1e-3)
    full = ls.linear_bwd_step(X, dY, st, opt.SGD, hp, 2, 5, want_dx=False)
    part = ls.linear_bwd_step_tiles(X, dY, st, opt.SGD, hp, 2, 5, [(0, 128)])[(0, 128)]
    assert np.array_equal(full["W"][:, 128:], part["W"])
    other = ls.linear_bwd_step(X, dY, st, opt.SGD, hp, 3, 5, want_dx=False)
    assert not np.array_equal(full["W"], other["W"])
