"""State variants of the oracle (the quantiser variants the pages point to).

BF16 moments: the rule runs in FP32 on the widened moments and the new
moments are stored rounded to nearest even; the weight update is the one the
same FP32 moments give.  Pinned by composition with the FP32-state step and by
the rounding pin (the nearest-even conversion equals torch's float->bfloat16
cast, tests/test_oracle_philox_rounding.py), plus a closed form.

Block size: the explainer (Technical Summary §2, "Precision and Fidelity")
says INT8 states use blocks of 64 rather than the 2048 of standard 8-bit
optimizers, to keep quantisation error small.  Checked on synthetic moments
with a few large channels (1 % of the columns at 100x scale), and over a short
AdamW trajectory against FP32 states.
"""

import numpy as np
import pytest
import torch

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import quant, rounding
from optimizer_tcgen05_dw_gb300 import inputs

RULES_WITH_STATE = [k for k in range(8) if opt.USES_S1[k] or opt.USES_S2[k]]


@pytest.mark.parametrize("kind", RULES_WITH_STATE, ids=[opt.NAMES[k] for k in RULES_WITH_STATE])
def test_bf16_moments_are_the_fp32_step_rounded(kind):
    rng = np.random.default_rng(100 + kind)
    R, C = 16, 128
    g = (rng.standard_normal((R, C)) * 1e-2).astype(np.float32)
    W = rounding.bf16_bits_rne((rng.standard_normal((R, C)) * 0.02).astype(np.float32))
    m_bits = rounding.bf16_bits_rne((rng.standard_normal((R, C)) * 1e-3).astype(np.float32))
    v_bits = rounding.bf16_bits_rne(np.abs(rng.standard_normal((R, C)) * 1e-5).astype(np.float32))
    hp = opt.Hparams(**inputs.SWEEP_HPARAMS[opt.NAMES[kind]])
    bf = ls.update_block(kind, hp, 3, 9, g, W, "bf16", m_bits, v_bits, s_dtype="bf16", K=C)
    f32 = ls.update_block(kind, hp, 3, 9, g, W, "bf16", rounding.bf16_bits_to_f32(m_bits),
                          rounding.bf16_bits_to_f32(v_bits), s_dtype="fp32", K=C)
    assert np.array_equal(bf["W"], f32["W"])
    for key in ("s1", "s2"):
        if f32[key] is None:
            assert bf[key] is None
            continue
        assert bf[key].dtype == np.uint16
        assert np.array_equal(bf[key], rounding.bf16_bits_rne(f32[key]))


def test_bf16_momentum_closed_form():
    """SGD-momentum from a zero buffer: b = g, stored as bf16(g) (torch's cast)."""
    rng = np.random.default_rng(7)
    g = (rng.standard_normal((8, 64)) * 3e-3).astype(np.float32)
    W = rounding.bf16_bits_rne(np.zeros((8, 64), np.float32))
    zero = np.zeros((8, 64), np.uint16)
    out = ls.update_block(opt.SGD_MOMENTUM, opt.Hparams(lr=1e-2, momentum=0.9), 1, 0, g, W, "bf16",
                          zero, None, s_dtype="bf16", K=64)
    want = torch.from_numpy(g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out["s1"], want)


def _channel_scale(cols, seed, factor=100.0):
    """Per-column scale with a few large channels: 1 % of the columns `factor`x."""
    rng = np.random.default_rng(seed)
    return np.where(rng.random(cols) < 0.01, factor, 1.0).astype(np.float32)


def test_block64_quantises_more_accurately_than_block2048():
    """Normalised RMS error of the ordinary columns: a block of 2048 almost
    always holds a large channel, whose absmax sets a step the ordinary values
    fall under; a block of 64 mostly does not."""
    rows, cols = 32, 4096
    scale = _channel_scale(cols, 11)
    rng = np.random.default_rng(12)
    m = (rng.standard_normal((rows, cols)) * scale * 1e-3).astype(np.float32)
    v = ((rng.standard_normal((rows, cols)) * scale * 1e-3) ** 2).astype(np.float32)
    ordinary = scale == 1.0
    for x, signed in ((m, True), (v, False)):
        err = {}
        for block in (64, 2048):
            codes, amax = quant.quantize_blocks(x, signed, block=block)
            back = quant.dequantize_blocks(codes, amax, signed, block=block)
            err[block] = float(np.sqrt(np.mean((back - x)[:, ordinary] ** 2) /
                                       np.mean(x[:, ordinary] ** 2)))
        assert err[64] < 0.6 * err[2048], (signed, err)


def test_block64_trajectory_tracks_fp32_states_closer_than_block2048():
    """Ten AdamW steps with INT8 moments at block 64 and at block 2048, against
    the same steps with FP32 moments: the block-64 weights stay much closer.
    (With the linear code both drift: a second moment far below its block's
    absmax rounds to code 0, and its update is then bounded only by eps.)"""
    rng = np.random.default_rng(5)
    R, C = 16, 4096
    scale = _channel_scale(C, 5, factor=10.0)
    W0 = (rng.standard_normal((R, C)) * 0.02).astype(np.float32)
    hp = opt.Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    state = {"fp32": (W0, np.zeros((R, C), np.float32), np.zeros((R, C), np.float32), None, None)}
    zc = (np.zeros((R, C), np.int8), np.zeros((R, C), np.uint8))
    for blk in (64, 2048):
        state[blk] = (W0, zc[0], zc[1], np.zeros((R, C // blk), np.float32),
                      np.zeros((R, C // blk), np.float32))
    for step in range(1, 11):
        g = (rng.standard_normal((R, C)) * scale * 1e-3).astype(np.float32)
        for key in list(state):
            W, s1, s2, a1, a2 = state[key]
            if key == "fp32":
                out = ls.update_block(opt.ADAMW, hp, step, 0, g, W, "fp32", s1, s2, K=C)
            else:
                out = ls.update_block(opt.ADAMW, hp, step, 0, g, W, "fp32", s1, s2, a1, a2,
                                      s_dtype="int8", K=C, block=key)
            state[key] = (out["W"], out["s1"], out["s2"], out["s1_scale"], out["s2_scale"])
    ref = state["fp32"][0].astype(np.float64)
    d64 = np.sqrt(np.mean((state[64][0] - ref) ** 2))
    d2048 = np.sqrt(np.mean((state[2048][0] - ref) ** 2))
    assert d64 < 0.3 * d2048, (d64, d2048)
