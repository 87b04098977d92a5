"""CPU self-test of the interval tolerance used by the GPU parity tests.

A simulated device result is the oracle's own step at a gradient perturbed by
at most the summation bound d (what a different summation order can do): it
must pass.  Results with a planted error (3 ULP on the weights, one INT8 code
step beyond rounding, a wrong scale) must fail.  The mistakes are planted in
oracle outputs on the CPU; no GPU is involved.
"""

import numpy as np
import pytest
import torch

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import quant, rounding
from optimizer_tcgen05_dw_gb300 import inputs

from _helpers import assert_in_interval, grad_error_bound, oracle_interval


def _case(kind, s_dtype, seed=5, T=2048, N=128, K=128):
    X = inputs.bf16_to_bits(inputs.normal((T, K), 1.0, seed))
    dY = inputs.bf16_to_bits(inputs.normal((T, N), 1e-3, seed + 1))
    W = rounding.bf16_bits_rne(inputs.normal((N, K), 0.02, seed + 2, torch.float32).numpy())
    m = inputs.normal((N, K), 1e-4, seed + 3, torch.float32).numpy()
    v = inputs.abs_normal((N, K), 1e-6, seed + 4).numpy()
    st = {"W": W}
    if opt.USES_S1[kind]:
        if s_dtype == "int8":
            st["s1"], st["s1_scale"] = quant.quantize_blocks(m, True)
        elif s_dtype == "bf16":
            st["s1"] = rounding.bf16_bits_rne(m)
        else:
            st["s1"] = m
    if opt.USES_S2[kind]:
        if s_dtype == "int8":
            st["s2"], st["s2_scale"] = quant.quantize_blocks(v, False)
        elif s_dtype == "bf16":
            st["s2"] = rounding.bf16_bits_rne(v)
        else:
            st["s2"] = v
    g = ls.weight_gradient(X, dY)
    d = grad_error_bound(X, dY)
    hp = opt.Hparams(**inputs.SWEEP_HPARAMS[opt.NAMES[kind]])
    iv = oracle_interval(kind, hp, 2, 9, g, st, "bf16", s_dtype, 0, 0, K, d)
    rng = np.random.default_rng(seed)
    g_sim = (g.astype(np.float64) + rng.uniform(-1, 1, g.shape) * d).astype(np.float32)
    sim = ls.update_block(kind, hp, 2, 9, g_sim, st["W"], "bf16", st.get("s1"), st.get("s2"),
                          st.get("s1_scale"), st.get("s2_scale"), s_dtype, 0, 0, K)
    sim = {k: torch.from_numpy(np.ascontiguousarray(v if k != "W" else v.view(np.int16))).view(
        torch.bfloat16) if k == "W" else torch.from_numpy(np.ascontiguousarray(v))
        for k, v in sim.items() if v is not None}
    return iv, sim


@pytest.mark.parametrize("kind", range(8), ids=opt.NAMES)
@pytest.mark.parametrize("s_dtype", ["fp32", "int8", "bf16"])
def test_perturbed_gradient_passes(kind, s_dtype):
    iv, sim = _case(kind, s_dtype)
    assert_in_interval(sim, iv, "bf16", s_dtype, "simulated")


def test_planted_weight_error_fails():
    iv, sim = _case(opt.ADAMW, "fp32")
    bits = inputs.bf16_to_bits(sim["W"]).astype(np.int32)
    bits[5, 7] += 3 if bits[5, 7] & 0x7FFF < 0x7F00 else -3
    sim["W"] = inputs.bits_to_bf16(bits.astype(np.uint16))
    with pytest.raises(AssertionError):
        assert_in_interval(sim, iv, "bf16", "fp32", "planted")


def test_planted_bf16_state_error_fails():
    iv, sim = _case(opt.ADAMW, "bf16")
    bits = sim["s2"].numpy().astype(np.int32)
    bits[2, 9] += 3
    with pytest.raises(AssertionError):
        assert_in_interval(dict(sim, s2=torch.from_numpy(bits.astype(np.uint16))), iv, "bf16", "bf16",
                           "planted bf16 v")


def test_planted_state_errors_fail():
    iv, sim = _case(opt.ADAMW, "fp32")
    sim["s1"] = sim["s1"].clone()
    sim["s1"][3, 3] *= 1.001
    with pytest.raises(AssertionError):
        assert_in_interval(sim, iv, "bf16", "fp32", "planted m")
    iv, sim = _case(opt.ADAMW, "int8")
    bad = sim["s1"].clone()
    bad[0, 0] = 100 if int(bad[0, 0]) < 0 else -100
    with pytest.raises(AssertionError):
        assert_in_interval(dict(sim, s1=bad), iv, "bf16", "int8", "planted code")
    sc = sim["s2_scale"].clone()
    sc[1, 1] *= 1.01
    with pytest.raises(AssertionError):
        assert_in_interval(dict(sim, s2_scale=sc), iv, "bf16", "int8", "planted scale")
