"""Seeded random layers against the oracle, bit for bit.

Twenty configurations drawn from one seed: T in 1..1200, N and K multiples of 8
(half of them of 64) in 8..640 (and twelve with T up to 300, N and K up to 2560), one of the eight rules, one of the weight/state dtypes (and for INT8
states with bf16 weights one of the four block widths that divide K), with or
without dX.  Integer-grid inputs keep every FP32 sum exact, so W, the states and
the INT8 scales must equal the oracle's bit for bit, and dX must lie within its
tolerance.  The draws cover the one-launch and two-launch forms, ragged tiles on
both axes, tiny and partly filled pair tiles, and the split last wave.
"""

import numpy as np
import pytest

from optimizer_tcgen05_dw_gb300 import api, inputs
from optimizer_tcgen05_dw_gb300.build import build
from oracle import linear_step as ls

from _helpers import Problem, assert_bitexact, assert_dx_close, to_bits

pytestmark = pytest.mark.gpu

RULES = ["adamw", "nadam", "radam", "lion", "rmsprop", "adagrad", "sgd", "sgd_momentum"]
DTYPES = [("fp32", "fp32"), ("bf16", "fp32"), ("bf16", "int8"), ("bf16", "bf16"), ("fp32", "int8")]


def _draw(i, t_max=1200, nk_max=640):
    rng = np.random.default_rng(9000 + i)
    T = int(rng.integers(1, t_max + 1))
    align = 64 if rng.integers(0, 2) else 8  # half the draws take the one-launch form's alignment
    N = align * int(rng.integers(1, nk_max // align + 1))
    K = align * int(rng.integers(1, nk_max // align + 1))
    w_dtype, s_dtype = DTYPES[int(rng.integers(0, len(DTYPES)))]
    qblock = 64
    if s_dtype == "int8":
        widths = [b for b in (32, 64, 128, 256) if K % b == 0] if w_dtype == "bf16" else [64]
        if K % 64 != 0 and w_dtype == "fp32":
            s_dtype = "fp32"  # fp32 weights keep the block of 64, which needs K % 64 == 0
        elif not widths:
            K = 64 * max(1, K // 64)  # INT8 blocks need K to be a multiple of the width
            widths = [b for b in (32, 64, 128, 256) if K % b == 0] if w_dtype == "bf16" else [64]
        if s_dtype == "int8":
            qblock = int(widths[int(rng.integers(0, len(widths)))])
    rule = RULES[int(rng.integers(0, len(RULES)))]
    want_dx = bool(rng.integers(0, 2))
    return dict(T=T, N=N, K=K, w_dtype=w_dtype, s_dtype=s_dtype, qblock=qblock, rule=rule, want_dx=want_dx)


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    api.lib()
    api.forge_set_wait_limit_ns(200_000_000)
    api.forge_set_step_fusion(True)
    yield
    api.forge_set_wait_limit_ns(0)


@pytest.mark.parametrize("i", range(20))
def test_random_layer_bitexact_on_integer_grid(i):
    _check_draw(i, _draw(i))


@pytest.mark.parametrize("i", range(12))
def test_random_mid_layer_bitexact_on_integer_grid(i):
    """Wider layers (N, K up to 2560, T up to 300): up to 100 pair tiles, so the
    draws fall on all three tile schedules: every tile as two column halves
    (at most 38 tiles), whole tiles in one partial wave, and a split last wave."""
    _check_draw(100 + i, _draw(100 + i, t_max=300, nk_max=2560))


def _check_draw(i, c):
    hp = dict(inputs.SWEEP_HPARAMS[c["rule"]])
    hp.setdefault("weight_decay", 0.01)
    prob = Problem(T=c["T"], N=c["N"], K=c["K"], w_dtype=c["w_dtype"], s_dtype=c["s_dtype"],
                   opt_name=c["rule"], hp=hp, grid=True, steps=2, seed=9100 + i, qblock=c["qblock"])
    gpu, gdx = prob.run_gpu(fused=True, want_dx=c["want_dx"])
    ref, _, _ = prob.run_oracle(want_dx=c["want_dx"])
    what = f"{c} "
    assert_bitexact(gpu["W"], ref["W"], what + "W")
    for k in ("s1", "s2", "s1_scale", "s2_scale"):
        if ref.get(k) is not None:
            assert_bitexact(gpu[k], ref[k], what + k)
    if c["want_dx"]:
        assert_dx_close(gdx[0], to_bits(prob.dY[0]), ls.weights_for_dx(prob.state0["W"], c["w_dtype"]),
                        what + "dX")
