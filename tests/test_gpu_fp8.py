"""GPU parity of the FORGE step from E4M3 operands against the oracle.

The oracle (oracle/fp8.py) decodes the codes exactly, forms the gradient
S * c (S the exact sum of code products, c = x_scale * dy_scale rounded once
to float) and applies the same optimizer update as the BF16 path.  Integer
codes with power-of-two scales make every sum exact, so those cases must match
bit for bit; normally distributed codes are checked against the interval
oracle of _helpers.py with the FP32 summation bound of the tensor-core sum.
"""

import numpy as np
import pytest
import torch

from oracle import fp8
from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import quant, rounding
from optimizer_tcgen05_dw_gb300 import api, inputs
from optimizer_tcgen05_dw_gb300.build import build

from _helpers import Problem, assert_bitexact, assert_in_interval, oracle_hparams, oracle_interval

pytestmark = pytest.mark.gpu

OPTS = list(opt.NAMES)
SDTYPES = ["fp32", "int8", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    api.lib()
    api.forge_set_wait_limit_ns(200_000_000)
    yield
    api.forge_set_wait_limit_ns(0)


def _hp(name):
    hp = dict(inputs.SWEEP_HPARAMS[name])
    hp.setdefault("weight_decay", 0.01)
    return hp


def _codes_np(t):
    return t.cpu().numpy().astype(np.uint8)


def _run_fp8(prob, xts, dyts, sx, sdy, state=None):
    g = prob.gpu_state() if state is None else state
    for s in range(len(xts)):
        api.forge_linear_bwd_step_fp8(xts[s].cuda(), dyts[s].cuda(), sx, sdy, g["W"], prob.opt,
                                      prob.hp, s + 1, prob.seed, g.get("s1"), g.get("s2"),
                                      g.get("s1_scale"), g.get("s2_scale"))
    api.forge_get_device_status()
    torch.cuda.synchronize()
    return g


def _oracle_fp8(prob, xts, dyts, sx, sdy):
    st = dict(prob.state0)
    hp = oracle_hparams(prob.hp)
    for s in range(len(xts)):
        g = fp8.weight_gradient_fp8(_codes_np(xts[s]), _codes_np(dyts[s]), sx, sdy)
        out = ls.update_block(prob.kind, hp, s + 1, prob.seed, g, st["W"], "bf16", st.get("s1"),
                              st.get("s2"), st.get("s1_scale"), st.get("s2_scale"), prob.s_dtype,
                              0, 0, prob.K)
        st.update({k: out[k] for k in ("W", "s1", "s2", "s1_scale", "s2_scale")})
    return st


def _grid_inputs(T, N, K, steps, seed):
    xts = [inputs.e4m3_integer_grid((K, T), -4, 4, inputs.layer_seed(seed, 0, s, 11)) for s in range(steps)]
    dyts = [inputs.e4m3_integer_grid((N, T), -4, 4, inputs.layer_seed(seed, 0, s, 12)) for s in range(steps)]
    return xts, dyts


def _compare_exact(gpu, ref):
    assert_bitexact(gpu["W"], ref["W"], "W")
    for k in ("s1", "s2", "s1_scale", "s2_scale"):
        if ref.get(k) is not None:
            assert_bitexact(gpu[k], ref[k], k)


# T % 128 != 0 (a ragged token stage), N % 256 and K % 256 != 0 (ragged tiles)
GRID = dict(T=208, N=320, K=384)


@pytest.mark.parametrize("opt_name", OPTS)
@pytest.mark.parametrize("s_dtype", SDTYPES)
def test_fp8_step_bitexact_on_integer_grid(opt_name, s_dtype):
    """Integer codes, power-of-two scales: S and S * c are exact, so two
    consecutive steps match the oracle bit for bit (weights by stochastic
    rounding, moments in every storage)."""
    prob = Problem(**GRID, w_dtype="bf16", s_dtype=s_dtype, opt_name=opt_name, hp=_hp(opt_name),
                   steps=1, seed=21)
    xts, dyts = _grid_inputs(GRID["T"], GRID["N"], GRID["K"], 2, 21)
    sx, sdy = 2.0 ** -3, 2.0 ** -12
    gpu = _run_fp8(prob, xts, dyts, sx, sdy)
    _compare_exact(gpu, _oracle_fp8(prob, xts, dyts, sx, sdy))


@pytest.mark.parametrize("shape", [dict(T=16, N=256, K=256), dict(T=128, N=264, K=200),
                                   dict(T=400, N=8, K=8), dict(T=1040, N=520, K=264)],
                         ids=["one_stage", "ragged_rows_cols", "single_group", "many_stages"])
@pytest.mark.parametrize("s_dtype", ["fp32", "bf16"])
def test_fp8_step_edge_shapes_bitexact(shape, s_dtype):
    prob = Problem(**shape, w_dtype="bf16", s_dtype=s_dtype, opt_name="adamw", hp=_hp("adamw"),
                   steps=1, seed=22)
    xts, dyts = _grid_inputs(shape["T"], shape["N"], shape["K"], 1, 22)
    gpu = _run_fp8(prob, xts, dyts, 2.0 ** -2, 2.0 ** -14)
    _compare_exact(gpu, _oracle_fp8(prob, xts, dyts, 2.0 ** -2, 2.0 ** -14))


def test_fp8_step_no_tokens_is_the_rule_on_a_zero_gradient():
    prob = Problem(T=0, N=256, K=320, w_dtype="bf16", s_dtype="int8", opt_name="adamw",
                   hp=_hp("adamw"), steps=1, seed=23)
    empty = torch.empty((320, 0), dtype=torch.uint8), torch.empty((256, 0), dtype=torch.uint8)
    gpu = _run_fp8(prob, [empty[0]], [empty[1]], 1.0, 1.0)
    _compare_exact(gpu, _oracle_fp8(prob, [empty[0]], [empty[1]], 1.0, 1.0))


def test_fp8_non_power_of_two_scales_bitexact():
    """c = RN32(x_scale * dy_scale) and g = RN32(S * c): scales with full
    mantissas exercise both roundings."""
    prob = Problem(T=208, N=320, K=384, w_dtype="bf16", s_dtype="fp32", opt_name="sgd_momentum",
                   hp=_hp("sgd_momentum"), steps=1, seed=24)
    xts, dyts = _grid_inputs(208, 320, 384, 2, 24)
    sx, sdy = 0.0123456789, 3.3e-4
    gpu = _run_fp8(prob, xts, dyts, sx, sdy)
    _compare_exact(gpu, _oracle_fp8(prob, xts, dyts, sx, sdy))


def _fp8_error_bound(xt, dyt, sx, sdy):
    """|g_gpu - g_exact| bound for the tensor-core sum of T E4M3 products:
    ceil(T/32) FP32 accumulator updates (32 products per instruction), each
    off by at most 2^-23 of a partial sum no larger than 3x the random-walk
    scale sqrt(sum_t (dY X)^2), then the rounding of S and of S * c."""
    table = fp8.e4m3_bits_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    X, dY = table[xt], table[dyt]
    T = X.shape[1]
    rw = np.sqrt((dY * dY) @ (X * X).T)
    S = dY @ X.T
    c = float(fp8.grad_scale(sx, sdy))
    return c * (2.0 ** -23 * np.ceil(T / 32.0) * 3.0 * rw + 2.0 ** -23 * np.abs(S)) + 1e-30, S * c


def test_fp8_gradient_within_the_summation_bound():
    """SGD-momentum from a zero buffer with fp32 states stores g itself
    (m = 0.9 * 0 + g): the tensor-core sum of realistic codes must be within
    the FP32 summation bound of the exact one."""
    T, N, K = 2048, 512, 640
    xt, sx = inputs.e4m3_normal((K, T), 1.0, 31)
    dyt, sdy = inputs.e4m3_normal((N, T), 1e-3, 32)
    prob = Problem(T=16, N=N, K=K, w_dtype="bf16", s_dtype="fp32", opt_name="sgd_momentum",
                   hp=dict(lr=1e-2, momentum=0.9), steps=1, seed=25)
    st = prob.gpu_state()
    st["s1"].zero_()
    api.forge_linear_bwd_step_fp8(xt.cuda(), dyt.cuda(), sx, sdy, st["W"], "sgd_momentum",
                                  dict(lr=1e-2, momentum=0.9), 1, 25, st["s1"])
    api.forge_get_device_status()
    got = st["s1"].cpu().numpy().astype(np.float64)
    bound, exact = _fp8_error_bound(_codes_np(xt), _codes_np(dyt), sx, sdy)
    ratio = np.abs(got - exact) / bound
    assert ratio.max() <= 1.0, f"max |g - exact| / bound = {ratio.max():.3f}"


@pytest.mark.parametrize("opt_name,s_dtype", [("adamw", "fp32"), ("adamw", "int8"),
                                              ("adamw", "bf16"), ("lion", "fp32"),
                                              ("rmsprop", "int8")])
def test_fp8_step_realistic_interval(opt_name, s_dtype):
    """Normally distributed codes (per-tensor power-of-two scales, as a
    quantiser would pick): every output within the oracle's interval."""
    T, N, K = 1024, 512, 768
    xt, sx = inputs.e4m3_normal((K, T), 1.0, 41)
    dyt, sdy = inputs.e4m3_normal((N, T), 1e-3, 42)
    prob = Problem(T=16, N=N, K=K, w_dtype="bf16", s_dtype=s_dtype, opt_name=opt_name,
                   hp=_hp(opt_name), steps=1, seed=26)
    gpu = _run_fp8(prob, [xt], [dyt], sx, sdy)
    delta, g = _fp8_error_bound(_codes_np(xt), _codes_np(dyt), sx, sdy)
    iv = oracle_interval(prob.kind, oracle_hparams(prob.hp), 1, prob.seed, g.astype(np.float32),
                         prob.state0, "bf16", s_dtype, 0, 0, K, delta)
    assert_in_interval(gpu, iv, "bf16", s_dtype, "fp8 step")


def test_fp8_q_proj_full_size_sampled_rows():
    """The Llama-3.1-8B q_proj (4096 x 4096) at T = 16384 from E4M3 codes,
    INT8 AdamW moments: the whole layer is stepped on the GPU; 256 sampled
    rows (whole rows, so their INT8 blocks are complete) must lie in the
    oracle's interval."""
    T, N, K = 16384, 4096, 4096
    xt, sx = inputs.e4m3_normal((K, T), 1.0, 51)
    dyt, sdy = inputs.e4m3_normal((N, T), 1e-3, 52)
    kind = opt.ADAMW
    hp = dict(inputs.ADAMW_LLAMA)
    W = rounding.bf16_bits_rne(inputs.normal((N, K), 0.02, 53, torch.float32).numpy())
    m, sm = quant.quantize_blocks(inputs.normal((N, K), 1e-4, 54, torch.float32).numpy(), True)
    v, sv = quant.quantize_blocks(inputs.abs_normal((N, K), 1e-6, 55).numpy(), False)
    dev = {"W": inputs.bits_to_bf16(W).cuda(), "s1": torch.from_numpy(m).cuda(),
           "s2": torch.from_numpy(v).cuda(), "s1_scale": torch.from_numpy(sm).cuda(),
           "s2_scale": torch.from_numpy(sv).cuda()}
    api.forge_linear_bwd_step_fp8(xt.cuda(), dyt.cuda(), sx, sdy, dev["W"], "adamw", hp, 3, 57,
                                  dev["s1"], dev["s2"], dev["s1_scale"], dev["s2_scale"])
    api.forge_get_device_status()
    rows = np.sort(np.random.default_rng(58).choice(N, 256, replace=False))
    rows[0], rows[-1] = 0, N - 1
    xc, dyc = _codes_np(xt), _codes_np(dyt)[rows]
    delta, g = _fp8_error_bound(xc, dyc, sx, sdy)
    st = {"W": W[rows], "s1": m[rows], "s2": v[rows], "s1_scale": sm[rows], "s2_scale": sv[rows]}
    sub = {k: dev[k][torch.from_numpy(rows).cuda()] for k in dev}
    _check_rows(sub, rows, K, kind, hp, g, delta, st)


def _check_rows(sub, rows, K, kind, hp, g, delta, st):
    """oracle_interval keys stochastic rounding by the element index n*K + k
    of its block; for scattered rows it runs row by row with n0 = the row."""
    outs_rows = []
    for i, r in enumerate(rows):
        blk = {k: st[k][i:i + 1] for k in st}
        outs_rows.append(oracle_interval(kind, oracle_hparams(hp), 3, 57, g[i:i + 1].astype(np.float32),
                                         blk, "bf16", "int8", int(r), 0, K, delta[i:i + 1]))
    outs = [{k: (None if o0[k] is None else np.concatenate([o[0][j][k] for o in outs_rows]))
             for k in o0} for j, o0 in enumerate(outs_rows[0][0])]
    fp32 = [{k: (None if f0[k] is None else np.concatenate([o[1][j][k] for o in outs_rows]))
             for k in f0} for j, f0 in enumerate(outs_rows[0][1])]
    assert_in_interval(sub, (outs, fp32), "bf16", "int8", "q_proj fp8 sampled rows")


@pytest.mark.parametrize("s_dtype", ["fp32", "int8"])
def test_fp8_nan_codes_propagate(s_dtype):
    """E4M3 has no infinity; its NaN codes (0x7F, 0xFF) make the columns they
    sit in NaN in the gradient, and the updated weights there NaN (0x7FC0),
    exactly as the oracle's decoding does."""
    prob = Problem(**GRID, w_dtype="bf16", s_dtype=s_dtype, opt_name="adamw", hp=_hp("adamw"),
                   steps=1, seed=27)
    xts, dyts = _grid_inputs(GRID["T"], GRID["N"], GRID["K"], 1, 27)
    xt = xts[0].clone()
    xt[10, 3] = 0x7F
    xt[300, 100] = 0xFF
    xts = [xt]
    gpu = _run_fp8(prob, xts, dyts, 2.0 ** -3, 2.0 ** -12)
    ref = _oracle_fp8(prob, xts, dyts, 2.0 ** -3, 2.0 ** -12)
    _compare_exact(gpu, ref)
    assert (ref["W"][:, 10] == 0x7FC0).all() and (ref["W"][:, 300] == 0x7FC0).all()


@pytest.mark.parametrize("s_dtype", ["fp32", "int8"])
def test_fp8_split_last_wave_bitexact(s_dtype):
    """80 pair tiles on 76 pairs: the last partial wave runs as 128-column
    halves (64-row boxes of X^T); bit-exact against the oracle."""
    T, N, K = 160, 2560, 2048
    prob = Problem(T=16, N=N, K=K, w_dtype="bf16", s_dtype=s_dtype, opt_name="adamw", hp=_hp("adamw"),
                   steps=1, seed=28)
    xts, dyts = _grid_inputs(T, N, K, 1, 28)
    gpu = _run_fp8(prob, xts, dyts, 2.0 ** -3, 2.0 ** -12)
    _compare_exact(gpu, _oracle_fp8(prob, xts, dyts, 2.0 ** -3, 2.0 ** -12))
