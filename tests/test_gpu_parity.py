"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Sizes span several 128 x 256 output tiles, a ragged edge in every dimension
(T % 64, N % 128, K % 256 all nonzero), and the edge cases the method has (no
tokens, a single 8-wide column group, rules without state).  Full-size layers
of the benchmark workloads are checked on sampled tiles in
test_gpu_fullsize.py.
"""

import numpy as np
import pytest
import torch

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import philox as oph
from oracle import quant
from optimizer_tcgen05_dw_gb300 import api, inputs
from optimizer_tcgen05_dw_gb300.build import build

from _helpers import (Problem, assert_bf16_close, assert_bitexact, assert_dx_close,
                      assert_fp32_close, oracle_hparams, to_bits)

pytestmark = pytest.mark.gpu

OPTS = list(opt.NAMES)
DTYPES = [("fp32", "fp32"), ("bf16", "fp32"), ("bf16", "int8"), ("bf16", "bf16")]
RAGGED = dict(T=200, N=264, K=320)     # dX as its own launch (N % 64 != 0)
RAGGED64 = dict(T=200, N=320, K=384)   # dX and the step in one launch


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    api.lib()
    api.forge_set_wait_limit_ns(200_000_000)  # any legitimate wait here is far shorter
    api.forge_debug_skip_loads(False)
    yield
    api.forge_set_wait_limit_ns(0)


def _hp(name, wd=True):
    hp = dict(inputs.SWEEP_HPARAMS[name])
    if wd and "weight_decay" not in hp:
        hp["weight_decay"] = 0.01  # exercises the L2 path of the coupled rules
    return hp


def _compare_exact(prob, gpu, ref):
    assert_bitexact(gpu["W"], ref["W"], "W")
    for k in ("s1", "s2", "s1_scale", "s2_scale"):
        if ref.get(k) is not None:
            assert_bitexact(gpu[k], ref[k], k)


# --------------------------------------------------------------- exact inputs

@pytest.mark.parametrize("shape", [RAGGED, RAGGED64], ids=["two_launch", "one_launch"])
@pytest.mark.parametrize("opt_name", OPTS)
@pytest.mark.parametrize("w_dtype,s_dtype", DTYPES)
def test_fused_step_bitexact_on_integer_grid(opt_name, w_dtype, s_dtype, shape):
    """Integer-grid X and dY make every FP32 sum exact, so the tensor-core
    gradient equals the oracle's and the fused step must match bit for bit:
    optimizer, stochastic rounding and INT8 requantisation included.  With
    bf16 weights and 64-aligned N, K the dX tiles run in the same launch."""
    prob = Problem(**shape, w_dtype=w_dtype, s_dtype=s_dtype, opt_name=opt_name,
                   hp=_hp(opt_name), grid=True, steps=3, seed=11)
    gpu, gdx = prob.run_gpu(fused=True, want_dx=True)
    ref, rdx, _ = prob.run_oracle(want_dx=True)
    _compare_exact(prob, gpu, ref)
    # dX of step 1 comes from the initial (pre-update) weights
    assert_dx_close(gdx[0], to_bits(prob.dY[0]), ls.weights_for_dx(prob.state0["W"], w_dtype), "dX")


@pytest.mark.parametrize("w_dtype,s_dtype", DTYPES)
def test_radam_rectified_branch_bitexact(w_dtype, s_dtype):
    """Seven steps cross RAdam's rectification threshold (rho_t > 5 from step 6)."""
    prob = Problem(T=128, N=136, K=192, w_dtype=w_dtype, s_dtype=s_dtype, opt_name="radam",
                   hp=_hp("radam"), grid=True, steps=7, seed=14)
    gpu, _ = prob.run_gpu(fused=True)
    ref, _, _ = prob.run_oracle()
    _compare_exact(prob, gpu, ref)


@pytest.mark.parametrize("opt_name", ["adamw", "lion", "sgd_momentum", "adagrad"])
@pytest.mark.parametrize("w_dtype,s_dtype", DTYPES)
def test_unfused_schedule_bitexact_on_integer_grid(opt_name, w_dtype, s_dtype):
    """The two-pass schedule (fp32 dW in global memory, then the optimizer
    kernel) computes the same result as the oracle on exact inputs."""
    prob = Problem(**RAGGED, w_dtype=w_dtype, s_dtype=s_dtype, opt_name=opt_name,
                   hp=_hp(opt_name), grid=True, steps=2, seed=12)
    gpu, _ = prob.run_gpu(fused=False)
    ref, _, _ = prob.run_oracle()
    _compare_exact(prob, gpu, ref)


def test_unfused_wgrad_equals_exact_gradient():
    prob = Problem(**RAGGED, w_dtype="fp32", s_dtype="fp32", opt_name="sgd", hp={"lr": 1e-2},
                   grid=True, steps=1, seed=13)
    dW = torch.empty((prob.N, prob.K), dtype=torch.float32, device="cuda")
    api.forge_unfused_wgrad(prob.X[0].cuda(), prob.dY[0].cuda(), dW)
    torch.cuda.synchronize()
    assert_bitexact(dW, ls.weight_gradient(to_bits(prob.X[0]), to_bits(prob.dY[0])), "dW")


@pytest.mark.parametrize("shape", [dict(T=200, N=264, K=320), dict(T=1000, N=256, K=648),
                                   dict(T=4096, N=1024, K=1024)],
                         ids=["small_grid", "full_grid", "long_dx"])
def test_fp32_master_dx_every_step(shape):
    """fp32 master weights with dX: the dX kernel (32 x 32 tiles split four
    ways on a small grid, 64 x 64 tiles once the grid fills the GPU, several
    waves of them in `long_dx`) and the step that starts while it runs.  Every
    step's dX must come from that step's pre-update weights, and the update
    must still match bit for bit."""
    prob = Problem(**shape, w_dtype="fp32", s_dtype="fp32", opt_name="adamw", hp=_hp("adamw"),
                   grid=True, steps=3, seed=17)
    gpu, gdx = prob.run_gpu(fused=True, want_dx=True)
    ref, _, _ = prob.run_oracle(want_dx=True)
    _compare_exact(prob, gpu, ref)
    for s in range(prob.steps):
        assert_dx_close(gdx[s], to_bits(prob.dY[s]), ls.weights_for_dx(prob.w_before[s], "fp32"),
                        f"dX step {s + 1}")


# --------------------------------------------------------------- realistic data

def test_single_layer_fp32_master_config():
    """256 x 256 fp32 master weights, T = 512, AdamW, 3 steps, with dX."""
    w = inputs.WORKLOADS["single_256"]
    _, N, K = w.linears[0]
    prob = Problem(w.T, N, K, w.w_dtype, w.s_dtype, w.opt, w.hparams, seed=1000, steps=w.steps,
                   x_std=w.x_std, dy_std=w.dy_std, w_std=w.w_std, m_std=0.0, v_std=0.0)
    # moments start at zero in this workload
    prob.state0["s1"] = np.zeros((N, K), dtype=np.float32)
    prob.state0["s2"] = np.zeros((N, K), dtype=np.float32)
    prob.per_step_from_common_state()
    gpu, gdx = prob.run_gpu(fused=True, want_dx=True)
    ref, rdx, sens = prob.run_oracle(want_dx=True)
    assert sens.mean() < 1e-3
    assert_fp32_close(gpu["W"], ref["W"], "W (free-running)", exclude=sens)
    assert_fp32_close(gpu["s1"], ref["s1"], "m (free-running)", exclude=sens)
    assert_fp32_close(gpu["s2"], ref["s2"], "v (free-running)", exclude=sens)
    assert_dx_close(gdx[0], to_bits(prob.dY[0]), ls.weights_for_dx(prob.state0["W"], "fp32"), "dX")


@pytest.mark.parametrize("opt_name", OPTS)
def test_optimizer_sweep_realistic(opt_name):
    """bf16 weights with stochastic rounding, fp32 states, every rule, the
    sweep's hyper-parameters, X ~ N(0,1), dY ~ N(0,1e-3)."""
    prob = Problem(T=576, N=384, K=512, w_dtype="bf16", s_dtype="fp32", opt_name=opt_name,
                   hp=inputs.SWEEP_HPARAMS[opt_name], seed=4000 + OPTS.index(opt_name), steps=3)
    prob.per_step_from_common_state()      # each step: GPU inside the oracle's interval
    gpu, _ = prob.run_gpu(fused=True)      # free-running trajectory
    ref, _, sens = prob.run_oracle()
    assert_bf16_close(gpu["W"], ref["W"], "W (3 free-running steps)", exclude=sens, free_running=True)


@pytest.mark.parametrize("opt_name", ["adamw", "nadam", "lion", "rmsprop"])
def test_bf16_moments_realistic(opt_name):
    """bf16 weights and bf16 moments (nearest even), realistic data, 3 steps
    each inside the oracle's interval from a common state."""
    prob = Problem(T=576, N=384, K=512, w_dtype="bf16", s_dtype="bf16", opt_name=opt_name,
                   hp=inputs.SWEEP_HPARAMS[opt_name], seed=4100 + OPTS.index(opt_name), steps=3)
    prob.per_step_from_common_state()


def test_int8_states_realistic():
    """bf16 weights, INT8 block-64 AdamW moments pre-warmed from N(0,1e-4) and
    |N(0,1e-6)|, the Llama hyper-parameters, 3 steps."""
    w = inputs.WORKLOADS["llama8b_bf16_int8state"]
    prob = Problem(T=512, N=392, K=576, w_dtype="bf16", s_dtype="int8", opt_name="adamw",
                   hp=w.hparams, seed=3000, steps=3, m_std=w.m_init_std, v_std=w.v_init_std)
    prob.per_step_from_common_state()
    gpu, _ = prob.run_gpu(fused=True)
    ref, _, sens = prob.run_oracle()
    assert_bf16_close(gpu["W"], ref["W"], "W (free-running)", exclude=sens, free_running=True)


# --------------------------------------------------------------- equal FP32 inputs

@pytest.mark.parametrize("opt_name", OPTS)
@pytest.mark.parametrize("w_dtype,s_dtype", DTYPES)
def test_optimizer_kernel_bitexact_given_oracle_gradient(opt_name, w_dtype, s_dtype):
    """With the oracle's own float32 gradient as input, the per-element
    arithmetic (rule, stochastic rounding, INT8 code) must match bit for bit."""
    prob = Problem(T=64, N=136, K=192, w_dtype=w_dtype, s_dtype=s_dtype, opt_name=opt_name,
                   hp=_hp(opt_name), seed=21, steps=1)
    g = ls.weight_gradient(to_bits(prob.X[0]), to_bits(prob.dY[0]))
    gpu = prob.gpu_state()
    api.forge_unfused_opt_step(torch.from_numpy(g).cuda(), gpu["W"], opt_name, prob.hp, 7, 99,
                               gpu.get("s1"), gpu.get("s2"), gpu.get("s1_scale"), gpu.get("s2_scale"))
    api.forge_get_device_status()
    st = prob.state0
    ref = ls.update_block(prob.kind, oracle_hparams(prob.hp), 7, 99, g, st["W"], w_dtype,
                          st.get("s1"), st.get("s2"), st.get("s1_scale"), st.get("s2_scale"),
                          s_dtype, 0, 0, prob.K)
    _compare_exact(prob, gpu, ref)


@pytest.mark.parametrize("signed", [True, False])
def test_quantize_dequantize_bitexact(signed):
    rows, cols = 136, 320
    x = inputs.normal((rows, cols), 1e-3, 5, torch.float32)
    if not signed:
        x = x.abs()
    x[3, 64:128] = 0.0
    xg = x.cuda()
    codes = torch.empty((rows, cols), dtype=torch.int8 if signed else torch.uint8, device="cuda")
    amax = torch.empty((rows, cols // 64), dtype=torch.float32, device="cuda")
    api.forge_quantize_state(xg, codes, amax, signed)
    back = torch.empty_like(xg)
    api.forge_dequantize_state(codes, amax, back, signed)
    torch.cuda.synchronize()
    rc, ra = quant.quantize_blocks(x.numpy(), signed)
    assert_bitexact(codes, rc, "codes")
    assert_bitexact(amax, ra, "absmax")
    assert_bitexact(back, quant.dequantize_blocks(rc, ra, signed), "dequantised")


def test_device_philox_matches_oracle_and_curand():
    import ctypes
    from optimizer_tcgen05_dw_gb300.build import lib_path
    tk = ctypes.CDLL(lib_path("libforge_testkit.so"))
    rng = np.random.default_rng(17)
    n = 4096
    q = rng.integers(0, 2 ** 32, size=(n, 6), dtype=np.uint64).astype(np.uint32)
    q[:, 1] >>= 2  # cuRAND reaches counter words (0, 1) through skipahead(4 * ctr), 64-bit
    q[0] = 0
    qi = torch.from_numpy(q.view(np.int32).copy()).cuda()
    out_a = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    out_b = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert tk.forge_testkit_philox(ctypes.c_void_p(qi.data_ptr()), ctypes.c_void_p(out_a.data_ptr()), n, s) == 0
    assert tk.forge_testkit_curand_philox(ctypes.c_void_p(qi.data_ptr()), ctypes.c_void_p(out_b.data_ptr()), n, s) == 0
    torch.cuda.synchronize()
    mine = out_a.cpu().numpy().view(np.uint32)
    curand = out_b.cpu().numpy().view(np.uint32)
    ref = oph.philox4x32_10(q[:, :4], q[:, 4], q[:, 5])
    assert np.array_equal(mine, ref)
    assert np.array_equal(curand, ref)


# --------------------------------------------------------------- edge cases

@pytest.mark.parametrize("shape", [dict(T=0, N=128, K=256), dict(T=1, N=8, K=64),
                                   dict(T=64, N=8, K=8), dict(T=63, N=128, K=256),
                                   dict(T=1000, N=1024, K=64)])
def test_edge_shapes(shape):
    s_dtype = "int8" if shape["K"] % 64 == 0 else "fp32"
    prob = Problem(**shape, w_dtype="bf16", s_dtype=s_dtype, opt_name="adamw",
                   hp=_hp("adamw"), grid=True, steps=2, seed=31)
    gpu, gdx = prob.run_gpu(fused=True, want_dx=True)
    ref, rdx, _ = prob.run_oracle(want_dx=True)
    _compare_exact(prob, gpu, ref)
    assert_dx_close(gdx[0], to_bits(prob.dY[0]), prob.state0["W"], "dX")


@pytest.mark.parametrize("s_dtype", ["fp32", "int8", "bf16"])
@pytest.mark.parametrize("opt_name", ["adamw", "lion", "sgd"])
def test_one_launch_step_equals_two_launches(opt_name, s_dtype):
    """dX and the step in one launch compute the same bits as the dX launch
    followed by the fused launch: same tiles, same reduction order.  96 pair
    tiles (64 dX + 32 dW) on 76 pairs, so pairs run several tiles and dW tiles
    wait on dX tiles of other pairs; large SGD steps make any weight written
    before its last dX read visible in dX."""
    hp = {"lr": 0.5} if opt_name == "sgd" else _hp(opt_name)
    prob = Problem(T=2048, N=1024, K=2048, w_dtype="bf16", s_dtype=s_dtype, opt_name=opt_name,
                   hp=hp, seed=71, steps=3, device_inputs=True)
    outs = []
    for fused_launch in (True, False):
        api.forge_set_step_fusion(fused_launch)
        try:
            outs.append(prob.run_gpu(fused=True, want_dx=True))
        finally:
            api.forge_set_step_fusion(True)
    (g1, dx1), (g2, dx2) = outs
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k
    for s_ in range(prob.steps):
        assert torch.equal(dx1[s_], dx2[s_]), f"dX step {s_ + 1}"
    # and dX of step 1 is the pre-update weights' product (oracle)
    assert_dx_close(dx1[0].cpu(), to_bits(prob.dY[0].cpu()), prob.state0["W"], "dX")


def test_resume_is_exact():
    """States are plain caller tensors and rounding noise is a function of
    (seed, step, index): 4 steps equal 2 steps, a host round-trip, 2 steps."""
    prob = Problem(T=256, N=256, K=256, w_dtype="bf16", s_dtype="int8", opt_name="adamw",
                   hp=_hp("adamw"), seed=41, steps=4)
    full, _ = prob.run_gpu()
    p2 = Problem(T=256, N=256, K=256, w_dtype="bf16", s_dtype="int8", opt_name="adamw",
                 hp=_hp("adamw"), seed=41, steps=4)
    g = p2.gpu_state()
    for s in range(4):
        if s == 2:
            g = {k: v.cpu().clone().cuda() for k, v in g.items()}
        api.forge_linear_bwd_step(p2.X[s].cuda(), p2.dY[s].cuda(), g["W"], "adamw", p2.hp, s + 1,
                                  p2.seed, g["s1"], g["s2"], g["s1_scale"], g["s2_scale"])
    torch.cuda.synchronize()
    for k in full:
        assert torch.equal(full[k], g[k]), k


def test_fused_step_allocates_no_device_memory():
    prob = Problem(T=1024, N=1024, K=1024, w_dtype="bf16", s_dtype="fp32", opt_name="adamw",
                   hp=_hp("adamw"), seed=51, steps=1)
    g = prob.gpu_state()
    X, dY = prob.X[0].cuda(), prob.dY[0].cuda()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for s in range(3):
        api.forge_linear_bwd_step(X, dY, g["W"], "adamw", prob.hp, s + 1, 1, g["s1"], g["s2"])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_invalid_arguments_raise_before_launch():
    W = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    dY = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.ForgeError) as e:
        api.forge_linear_bwd_step(X, dY, W, "adamw", {}, 1, 0)  # AdamW needs s1/s2
    assert e.value.status == 1
    m = torch.zeros((128, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(api.ForgeError):
        api.forge_linear_bwd_step(X, dY, W, "adamw", {}, 0, 0, m, m.clone())  # step 0


def test_bounded_wait_reports_timeout_and_context_survives():
    """A test hook makes the load warp issue nothing, so the consumers'
    bounded waits expire: the kernel must report FORGE_ERR_TIMEOUT, release
    its resources and leave the context usable."""
    prob = Problem(T=128, N=256, K=256, w_dtype="bf16", s_dtype="fp32", opt_name="sgd",
                   hp={"lr": 1e-2}, grid=True, seed=61, steps=1)
    g = prob.gpu_state()
    api.forge_set_wait_limit_ns(50_000_000)
    api.forge_debug_skip_loads(True)
    try:
        api.forge_linear_bwd_step(prob.X[0].cuda(), prob.dY[0].cuda(), g["W"], "sgd", prob.hp, 1, 1)
        with pytest.raises(api.ForgeError) as e:
            api.forge_get_device_status()
        assert e.value.status == 4
    finally:
        api.forge_debug_skip_loads(False)
        api.forge_set_wait_limit_ns(200_000_000)
    api.forge_get_device_status()  # cleared
    gpu, _ = prob.run_gpu()
    ref, _, _ = prob.run_oracle()
    _compare_exact(prob, gpu, ref)


def test_one_launch_step_timeout_reports_and_context_survives():
    """The same with dX in the launch: the dX tiles' and dW tiles' waits (and
    the wait on the dX counters) all end, and the next step is exact."""
    prob = Problem(T=512, N=256, K=512, w_dtype="bf16", s_dtype="fp32", opt_name="sgd",
                   hp={"lr": 1e-2}, grid=True, seed=62, steps=1)
    g = prob.gpu_state()
    dX = torch.empty((prob.T, prob.K), dtype=torch.bfloat16, device="cuda")
    api.forge_set_wait_limit_ns(50_000_000)
    api.forge_debug_skip_loads(True)
    try:
        api.forge_linear_bwd_step(prob.X[0].cuda(), prob.dY[0].cuda(), g["W"], "sgd", prob.hp, 1, 1,
                                  dX=dX)
        with pytest.raises(api.ForgeError) as e:
            api.forge_get_device_status()
        assert e.value.status == 4
    finally:
        api.forge_debug_skip_loads(False)
        api.forge_set_wait_limit_ns(200_000_000)
    api.forge_get_device_status()  # cleared
    gpu, gdx = prob.run_gpu(want_dx=True)
    ref, rdx, _ = prob.run_oracle(want_dx=True)
    _compare_exact(prob, gpu, ref)
    assert_dx_close(gdx[0], to_bits(prob.dY[0]), prob.state0["W"], "dX")


def test_int8_requantisation_ties_and_zero_blocks_bitexact():
    """The fused epilogue's INT8 requantisation on exact ties: SGD-momentum
    with momentum 0 stores g itself in the signed code buffer; one token
    makes g the outer product dY[0] X[0], with X[0] holding 127 and the
    half-integers 0.5 .. 62.5 (alternating signs, times 2^-6) in every block
    of 64, so g / (absmax / 127) lands exactly on half-integers (ties to even
    on both the reciprocal and the exact-division path); a zero row of dY
    leaves zero blocks (scale 0, codes 0)."""
    T, N, K = 16, 256, 320
    blk = np.array([127.0] + [(j + 0.5) * (-1) ** j for j in range(63)]) * 2.0 ** -6
    x = np.zeros((T, K), np.float32)
    x[0] = np.tile(blk, K // 64)
    dy = np.zeros((T, N), np.float32)
    dy[0] = np.where(np.arange(N) % 3 == 1, 0.0, np.where(np.arange(N) % 3 == 2, -1.0, 1.0))
    X = torch.from_numpy(x).to(torch.bfloat16)
    dY = torch.from_numpy(dy).to(torch.bfloat16)
    hp = dict(lr=1e-2, momentum=0.0)
    prob = Problem(T=T, N=N, K=K, w_dtype="bf16", s_dtype="int8", opt_name="sgd_momentum", hp=hp,
                   grid=True, steps=1, seed=31)
    prob.X, prob.dY = [X], [dY]
    st0 = dict(prob.state0)
    st0["s1"] = np.zeros((N, K), np.int8)
    st0["s1_scale"] = np.zeros((N, K // 64), np.float32)
    prob.state0 = st0
    gpu, _ = prob.run_gpu(fused=True)
    ref, _, _ = prob.run_oracle()
    _compare_exact(prob, gpu, ref)
    codes = ref["s1"].astype(np.int64)
    assert (codes[0, 1:64] % 2 == 0).all() and np.abs(codes[0, 1:64]).max() > 60  # ties went to even
    assert (ref["s1_scale"][1::3] == 0).all() and (codes[1::3] == 0).all()          # zero blocks


@pytest.mark.parametrize("T", [8192, 8208], ids=["staged_weights", "direct_weights"])
@pytest.mark.parametrize("dx", [False, True], ids=["fused", "one_launch"])
def test_int8_epilogue_variants_bitexact(T, dx):
    """INT8 states take one of two epilogues by token count: up to 8192
    tokens the bf16 weights are staged through shared memory with the codes,
    beyond it they are read and written by the compute warps directly.  Both
    sides of the switch match the oracle bit for bit (integer grid), with and
    without dX in the same launch."""
    prob = Problem(T=T, N=256, K=320, w_dtype="bf16", s_dtype="int8", opt_name="adamw",
                   hp=_hp("adamw"), grid=True, steps=2, seed=41)
    gpu, gdx = prob.run_gpu(fused=True, want_dx=dx)
    ref, _, _ = prob.run_oracle(want_dx=dx)
    _compare_exact(prob, gpu, ref)
    if dx:
        assert_dx_close(gdx[0], to_bits(prob.dY[0]), ls.weights_for_dx(prob.state0["W"], "bf16"), "dX")


@pytest.mark.parametrize("s_dtype", ["fp32", "int8"])
@pytest.mark.parametrize("opt_name", ["adamw", "sgd_momentum"])
def test_nonfinite_activations_match_oracle(opt_name, s_dtype):
    """NaN and +-Inf in X (integer grid elsewhere) reach the gradient through
    the tensor-core sums (Inf * 0 and Inf - Inf are NaN, in any order), then
    the rule: weights become NaN (stored as 0x7FC0), fp32 moments NaN or Inf,
    INT8 blocks take an infinite absmax and zero codes for NaN.  Weights and
    states match the oracle bit for bit (NaN equal to NaN)."""
    prob = Problem(T=200, N=320, K=384, w_dtype="bf16", s_dtype=s_dtype, opt_name=opt_name,
                   hp=_hp(opt_name), grid=True, steps=1, seed=43)
    x = prob.X[0].float().numpy().copy()
    x[3, 5] = np.nan
    x[7, 70] = np.inf
    x[9, 200] = -np.inf
    x[11, 200] = np.inf  # +Inf and -Inf in one column: NaN wherever both dY are nonzero
    prob.X[0] = torch.from_numpy(x).to(torch.bfloat16)
    gpu, gdx = prob.run_gpu(fused=True, want_dx=True)
    ref, _, _ = prob.run_oracle(want_dx=False)
    _compare_exact(prob, gpu, ref)
    assert (ref["W"][:, 5] == 0x7FC0).all() and (ref["W"][:, 200] == 0x7FC0).any()
    # dX = dY W does not read X: finite, within the usual dX tolerance
    assert_dx_close(gdx[0], to_bits(prob.dY[0]), ls.weights_for_dx(prob.state0["W"], "bf16"), "dX")


@pytest.mark.parametrize("shape", [dict(T=208, N=2560, K=2048), dict(T=144, N=2568, K=2048)],
                         ids=["aligned", "ragged_rows"])
@pytest.mark.parametrize("w_dtype,opt_name,s_dtype", [("bf16", "adamw", "fp32"), ("bf16", "adamw", "int8"),
                                                      ("bf16", "lion", "bf16"), ("bf16", "sgd_momentum", "fp32"),
                                                      ("fp32", "adamw", "fp32"), ("fp32", "sgd_momentum", "fp32")])
def test_split_last_wave_bitexact(shape, w_dtype, opt_name, s_dtype):
    """More pair tiles than CTA pairs with a short last wave (80 or 88 tiles
    on 76 pairs): the last partial wave runs as 128-column half tiles (N = 128
    MMAs, half-width operand boxes).  Every element still matches the oracle
    bit for bit, in the split tiles as elsewhere."""
    prob = Problem(**shape, w_dtype=w_dtype, s_dtype=s_dtype, opt_name=opt_name, hp=_hp(opt_name),
                   grid=True, steps=2, seed=47)
    gpu, _ = prob.run_gpu(fused=True)
    ref, _, _ = prob.run_oracle()
    _compare_exact(prob, gpu, ref)


@pytest.mark.parametrize("shape", [dict(T=300, N=256, K=256), dict(T=136, N=1288, K=1408),
                                   dict(T=64, N=512, K=4864)],
                         ids=["one_tile", "ragged_36_tiles", "38_tiles"])
@pytest.mark.parametrize("w_dtype,s_dtype", [("bf16", "fp32"), ("bf16", "int8"), ("fp32", "fp32")])
def test_small_layer_half_units_bitexact(shape, w_dtype, s_dtype):
    """A layer of at most 38 pair tiles (half the 76 pairs) runs every tile as
    two 128-column halves on twice the pairs; the result is the oracle's bit
    for bit, ragged edges included."""
    prob = Problem(**shape, w_dtype=w_dtype, s_dtype=s_dtype, opt_name="adamw", hp=_hp("adamw"),
                   grid=True, steps=2, seed=53)
    gpu, _ = prob.run_gpu(fused=True)
    ref, _, _ = prob.run_oracle()
    _compare_exact(prob, gpu, ref)


# (T, N, K) chosen for the dealing regimes of the one-launch step on 76 CTA
# pairs: F weight tiles and D dX tiles fewer than the pairs, exactly a wave,
# one over a wave, dX-dominated, weight-dominated, and ragged T.
DEALING = {
    "F1_D1": (256, 256, 256),
    "F76_D19": (256, 1024, 4864),
    "F152_D38": (512, 2048, 4864),
    "F77_D44": (1024, 1792, 2816),
    "F2_D128": (16384, 256, 512),
    "F224_D16": (1024, 14336, 1024),
    "F160_D32": (512, 2560, 4096),
    "ragged_T": (1000, 1024, 2048),
}


@pytest.mark.parametrize("case", list(DEALING))
def test_one_launch_dealing_regimes_equal_two_launches(case):
    """The host deals dX tiles over the pairs by a load model (full rounds,
    then the rest to the pairs with fewer weight tiles); every regime must
    still cover each dX tile exactly once and write no weight before its
    column block's dX tiles are done: the one launch gives the same bits as
    two launches (a large SGD-momentum step makes an early weight write
    visible in dX of the next step)."""
    T, N, K = DEALING[case]
    prob = Problem(T=T, N=N, K=K, w_dtype="bf16", s_dtype="fp32", opt_name="sgd_momentum",
                   hp={"lr": 0.5, "momentum": 0.9}, seed=73, steps=2, device_inputs=True)
    outs = []
    for fused_launch in (True, False):
        api.forge_set_step_fusion(fused_launch)
        try:
            outs.append(prob.run_gpu(fused=True, want_dx=True))
        finally:
            api.forge_set_step_fusion(True)
    (g1, dx1), (g2, dx2) = outs
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k
    for s_ in range(prob.steps):
        assert torch.equal(dx1[s_], dx2[s_]), f"dX step {s_ + 1}"
