"""Full-size parity on sampled tiles, in the launch configuration the bench times.

The oracle cannot form dW for a whole Llama/Qwen layer at T = 16384 in a test,
but every element's update depends only on its own coordinate (FORGE
explainer, Technical Summary §2 "Exactness").  So it follows a set of sampled
128 x 128 tiles (the four corners plus random interior tiles).  Before every
step those tiles of the GPU state are set to the oracle's state, the full
layer is stepped on the GPU, and the sampled tiles must lie in the oracle's
interval for that step (tests/_helpers.py: the oracle evaluated at g - d, g,
g + d with d the tensor-core summation bound).
"""

import numpy as np
import pytest
import torch

from oracle import linear_step as ls
from oracle import optimizers as opt
from oracle import quant, rounding
from optimizer_tcgen05_dw_gb300 import api, inputs
from optimizer_tcgen05_dw_gb300.build import build

from _helpers import (assert_dx_close, assert_in_interval, grad_error_bound, oracle_hparams,
                      oracle_interval, to_bits)

pytestmark = pytest.mark.gpu

TILE = 128
KEYS = ("W", "s1", "s2", "s1_scale", "s2_scale")


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    api.lib()
    api.forge_set_wait_limit_ns(200_000_000)
    yield
    api.forge_set_wait_limit_ns(0)


def _tiles(N, K, count, seed):
    rng = np.random.default_rng(seed)
    tn, tk = N // TILE, K // TILE
    picks = {(0, 0), (0, tk - 1), (tn - 1, 0), (tn - 1, tk - 1)}
    while len(picks) < count:
        picks.add((int(rng.integers(0, tn)), int(rng.integers(0, tk))))
    return sorted((a * TILE, b * TILE) for a, b in picks)


def _region(key, n0, k0):
    blk = 64 if key.endswith("scale") else 1
    return slice(n0, n0 + TILE), slice(k0 // blk, (k0 + TILE) // blk)


def _to_dev(key, arr, w_dtype):
    if key == "W" and w_dtype == "bf16":
        return inputs.bits_to_bf16(arr)
    return torch.from_numpy(np.ascontiguousarray(arr))


def run_sampled(N, K, T, w_dtype, s_dtype, opt_name, hp, steps, seed, m_std=0.0, v_std=0.0,
                x_std=1.0, dy_std=1e-3, n_tiles=12):
    kind = opt.NAMES.index(opt_name)
    tiles = _tiles(N, K, n_tiles, seed)
    # initial state, drawn on the CPU from seeds; INT8 codes from the oracle quantiser
    W = inputs.normal((N, K), 0.02, inputs.layer_seed(seed, 0, 0, 3), torch.float32)
    st = {"W": W.numpy() if w_dtype == "fp32" else rounding.bf16_bits_rne(W.numpy())}
    del W
    if opt.USES_S1[kind]:
        m = inputs.normal((N, K), m_std, inputs.layer_seed(seed, 0, 0, 4), torch.float32).numpy()
        if s_dtype == "int8":
            st["s1"], st["s1_scale"] = quant.quantize_blocks(m, True)
        else:
            st["s1"] = m
    if opt.USES_S2[kind]:
        v = inputs.abs_normal((N, K), v_std, inputs.layer_seed(seed, 0, 0, 5)).numpy()
        if s_dtype == "int8":
            st["s2"], st["s2_scale"] = quant.quantize_blocks(v, False)
        else:
            st["s2"] = v
    gpu = {k: _to_dev(k, st[k], w_dtype).cuda() for k in KEYS if st.get(k) is not None}
    ost = {t: {k: np.ascontiguousarray(st[k][_region(k, *t)]) for k in KEYS if st.get(k) is not None}
           for t in tiles}
    del st
    ohp = oracle_hparams(hp)
    for s in range(steps):
        # sampled tiles of the GPU state := the oracle's state
        for t, o in ost.items():
            for k, arr in o.items():
                gpu[k][_region(k, *t)] = _to_dev(k, arr, w_dtype).cuda()
        X = inputs.normal((T, K), x_std, inputs.layer_seed(seed, 0, s, 1), device="cuda")
        dY = inputs.normal((T, N), dy_std, inputs.layer_seed(seed, 0, s, 2), device="cuda")
        api.forge_linear_bwd_step(X, dY, gpu["W"], opt_name, hp, s + 1, seed, gpu.get("s1"),
                                  gpu.get("s2"), gpu.get("s1_scale"), gpu.get("s2_scale"))
        api.forge_get_device_status()
        Xc = {k0: to_bits(X[:, k0:k0 + TILE].contiguous()) for k0 in {k0 for _, k0 in tiles}}
        dYc = {n0: to_bits(dY[:, n0:n0 + TILE].contiguous()) for n0 in {n0 for n0, _ in tiles}}
        del X, dY
        for (n0, k0) in tiles:
            g = ls.weight_gradient(Xc[k0], dYc[n0])
            o = ost[(n0, k0)]
            iv = oracle_interval(kind, ohp, s + 1, seed, g, o, w_dtype, s_dtype, n0, k0, K,
                                 grad_error_bound(Xc[k0], dYc[n0]))
            got = {k: gpu[k][_region(k, n0, k0)].contiguous() for k in o}
            assert_in_interval(got, iv, w_dtype, s_dtype, f"step {s + 1} tile ({n0},{k0})")
            ost[(n0, k0)] = {k: iv[0][0][k] for k in o}


LLAMA = {n: (N, K) for n, N, K in inputs.LLAMA31_8B_LINEARS}
QWEN = {n: (N, K) for n, N, K in inputs.QWEN3_14B_LINEARS}


@pytest.mark.parametrize("layer", ["gate_proj", "down_proj", "k_proj"])
def test_llama8b_bf16_fp32state_sampled(layer):
    w = inputs.WORKLOADS["llama8b_bf16_fp32state"]
    N, K = LLAMA[layer]
    run_sampled(N, K, w.T, "bf16", "fp32", "adamw", w.hparams, steps=2, seed=2000 + N % 97,
                m_std=1e-4, v_std=1e-6)


@pytest.mark.parametrize("layer", ["up_proj", "o_proj"])
def test_llama8b_bf16_int8state_sampled(layer):
    w = inputs.WORKLOADS["llama8b_bf16_int8state"]
    N, K = LLAMA[layer]
    run_sampled(N, K, w.T, "bf16", "int8", "adamw", w.hparams, steps=2, seed=3000 + N % 89,
                m_std=w.m_init_std, v_std=w.v_init_std)


@pytest.mark.parametrize("opt_name", list(opt.NAMES))
def test_optimizer_sweep_4096_sampled(opt_name):
    w = inputs.WORKLOADS["sweep_4096"]
    _, N, K = w.linears[0]
    run_sampled(N, K, w.T, "bf16", "fp32", opt_name, inputs.SWEEP_HPARAMS[opt_name],
                steps=w.steps, seed=4000 + opt.NAMES.index(opt_name), n_tiles=8)


@pytest.mark.parametrize("layer", ["down_proj", "v_proj"])
def test_qwen14b_int8_sampled(layer):
    w = inputs.WORKLOADS["qwen14b_int8"]
    N, K = QWEN[layer]
    run_sampled(N, K, w.T, "bf16", "int8", "adamw", w.hparams, steps=2, seed=5000 + N % 83,
                m_std=1e-4, v_std=1e-6)


@pytest.mark.parametrize("layer", ["q_proj", "k_proj"])
def test_llama8b_one_launch_step_with_dx(layer):
    """The bench's launch: dX and the FORGE step of a full-size layer in one
    launch.  Same bits as the two-launch form (dX launch, then the fused
    launch) for W, m, v and dX, and sampled 128 x 128 tiles of dX equal the
    oracle's dY W from the pre-update weights."""
    w = inputs.WORKLOADS["llama8b_bf16_fp32state"]
    N, K = LLAMA[layer]
    T = w.T
    seed = 6000 + N % 79
    X = inputs.normal((T, K), 1.0, inputs.layer_seed(seed, 0, 0, 1), device="cuda")
    dY = inputs.normal((T, N), w.dy_std, inputs.layer_seed(seed, 0, 0, 2), device="cuda")
    W0 = inputs.normal((N, K), 0.02, inputs.layer_seed(seed, 0, 0, 3), torch.bfloat16, "cuda")
    outs = []
    for one_launch in (True, False):
        W = W0.clone()
        m = torch.zeros((N, K), dtype=torch.float32, device="cuda")
        v = torch.zeros((N, K), dtype=torch.float32, device="cuda")
        dX = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        api.forge_set_step_fusion(one_launch)
        try:
            api.forge_linear_bwd_step(X, dY, W, "adamw", w.hparams, 1, seed, m, v, dX=dX)
            api.forge_get_device_status()
        finally:
            api.forge_set_step_fusion(True)
        outs.append((W, m, v, dX))
    for a, b, name in zip(outs[0], outs[1], ("W", "m", "v", "dX")):
        assert torch.equal(a, b), name
    dX = outs[0][3]
    rng = np.random.default_rng(seed)
    W0b = to_bits(W0)
    for _ in range(6):
        t0 = int(rng.integers(0, T // TILE)) * TILE
        k0 = int(rng.integers(0, K // TILE)) * TILE
        assert_dx_close(dX[t0:t0 + TILE, k0:k0 + TILE].contiguous(), to_bits(dY[t0:t0 + TILE].contiguous()),
                        np.ascontiguousarray(W0b[:, k0:k0 + TILE]), f"dX tile ({t0},{k0})")


@pytest.mark.parametrize("layer", ["gate_proj", "k_proj"])
def test_qwen14b_int8_one_launch_step_with_dx(layer):
    """The Qwen3-14B configuration's launch: dX and the FORGE step with INT8
    block-64 AdamW moments of a full-size layer at T = 4096 in one launch (the
    staged-weights INT8 epilogue).  Same bits as the two-launch form for W, the
    codes, the scales and dX (k_proj: 80 weight tiles on 76 pairs, so some pairs
    take two), and sampled dX tiles equal the oracle's dY W from the pre-update
    weights."""
    w = inputs.WORKLOADS["qwen14b_int8"]
    N, K = QWEN[layer]
    T = w.T
    seed = 7000 + N % 71
    X = inputs.normal((T, K), 1.0, inputs.layer_seed(seed, 0, 0, 1), device="cuda")
    dY = inputs.normal((T, N), w.dy_std, inputs.layer_seed(seed, 0, 0, 2), device="cuda")
    W0 = inputs.normal((N, K), 0.02, inputs.layer_seed(seed, 0, 0, 3), torch.bfloat16, "cuda")
    m0 = torch.empty((N, K), dtype=torch.int8, device="cuda")
    v0 = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    ms0 = torch.empty((N, K // 64), device="cuda")
    vs0 = torch.empty((N, K // 64), device="cuda")
    api.forge_quantize_state(inputs.normal((N, K), 1e-4, inputs.layer_seed(seed, 0, 0, 4), torch.float32, "cuda"),
                             m0, ms0, True)
    api.forge_quantize_state(inputs.abs_normal((N, K), 1e-6, inputs.layer_seed(seed, 0, 0, 5), torch.float32, "cuda"),
                             v0, vs0, False)
    outs = []
    for one_launch in (True, False):
        W, m, v, ms, vs = W0.clone(), m0.clone(), v0.clone(), ms0.clone(), vs0.clone()
        dX = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        api.forge_set_step_fusion(one_launch)
        try:
            api.forge_linear_bwd_step(X, dY, W, "adamw", w.hparams, 1, seed, m, v, ms, vs, dX=dX)
            api.forge_get_device_status()
        finally:
            api.forge_set_step_fusion(True)
        outs.append((W, m, v, ms, vs, dX))
    for a, b, name in zip(outs[0], outs[1], ("W", "m codes", "v codes", "m scales", "v scales", "dX")):
        assert torch.equal(a, b), name
    dX = outs[0][5]
    rng = np.random.default_rng(seed)
    W0b = to_bits(W0)
    for _ in range(6):
        t0 = int(rng.integers(0, T // TILE)) * TILE
        k0 = int(rng.integers(0, K // TILE)) * TILE
        assert_dx_close(dX[t0:t0 + TILE, k0:k0 + TILE].contiguous(), to_bits(dY[t0:t0 + TILE].contiguous()),
                        np.ascontiguousarray(W0b[:, k0:k0 + TILE]), f"dX tile ({t0},{k0})")
