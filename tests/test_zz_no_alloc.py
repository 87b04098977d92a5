"""forge_linear_bwd_step_static: the one-launch step with its scratch (the
dX-completion counters) in the library's static device array.  It must give
the same bits as forge_linear_bwd_step over two calls in a row, allocate no
device memory, and reject a request its scratch cannot hold before any CUDA
call.  Kept in its own file, collected last; it also passes alone."""

import ctypes

import numpy as np
import pytest
import torch

from optimizer_tcgen05_dw_gb300 import api, inputs
from optimizer_tcgen05_dw_gb300.build import build


def test_oversize_request_rejected_before_any_cuda_call():
    build()
    L = api.lib()
    # K = 270336: 1056 column blocks > the 1024 words of static scratch.  The
    # pointers are never dereferenced: the call must fail on the host.
    fake = 1 << 20
    lin = api.ForgeLinear(64, 128, 270336, fake, fake, fake)
    st = api.ForgeState(fake, api.W_BF16_SR, api.STATE_FP32, fake, fake, None, None)
    hp = api.hparams(lr=1e-3)
    r = L.forge_linear_bwd_step_static(ctypes.byref(lin), ctypes.byref(st), api.OPT_KINDS["adamw"],
                                       ctypes.byref(hp), 1, 0, None)
    assert r == 2, r  # FORGE_ERR_UNSUPPORTED
    assert b"static scratch" in L.forge_last_error_message()


def _static_call(K, s_dtype=None, N=128):
    """forge_linear_bwd_step_static with never-dereferenced fake pointers."""
    L = api.lib()
    fake = 1 << 20
    lin = api.ForgeLinear(64, N, K, fake, fake, fake)
    sd = api.STATE_FP32 if s_dtype is None else s_dtype
    st = api.ForgeState(fake, api.W_BF16_SR, sd, fake, fake, fake, fake)
    hp = api.hparams(lr=1e-3)
    r = L.forge_linear_bwd_step_static(ctypes.byref(lin), ctypes.byref(st), api.OPT_KINDS["adamw"],
                                       ctypes.byref(hp), 1, 0, None)
    return r, L.forge_last_error_message()


def test_size_limit_edge_one_block_over_is_rejected():
    build()
    # K = 262144 + 64: 1025 column blocks of 256, one more than the scratch holds
    r, msg = _static_call(262144 + 64)
    assert r == 2 and b"static scratch" in msg, (r, msg)


def test_requests_outside_the_one_launch_reach_the_two_launch_checks():
    build()
    # K above the limit but not a multiple of 64: no one launch, so no scratch;
    # with INT8 states the two-launch path's own check (K % 64) refuses it on
    # the host, not the scratch limit
    r, msg = _static_call(270336 + 8, api.STATE_INT8_B64)
    assert r == 1 and b"K % 64" in msg, (r, msg)
    assert b"static scratch" not in msg


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers on a GPU host")
def test_size_limit_edge_largest_accepted_passes_the_host_check():
    build()
    # K = 262144: exactly 1024 blocks, accepted by the size check; on a host
    # without a GPU the call then fails at its first CUDA call instead
    r, msg = _static_call(262144)
    assert r == 3 and b"static scratch" not in msg, (r, msg)


@pytest.mark.gpu
@pytest.mark.parametrize("s_dtype", ["fp32", "int8"])
def test_static_scratch_step_equals_regular_step(cuda_device, s_dtype):
    build()
    api.lib()
    api.forge_set_wait_limit_ns(200_000_000)
    api.forge_debug_skip_loads(False)
    api.forge_set_step_fusion(True)
    T, N, K = 1024, 512, 768  # 12 dX tiles + 6 weight tiles, ragged in K
    seed = 91
    X = [inputs.normal((T, K), 1.0, seed + 10 * s, torch.bfloat16, "cuda") for s in range(2)]
    dY = [inputs.normal((T, N), 1e-3, seed + 10 * s + 1, torch.bfloat16, "cuda") for s in range(2)]
    W0 = inputs.normal((N, K), 0.02, seed + 2, torch.bfloat16, "cuda")
    hp = dict(inputs.SWEEP_HPARAMS["adamw"])

    def fresh():
        if s_dtype == "int8":
            m = torch.zeros((N, K), dtype=torch.int8, device="cuda")
            v = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
            return [W0.clone(), m, v, torch.zeros((N, K // 64), device="cuda"),
                    torch.zeros((N, K // 64), device="cuda")]
        return [W0.clone(), torch.zeros((N, K), device="cuda"), torch.zeros((N, K), device="cuda"),
                None, None]

    # load the kernels first (lazy module loading allocates code memory on a
    # kernel's first launch in a process, which is not the library's doing)
    warm = fresh()
    dx_warm = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    api.forge_linear_bwd_step(X[0], dY[0], warm[0], "adamw", hp, 1, seed, *warm[1:], dX=dx_warm)
    api.forge_linear_bwd_step_static(X[0], dY[0], warm[0], "adamw", hp, 2, seed, *warm[1:], dX=dx_warm)
    api.forge_get_device_status()

    reg, sta = fresh(), fresh()
    dx_reg = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    dx_sta = torch.empty_like(dx_reg)
    # snapshots of both calls' results, allocated up front so that nothing in
    # the measured region allocates except (if it did) the library
    snaps = [[None if t is None else torch.empty_like(t) for t in reg + sta + [dx_reg, dx_sta]]
             for _ in range(2)]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for s in range(2):  # two calls in a row through each entry point
        api.forge_linear_bwd_step(X[s], dY[s], reg[0], "adamw", hp, s + 1, seed, *reg[1:], dX=dx_reg)
        api.forge_linear_bwd_step_static(X[s], dY[s], sta[0], "adamw", hp, s + 1, seed, *sta[1:],
                                         dX=dx_sta)
        api.forge_get_device_status()
        for dst, src in zip(snaps[s], reg + sta + [dx_reg, dx_sta]):
            if src is not None:
                dst.copy_(src)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    names = ("W", "s1", "s2", "s1_scale", "s2_scale")
    for s in range(2):
        r, t = snaps[s][:5], snaps[s][5:10]
        for name, a, b in zip(names, r, t):
            if a is not None:
                assert torch.equal(a, b), f"call {s + 1}: {name}"
        assert torch.equal(snaps[s][10], snaps[s][11]), f"call {s + 1}: dX"
    assert not torch.equal(snaps[1][0], W0)  # the steps did update the weights
