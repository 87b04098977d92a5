"""The one-launch step when the device is not free.

A dW tile of the one-launch step waits for dX tiles that other pairs of the
same launch compute, so the launch needs all its pairs running at once.  If
another kernel holds SMs, some pairs cannot start; the launch's residency gate
then lets no pair write a weight: after the wait limit every CTA stops, the
status word reports a timeout and W and the moments are exactly as before the
call.  Here the step first runs on the free device and matches the oracle;
then a test-kit kernel holds 40 SMs (one block each, 200 KiB of shared memory,
so no step CTA fits beside it) for 0.4 s while the same step launches with a
50 ms wait limit.
"""

import ctypes
import time

import pytest
import torch

from optimizer_tcgen05_dw_gb300 import api
from optimizer_tcgen05_dw_gb300.build import build, lib_path

from _helpers import Problem, assert_bitexact, assert_dx_close, to_bits

pytestmark = pytest.mark.gpu


def test_step_without_all_pairs_resident_stops_before_writing(cuda_device):
    build()
    api.lib()
    api.forge_set_step_fusion(True)
    api.forge_debug_skip_loads(False)
    # 64 weight tiles and 16 dX tiles: a grid of all 76 pairs
    prob = Problem(T=512, N=2048, K=2048, w_dtype="bf16", s_dtype="fp32", opt_name="adamw",
                   hp={"lr": 1e-2, "weight_decay": 0.01}, grid=True, seed=91, steps=1)
    # first the step on the free device, against the oracle (this also loads
    # the kernels' modules, whose first load would wait for the holding kernel)
    gpu, gdx = prob.run_gpu(want_dx=True)
    ref, _, _ = prob.run_oracle(want_dx=True)
    for k in ("W", "s1", "s2"):
        if ref.get(k) is not None:
            assert_bitexact(gpu[k], ref[k], k)
    assert_dx_close(gdx[0], to_bits(prob.dY[0]), prob.state0["W"], "dX")
    tk = ctypes.CDLL(lib_path("libforge_testkit.so"))
    tk.forge_testkit_hold_sms.argtypes = [ctypes.c_int, ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p]
    side, main = torch.cuda.Stream(), torch.cuda.Stream()
    assert tk.forge_testkit_hold_sms(1, 1000, 200 * 1024, ctypes.c_void_p(side.cuda_stream)) == 0  # loaded
    g = prob.gpu_state()
    before = {k: v.clone() for k, v in g.items() if v is not None}
    X, dY = prob.X[0].cuda(), prob.dY[0].cuda()
    dX = torch.empty((prob.T, prob.K), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    api.forge_set_wait_limit_ns(50_000_000)
    try:
        assert tk.forge_testkit_hold_sms(40, 400_000_000, 200 * 1024, ctypes.c_void_p(side.cuda_stream)) == 0
        time.sleep(0.02)  # the holding blocks are on their SMs before the step launches
        api.forge_linear_bwd_step(X, dY, g["W"], "adamw", prob.hp, 1, prob.seed, g.get("s1"), g.get("s2"),
                                  dX=dX, stream=main)
        with pytest.raises(api.ForgeError) as e:
            api.forge_get_device_status(main)
        assert e.value.status == 4  # timeout
        torch.cuda.synchronize()
    finally:
        api.forge_set_wait_limit_ns(200_000_000)
    api.forge_get_device_status(main)  # cleared
    for k, v in before.items():
        assert torch.equal(g[k], v), f"{k} was written by a step that stopped at the residency gate"
