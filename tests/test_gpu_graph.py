"""The FORGE step captured in a CUDA graph.

Every launch of one call is a stream operation (no host synchronisation, no
allocation), so a call made while the current stream is being captured records
its launches, and replaying the graph performs the step.  The replayed step
must give the oracle's bits on integer-grid inputs and the same dX bits as the
call made directly: for the one-launch form (bf16 weights) and for the fp32
master weights, where the step is a programmatic dependent launch of dX.
"""

import pytest
import torch

from optimizer_tcgen05_dw_gb300 import api
from optimizer_tcgen05_dw_gb300.build import build

from _helpers import Problem, assert_bitexact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    build()
    api.lib()
    api.forge_set_wait_limit_ns(200_000_000)
    yield
    api.forge_set_wait_limit_ns(0)


def _call(prob, g, X, dY, dX):
    api.forge_linear_bwd_step(X, dY, g["W"], prob.opt, prob.hp, 1, prob.seed, g.get("s1"), g.get("s2"),
                              g.get("s1_scale"), g.get("s2_scale"), dX=dX)


@pytest.mark.parametrize("w_dtype,s_dtype", [("bf16", "fp32"), ("bf16", "int8"), ("fp32", "fp32")],
                         ids=["one_launch_fp32_states", "one_launch_int8_states", "fp32_master"])
def test_captured_step_replays_to_the_oracle_bits(w_dtype, s_dtype):
    prob = Problem(T=200, N=320, K=384, w_dtype=w_dtype, s_dtype=s_dtype, opt_name="adamw",
                   hp=dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
                   grid=True, steps=1, seed=23)
    X, dY = prob.X[0].cuda(), prob.dY[0].cuda()
    # the direct call (it also does the library's one-time set-up before capture)
    g_direct = prob.gpu_state()
    dx_direct = torch.empty((prob.T, prob.K), dtype=torch.bfloat16, device="cuda")
    _call(prob, g_direct, X, dY, dx_direct)
    api.forge_get_device_status()
    torch.cuda.synchronize()

    g = prob.gpu_state()
    dX = torch.zeros((prob.T, prob.K), dtype=torch.bfloat16, device="cuda")
    w0 = g["W"].clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(prob, g, X, dY, dX)
    torch.cuda.synchronize()
    assert torch.equal(g["W"], w0), "capturing must not run the step"
    graph.replay()
    torch.cuda.synchronize()
    api.forge_get_device_status()

    ref, _, _ = prob.run_oracle()
    assert_bitexact(g["W"], ref["W"], "W (replayed)")
    for k in ("s1", "s2", "s1_scale", "s2_scale"):
        if ref.get(k) is not None:
            assert_bitexact(g[k], ref[k], k + " (replayed)")
    assert torch.equal(dX, dx_direct), "replayed dX differs from the direct call's"
