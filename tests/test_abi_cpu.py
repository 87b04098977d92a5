"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/forge.h declares, and rejects invalid arguments on the host
before any CUDA call.  No computation is launched here."""

import ctypes
import os
import re

import pytest

from optimizer_tcgen05_dw_gb300 import api
from optimizer_tcgen05_dw_gb300.build import build, lib_path

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return api.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "forge.h")) as f:
        src = f.read()
    return re.findall(r"FORGE_API\s+[\w\s\*]+?\b(forge_\w+)\s*\(", src)


def test_header_declares_the_entry_points():
    names = set(_declared())
    for n in ("forge_linear_bwd_step", "forge_linear_dgrad", "forge_unfused_wgrad",
              "forge_unfused_opt_step", "forge_quantize_state", "forge_dequantize_state",
              "forge_get_device_status", "forge_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    raw = ctypes.CDLL(lib_path("libforge.so"))
    for name in _declared():
        assert hasattr(raw, name), name
    assert L.forge_abi_version() == 1


def test_status_strings(L):
    for code, name in api.STATUS.items():
        assert L.forge_status_string(code).decode().startswith(name)


def _lin(T=64, N=128, K=256, x=16, dy=16, dx=None):
    return api.ForgeLinear(T, N, K, ctypes.c_void_p(x), ctypes.c_void_p(dy),
                           None if dx is None else ctypes.c_void_p(dx))


def _state(w=32, s1=48, s2=64, wdt=1, sdt=0, sc1=None, sc2=None):
    return api.ForgeState(ctypes.c_void_p(w), wdt, sdt, ctypes.c_void_p(s1) if s1 else None,
                          ctypes.c_void_p(s2) if s2 else None,
                          ctypes.c_void_p(sc1) if sc1 else None, ctypes.c_void_p(sc2) if sc2 else None)


@pytest.mark.parametrize("case", [
    "null_lin", "bad_kind", "step0", "n_not_mult8", "int8_k_not_mult64", "missing_state",
    "misaligned_x", "null_hp", "bad_wdtype", "int8_missing_scale"])
def test_invalid_arguments_rejected_on_host(L, case):
    hp = api.hparams()
    lin, st, kind, step, hpp = _lin(), _state(), 0, 1, ctypes.byref(hp)
    if case == "null_lin":
        lin = None
    elif case == "bad_kind":
        kind = 9
    elif case == "step0":
        step = 0
    elif case == "n_not_mult8":
        lin = _lin(N=100)
    elif case == "int8_k_not_mult64":
        lin = _lin(K=200)
        st = _state(sdt=1, sc1=80, sc2=96)
    elif case == "missing_state":
        st = _state(s2=0)
    elif case == "misaligned_x":
        lin = _lin(x=17)
    elif case == "null_hp":
        hpp = None
    elif case == "bad_wdtype":
        st = _state(wdt=5)
    elif case == "int8_missing_scale":
        st = _state(sdt=1, sc1=80)
    rc = L.forge_linear_bwd_step(None if lin is None else ctypes.byref(lin), ctypes.byref(st),
                                 kind, hpp, step, 0, None)
    assert rc == 1, (case, rc, L.forge_last_error_message())
    assert L.forge_last_error_message().decode() != ""


def test_bf16_moments_with_fp32_weights_unsupported_in_the_fused_step(L):
    hp = api.hparams()
    st = _state(wdt=api.W_FP32, sdt=api.STATE_BF16)
    rc = L.forge_linear_bwd_step(ctypes.byref(_lin()), ctypes.byref(st), 0, ctypes.byref(hp), 1, 0, None)
    assert rc == 2, (rc, L.forge_last_error_message())
    assert b"bf16 moments" in L.forge_last_error_message()


@pytest.mark.parametrize("sdt,K,rc", [(api.STATE_INT8_B256, 320, 1), (api.STATE_INT8_B128, 320, 1),
                                      (api.STATE_INT8_B32, 200, 1), (9, 256, 1)],
                         ids=["b256_k320", "b128_k320", "b32_k200", "unknown_sdtype"])
def test_int8_block_width_checked_on_host(L, sdt, K, rc):
    """K must be a multiple of the INT8 block width (and of 64); unknown state
    dtypes are refused."""
    hp = api.hparams()
    st = _state(sdt=sdt, sc1=80, sc2=96)
    got = L.forge_linear_bwd_step(ctypes.byref(_lin(K=K)), ctypes.byref(st), 0, ctypes.byref(hp), 1, 0, None)
    assert got == rc, (got, L.forge_last_error_message())


@pytest.mark.parametrize("sdt", [api.STATE_INT8_B32, api.STATE_INT8_B128, api.STATE_INT8_B256])
def test_int8_block_widths_other_than_64_need_bf16_weights_in_the_fused_step(L, sdt):
    hp = api.hparams()
    st = _state(wdt=api.W_FP32, sdt=sdt, sc1=80, sc2=96)
    rc = L.forge_linear_bwd_step(ctypes.byref(_lin(K=512)), ctypes.byref(st), 0, ctypes.byref(hp), 1, 0, None)
    assert rc == 2 and b"bf16 weights" in L.forge_last_error_message()


def test_quantiser_block_width_checked_on_host(L):
    assert L.forge_quantize_state_block(None, None, None, 4, 256, 1, 48, None) == 1   # width 48
    assert L.forge_quantize_state_block(None, None, None, 4, 320, 1, 256, None) == 1  # cols % 256
    assert L.forge_dequantize_state_block(None, None, None, 4, 192, 0, 128, None) == 1  # cols % 128
    assert b"cols" in L.forge_last_error_message()


def test_other_entry_points_validate(L):
    assert L.forge_unfused_opt_step(None, None, 8, 8, 0, None, 1, 0, None) == 1
    assert L.forge_quantize_state(None, None, None, 4, 100, 1, None) == 1  # cols % 64
    assert L.forge_unfused_wgrad(ctypes.byref(_lin()), ctypes.c_void_p(3), None) == 1  # misaligned dW
    assert L.forge_linear_dgrad(ctypes.byref(_lin(dx=16)), None, 7, None) == 1  # bad w_dtype


def test_empty_problem_is_a_no_op(L):
    """N == 0 or K == 0: nothing to do, no device touched."""
    hp = api.hparams()
    assert L.forge_linear_bwd_step(ctypes.byref(_lin(N=0)), ctypes.byref(_state()), 0,
                                   ctypes.byref(hp), 1, 0, None) == 0


def test_valid_call_without_a_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    hp = api.hparams()
    rc = L.forge_linear_bwd_step(ctypes.byref(_lin()), ctypes.byref(_state()), 0,
                                 ctypes.byref(hp), 1, 0, None)
    assert rc == 3


def _lin8(T=128, N=256, K=256, x=16, dy=32, sx=1.0, sdy=1.0):
    return api.ForgeLinearFp8(T, N, K, ctypes.c_void_p(x), ctypes.c_void_p(dy), sx, sdy)


@pytest.mark.parametrize("case,rc", [
    ("null_lin", 1), ("t_not_mult16", 1), ("k_not_mult8", 1), ("misaligned_xt", 1), ("null_dyt", 1),
    ("nan_scale", 1), ("scale_product_overflows", 1), ("bad_kind", 1), ("fp32_weights", 2),
    ("negative_t", 1)])
def test_fp8_step_arguments_checked_on_host(L, case, rc):
    hp = api.hparams()
    lin, st, kind = _lin8(), _state(), 0
    if case == "null_lin":
        lin = None
    elif case == "t_not_mult16":
        lin = _lin8(T=120)
    elif case == "k_not_mult8":
        lin = _lin8(K=100)
    elif case == "misaligned_xt":
        lin = _lin8(x=24)
    elif case == "null_dyt":
        lin = api.ForgeLinearFp8(128, 256, 256, ctypes.c_void_p(16), None, 1.0, 1.0)
    elif case == "nan_scale":
        lin = _lin8(sx=float("nan"))
    elif case == "scale_product_overflows":
        lin = _lin8(sx=1e30, sdy=1e30)
    elif case == "bad_kind":
        kind = 11
    elif case == "fp32_weights":
        st = _state(wdt=api.W_FP32)
    elif case == "negative_t":
        lin = _lin8(T=-16)
    got = L.forge_linear_bwd_step_fp8(None if lin is None else ctypes.byref(lin), ctypes.byref(st),
                                      kind, ctypes.byref(hp), 1, 0, None)
    assert got == rc, (case, got, L.forge_last_error_message())
    assert L.forge_last_error_message().decode() != ""


def test_fp8_step_empty_problem_is_a_no_op(L):
    hp = api.hparams()
    assert L.forge_linear_bwd_step_fp8(ctypes.byref(_lin8(N=0)), ctypes.byref(_state()), 0,
                                       ctypes.byref(hp), 1, 0, None) == 0


def test_fp8_binding_rejects_wrong_dtypes_before_the_library():
    import torch
    Xt = torch.zeros((64, 32), dtype=torch.bfloat16)
    dYt = torch.zeros((64, 32), dtype=torch.uint8)
    W = torch.zeros((64, 64), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="E4M3"):
        api.forge_linear_bwd_step_fp8(Xt, dYt, 1.0, 1.0, W, "sgd", {}, 1, 0)
