"""ctypes binding of libforge (include/forge.h), same names as the C ABI.

This module only marshals arguments: it checks that torch tensors have the
dtype, shape, device and contiguity the C ABI documents, passes their data
pointers and the current CUDA stream, and turns a non-OK status into
ForgeError.  Every step of the computation runs in the library's kernels.
Loading fails loudly if the library has not been built.
"""

import ctypes
import os
import threading

import torch

from . import build as _build

c_int32, c_int64, c_uint64, c_float, c_void_p = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                                 ctypes.c_float, ctypes.c_void_p)

OPT_KINDS = {"adamw": 0, "nadam": 1, "radam": 2, "lion": 3, "rmsprop": 4, "adagrad": 5,
             "sgd": 6, "sgd_momentum": 7}
W_FP32, W_BF16_SR = 0, 1
STATE_FP32, STATE_INT8_B64, STATE_BF16 = 0, 1, 2
STATE_INT8_B32, STATE_INT8_B128, STATE_INT8_B256 = 3, 4, 5
INT8_STATE_OF_BLOCK = {32: STATE_INT8_B32, 64: STATE_INT8_B64, 128: STATE_INT8_B128,
                       256: STATE_INT8_B256}
USES_S1 = {"adamw", "nadam", "radam", "lion", "sgd_momentum"}
USES_S2 = {"adamw", "nadam", "radam", "rmsprop", "adagrad"}

STATUS = {0: "FORGE_OK", 1: "FORGE_ERR_INVALID_ARG", 2: "FORGE_ERR_UNSUPPORTED",
          3: "FORGE_ERR_CUDA", 4: "FORGE_ERR_TIMEOUT", 5: "FORGE_ERR_DEVICE"}


class ForgeLinear(ctypes.Structure):
    _fields_ = [("T", c_int64), ("N", c_int64), ("K", c_int64),
                ("X", c_void_p), ("dY", c_void_p), ("dX", c_void_p)]


class ForgeLinearFp8(ctypes.Structure):
    _fields_ = [("T", c_int64), ("N", c_int64), ("K", c_int64),
                ("Xt", c_void_p), ("dYt", c_void_p), ("x_scale", c_float), ("dy_scale", c_float)]


class ForgeState(ctypes.Structure):
    _fields_ = [("W", c_void_p), ("w_dtype", c_int32), ("s_dtype", c_int32),
                ("s1", c_void_p), ("s2", c_void_p), ("s1_scale", c_void_p), ("s2_scale", c_void_p)]


class ForgeHparams(ctypes.Structure):
    _fields_ = [(n, c_float) for n in ("lr", "beta1", "beta2", "eps", "weight_decay", "alpha",
                                       "momentum")]


HPARAM_DEFAULTS = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, alpha=0.99,
                       momentum=0.0)


class ForgeError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {message}")


_lock = threading.Lock()
_lib = None

_SIGNATURES = {
    "forge_linear_bwd_step": (c_int32, [ctypes.POINTER(ForgeLinear), ctypes.POINTER(ForgeState),
                                        c_int32, ctypes.POINTER(ForgeHparams), c_int64, c_uint64,
                                        c_void_p]),
    "forge_linear_bwd_step_static": (c_int32, [ctypes.POINTER(ForgeLinear), ctypes.POINTER(ForgeState),
                                               c_int32, ctypes.POINTER(ForgeHparams), c_int64, c_uint64,
                                               c_void_p]),
    "forge_linear_bwd_step_shard": (c_int32, [ctypes.POINTER(ForgeLinear), ctypes.POINTER(ForgeState),
                                              c_int32, ctypes.POINTER(ForgeHparams), c_int64, c_uint64,
                                              c_int64, c_void_p]),
    "forge_linear_bwd_step_fp8": (c_int32, [ctypes.POINTER(ForgeLinearFp8), ctypes.POINTER(ForgeState),
                                            c_int32, ctypes.POINTER(ForgeHparams), c_int64, c_uint64,
                                            c_void_p]),
    "forge_linear_dgrad": (c_int32, [ctypes.POINTER(ForgeLinear), c_void_p, c_int32, c_void_p]),
    "forge_unfused_wgrad": (c_int32, [ctypes.POINTER(ForgeLinear), c_void_p, c_void_p]),
    "forge_unfused_opt_step": (c_int32, [c_void_p, ctypes.POINTER(ForgeState), c_int64, c_int64,
                                         c_int32, ctypes.POINTER(ForgeHparams), c_int64, c_uint64,
                                         c_void_p]),
    "forge_quantize_state": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int32,
                                       c_void_p]),
    "forge_dequantize_state": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int32,
                                         c_void_p]),
    "forge_quantize_state_block": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int32,
                                             c_int32, c_void_p]),
    "forge_dequantize_state_block": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int32,
                                               c_int32, c_void_p]),
    "forge_get_device_status": (c_int32, [c_void_p]),
    "forge_set_wait_limit_ns": (c_int32, [c_uint64]),
    "forge_debug_skip_loads": (c_int32, [c_int32]),
    "forge_set_step_fusion": (None, [c_int32]),
    "forge_status_string": (ctypes.c_char_p, [c_int32]),
    "forge_last_error_message": (ctypes.c_char_p, []),
    "forge_abi_version": (c_int32, []),
}


def library_path() -> str:
    return os.environ.get("FORGE_LIBRARY", _build.lib_path("libforge.so"))


def lib() -> ctypes.CDLL:
    """The loaded libforge.  Raises if it has not been built (no fallback)."""
    global _lib
    L = _lib
    if L is not None:
        return L
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libforge is not built ({path} missing); run "
                                   "optimizer_tcgen05_dw_gb300.build.build() first")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _check(status: int):
    if status != 0:
        msg = lib().forge_last_error_message().decode(errors="replace")
        raise ForgeError(status, msg)


def _ptr(t):
    return None if t is None else t.data_ptr()


# The current stream's handle without building a torch.cuda.Stream object
# (the call's largest fixed cost otherwise); the public route until CUDA is
# initialised or where these accessors are missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None and _cur_device is not None and torch.cuda.is_initialized():
            return _raw_stream(_cur_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t, name, dtype, shape):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.shape != shape:
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def hparams(**kw) -> ForgeHparams:
    h = dict(HPARAM_DEFAULTS)
    for k, v in kw.items():
        if k not in h:
            raise KeyError(f"unknown hyper-parameter {k}")
        h[k] = v
    return ForgeHparams(**{k: float(v) for k, v in h.items()})


_hp_cache = {}


def _hparams_of(hp: dict) -> ForgeHparams:
    """hparams(**hp), kept for dicts of plain Python numbers (the library only
    reads the struct during the call, so calls may share it)."""
    try:
        key = tuple(hp.items())
        h = _hp_cache.get(key)
    except TypeError:  # an unhashable value
        return hparams(**hp)
    if h is None:
        h = hparams(**hp)
        if all(type(v) in (float, int) for _, v in key):
            if len(_hp_cache) >= 256:
                _hp_cache.clear()
            _hp_cache[key] = h
    return h


def make_state(W, s1=None, s2=None, s1_scale=None, s2_scale=None) -> ForgeState:
    """A forge_state_t for W (fp32 or bf16) and optional fp32 / INT8 states."""
    N, K = W.shape
    wd = W.dtype
    if wd == torch.float32:
        wdt = W_FP32
    elif wd == torch.bfloat16:
        wdt = W_BF16_SR
    else:
        raise TypeError(f"W must be float32 or bfloat16, got {W.dtype}")
    _need(W, "W", wd, (N, K))
    d1 = None if s1 is None else s1.dtype
    d2 = None if s2 is None else s2.dtype
    if d1 in (None, torch.float32) and d2 in (None, torch.float32):  # fp32 or no states
        if s1 is not None:
            _need(s1, "s1", torch.float32, (N, K))
        if s2 is not None:
            _need(s2, "s2", torch.float32, (N, K))
        return ForgeState(W.data_ptr(), wdt, STATE_FP32, _ptr(s1), _ptr(s2), _ptr(s1_scale),
                          _ptr(s2_scale))
    int8 = d1 in (torch.int8, torch.uint8) or d2 in (torch.int8, torch.uint8)
    bf16 = d1 == torch.bfloat16 or d2 == torch.bfloat16
    if bf16:
        for t, nm in ((s1, "s1"), (s2, "s2")):
            if t is not None:
                _need(t, nm, torch.bfloat16, (N, K))
        return ForgeState(_ptr(W), wdt, STATE_BF16, _ptr(s1), _ptr(s2), None, None)
    sdt = STATE_FP32
    if int8:
        # the block width follows from the scale arrays: [N, K / block]
        sc = s1_scale if s1_scale is not None else s2_scale
        if sc is None or sc.dim() != 2 or sc.shape[1] == 0 or K % sc.shape[1] != 0 \
                or K // sc.shape[1] not in INT8_STATE_OF_BLOCK:
            raise ValueError("INT8 states need [N, K / B] float32 scales with B in 32, 64, 128, 256")
        block = K // sc.shape[1]
        sdt = INT8_STATE_OF_BLOCK[block]
        if s1 is not None:
            _need(s1, "s1", torch.int8, (N, K))
            _need(s1_scale, "s1_scale", torch.float32, (N, K // block))
        if s2 is not None:
            _need(s2, "s2", torch.uint8, (N, K))
            _need(s2_scale, "s2_scale", torch.float32, (N, K // block))
    else:
        for t, nm in ((s1, "s1"), (s2, "s2")):
            if t is not None:
                _need(t, nm, torch.float32, (N, K))
    return ForgeState(_ptr(W), wdt, sdt, _ptr(s1), _ptr(s2), _ptr(s1_scale), _ptr(s2_scale))


def forge_linear_bwd_step(X, dY, W, opt: str, hp: dict, step: int, seed: int, s1=None, s2=None,
                          s1_scale=None, s2_scale=None, dX=None, stream=None):
    """The fused FORGE step on one linear layer (updates W and states in place;
    writes dX from the pre-update W when dX is given)."""
    T, K = X.shape
    N = W.shape[0]
    _need(X, "X", torch.bfloat16, (T, K))
    _need(dY, "dY", torch.bfloat16, (T, N))
    if dX is not None:
        _need(dX, "dX", torch.bfloat16, (T, K))
    st = make_state(W, s1, s2, s1_scale, s2_scale)
    lin = ForgeLinear(T, N, K, _ptr(X), _ptr(dY), _ptr(dX))
    _check(lib().forge_linear_bwd_step(ctypes.byref(lin), ctypes.byref(st), OPT_KINDS[opt],
                                       ctypes.byref(_hparams_of(hp)), int(step),
                                       int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def forge_linear_bwd_step_shard(X, dY, W, opt: str, hp: dict, step: int, seed: int, row_offset: int,
                                s1=None, s2=None, s1_scale=None, s2_scale=None, dX=None, stream=None):
    """The FORGE step on rows [row_offset, row_offset + N) of a larger weight
    matrix (a column-parallel shard): dY holds the shard's N columns of the
    upstream gradient, W and the states the shard's rows; stochastic rounding
    uses the elements' indices in the whole matrix.  dX, if given, receives the
    shard's partial input gradient (the layer's dX is the sum over shards)."""
    T, K = X.shape
    N = W.shape[0]
    _need(X, "X", torch.bfloat16, (T, K))
    _need(dY, "dY", torch.bfloat16, (T, N))
    if dX is not None:
        _need(dX, "dX", torch.bfloat16, (T, K))
    st = make_state(W, s1, s2, s1_scale, s2_scale)
    lin = ForgeLinear(T, N, K, _ptr(X), _ptr(dY), _ptr(dX))
    _check(lib().forge_linear_bwd_step_shard(ctypes.byref(lin), ctypes.byref(st), OPT_KINDS[opt],
                                             ctypes.byref(_hparams_of(hp)), int(step),
                                             int(seed) & 0xFFFFFFFFFFFFFFFF, int(row_offset),
                                             _stream(stream)))


def forge_linear_bwd_step_static(X, dY, W, opt: str, hp: dict, step: int, seed: int, s1=None,
                                 s2=None, s1_scale=None, s2_scale=None, dX=None, stream=None):
    """forge_linear_bwd_step with its one-launch scratch in the library's own
    static device array (no allocation; calls on one device must not overlap)."""
    T, K = X.shape
    N = W.shape[0]
    _need(X, "X", torch.bfloat16, (T, K))
    _need(dY, "dY", torch.bfloat16, (T, N))
    if dX is not None:
        _need(dX, "dX", torch.bfloat16, (T, K))
    st = make_state(W, s1, s2, s1_scale, s2_scale)
    lin = ForgeLinear(T, N, K, _ptr(X), _ptr(dY), _ptr(dX))
    _check(lib().forge_linear_bwd_step_static(ctypes.byref(lin), ctypes.byref(st), OPT_KINDS[opt],
                                              ctypes.byref(_hparams_of(hp)), int(step),
                                              int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def forge_linear_bwd_step_fp8(Xt, dYt, x_scale: float, dy_scale: float, W, opt: str, hp: dict,
                              step: int, seed: int, s1=None, s2=None, s1_scale=None, s2_scale=None,
                              stream=None):
    """The FORGE step from E4M3 operands: Xt [K, T] and dYt [N, T] codes
    (torch.float8_e4m3fn or uint8), token-contiguous, with one scale each;
    updates the bf16 W and the states in place (no dX)."""
    K, T = Xt.shape
    N = W.shape[0]
    for t, name, shape in ((Xt, "Xt", (K, T)), (dYt, "dYt", (N, T))):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError(f"{name}: expected torch.float8_e4m3fn or uint8 E4M3 codes, got {t.dtype}")
        _need(t, name, t.dtype, shape)
    st = make_state(W, s1, s2, s1_scale, s2_scale)
    lin = ForgeLinearFp8(T, N, K, _ptr(Xt), _ptr(dYt), float(x_scale), float(dy_scale))
    _check(lib().forge_linear_bwd_step_fp8(ctypes.byref(lin), ctypes.byref(st), OPT_KINDS[opt],
                                           ctypes.byref(_hparams_of(hp)), int(step),
                                           int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def forge_linear_dgrad(dY, W, dX, stream=None):
    T, N = dY.shape
    K = W.shape[1]
    _need(dY, "dY", torch.bfloat16, (T, N))
    _need(dX, "dX", torch.bfloat16, (T, K))
    _need(W, "W", W.dtype, (N, K))
    wdt = W_FP32 if W.dtype == torch.float32 else W_BF16_SR
    lin = ForgeLinear(T, N, K, None, _ptr(dY), _ptr(dX))
    _check(lib().forge_linear_dgrad(ctypes.byref(lin), _ptr(W), wdt, _stream(stream)))


def forge_unfused_wgrad(X, dY, dW, stream=None):
    T, K = X.shape
    N = dY.shape[1]
    _need(X, "X", torch.bfloat16, (T, K))
    _need(dY, "dY", torch.bfloat16, (T, N))
    _need(dW, "dW", torch.float32, (N, K))
    lin = ForgeLinear(T, N, K, _ptr(X), _ptr(dY), None)
    _check(lib().forge_unfused_wgrad(ctypes.byref(lin), _ptr(dW), _stream(stream)))


def forge_unfused_opt_step(dW, W, opt: str, hp: dict, step: int, seed: int, s1=None, s2=None,
                           s1_scale=None, s2_scale=None, stream=None):
    N, K = W.shape
    if dW is not None:
        _need(dW, "dW", torch.float32, (N, K))
    st = make_state(W, s1, s2, s1_scale, s2_scale)
    _check(lib().forge_unfused_opt_step(_ptr(dW), ctypes.byref(st), N, K, OPT_KINDS[opt],
                                        ctypes.byref(_hparams_of(hp)), int(step),
                                        int(seed) & 0xFFFFFFFFFFFFFFFF, _stream(stream)))


def forge_quantize_state(x, codes, absmax, is_signed: bool, stream=None, block: int = 64):
    """x fp32 [rows, cols] -> INT8 codes and absmax [rows, cols / block]."""
    rows, cols = x.shape
    _need(x, "x", torch.float32, (rows, cols))
    _need(codes, "codes", torch.int8 if is_signed else torch.uint8, (rows, cols))
    _need(absmax, "absmax", torch.float32, (rows, cols // block))
    _check(lib().forge_quantize_state_block(_ptr(x), _ptr(codes), _ptr(absmax), rows, cols,
                                            1 if is_signed else 0, int(block), _stream(stream)))


def forge_dequantize_state(codes, absmax, x, is_signed: bool, stream=None, block: int = 64):
    rows, cols = x.shape
    _need(x, "x", torch.float32, (rows, cols))
    _need(codes, "codes", torch.int8 if is_signed else torch.uint8, (rows, cols))
    _need(absmax, "absmax", torch.float32, (rows, cols // block))
    _check(lib().forge_dequantize_state_block(_ptr(codes), _ptr(absmax), _ptr(x), rows, cols,
                                              1 if is_signed else 0, int(block), _stream(stream)))


def forge_get_device_status(stream=None):
    """Synchronises the stream; raises ForgeError if a kernel reported an error."""
    _check(lib().forge_get_device_status(_stream(stream)))


def forge_set_wait_limit_ns(ns: int):
    _check(lib().forge_set_wait_limit_ns(int(ns)))


def forge_set_step_fusion(enable: bool):
    """Allow (default) or forbid the one-launch dX + FORGE step."""
    lib().forge_set_step_fusion(1 if enable else 0)


def forge_debug_skip_loads(enable: bool):
    _check(lib().forge_debug_skip_loads(1 if enable else 0))


def forge_abi_version() -> int:
    return int(lib().forge_abi_version())
