"""Seeded synthetic inputs for FORGE linear-layer steps.

This module only draws random tensors and describes workload shapes; it holds
none of the method's arithmetic.  Both the CUDA path's callers (tests, bench)
and the CPU oracle's callers take their inputs from here.

Distributions follow the workloads the FORGE explainer evaluates (Technical
Summary §4: Llama-3.1-8B and the Qwen3 family) as linear-layer shapes only:
activations X ~ N(0, 1), upstream gradients dY ~ N(0, sigma) with small sigma,
weights ~ N(0, 0.02); "N(0, s)" means standard deviation s.  No weights,
datasets or benchmark items are used: everything is drawn from a seed.
"""

from dataclasses import dataclass, field

import numpy as np
import torch

# ----------------------------------------------------------------------------
# Layer shapes (out_features N, in_features K) of one decoder layer
# ----------------------------------------------------------------------------

LLAMA31_8B_LINEARS = [  # hidden 4096, 32 q heads / 8 kv heads of 128, MLP 14336
    ("q_proj", 4096, 4096), ("k_proj", 1024, 4096), ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096), ("gate_proj", 14336, 4096), ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
]
QWEN3_14B_LINEARS = [  # hidden 5120, 40 q heads / 8 kv heads of 128, MLP 17408
    ("q_proj", 5120, 5120), ("k_proj", 1024, 5120), ("v_proj", 1024, 5120),
    ("o_proj", 5120, 5120), ("gate_proj", 17408, 5120), ("up_proj", 17408, 5120),
    ("down_proj", 5120, 17408),
]
QWEN3_14B_LAYERS = 40


@dataclass
class Workload:
    """One synthetic workload: layer shapes, token count, dtypes, optimizer."""
    name: str
    linears: list
    T: int
    w_dtype: str            # "fp32" | "bf16"
    s_dtype: str            # "fp32" | "int8"
    opt: str                # optimizer name
    hparams: dict
    steps: int
    x_std: float = 1.0
    dy_std: float = 1e-3
    w_std: float = 0.02
    m_init_std: float = 0.0  # pre-warmed moments (0 = start from zero)
    v_init_std: float = 0.0
    layers: int = 1
    extra: dict = field(default_factory=dict)


ADAMW_LLAMA = dict(lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)

WORKLOADS = {
    "single_256": Workload(
        "single linear 256x256, T=512, fp32 master W, fp32 AdamW, 3 steps",
        [("linear", 256, 256)], 512, "fp32", "fp32", "adamw",
        dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01), 3,
        x_std=1.0, dy_std=1e-2),
    "llama8b_bf16_fp32state": Workload(
        "Llama-3.1-8B decoder-layer linears, T=16384, bf16 W (stochastic rounding), "
        "fp32 AdamW moments, 10 steps",
        LLAMA31_8B_LINEARS, 16384, "bf16", "fp32", "adamw", ADAMW_LLAMA, 10),
    "llama8b_bf16_int8state": Workload(
        "Llama-3.1-8B decoder-layer linears, T=16384, bf16 W (stochastic rounding), "
        "INT8 block-64 AdamW moments (pre-warmed), 10 steps",
        LLAMA31_8B_LINEARS, 16384, "bf16", "int8", "adamw", ADAMW_LLAMA, 10,
        m_init_std=1e-4, v_init_std=1e-6),
    "sweep_4096": Workload(
        "W 4096x4096 bf16, T=8192, fp32 states, 8 optimizers x 5 steps",
        [("linear", 4096, 4096)], 8192, "bf16", "fp32", "all", {}, 5),
    "qwen14b_int8": Workload(
        "Qwen3-14B decoder-layer linears x 40 layers, T=4096, bf16 W (stochastic "
        "rounding), INT8 block-64 AdamW moments",
        QWEN3_14B_LINEARS, 4096, "bf16", "int8", "adamw", ADAMW_LLAMA, 1,
        layers=QWEN3_14B_LAYERS),
}

SWEEP_HPARAMS = {
    "adamw": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
    "nadam": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
    "radam": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
    "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=0.1),
    "rmsprop": dict(lr=1e-3, alpha=0.99, eps=1e-8),
    "adagrad": dict(lr=1e-2, eps=1e-10),
    "sgd": dict(lr=1e-2),
    "sgd_momentum": dict(lr=1e-2, momentum=0.9),
}


# ----------------------------------------------------------------------------
# Random tensors
# ----------------------------------------------------------------------------

def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal(shape, std: float, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0, std) drawn in float32 from a seeded generator, then cast (bf16 casts
    round to nearest even)."""
    t = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return (t * std).to(dtype)


def abs_normal(shape, std: float, seed: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    return normal(shape, std, seed, torch.float32, device).abs().to(dtype)


def integer_grid(shape, lo: int, hi: int, pow2_scale: int, seed: int,
                 dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Integers uniform in [lo, hi] times 2**pow2_scale (exact in bf16 for small
    ranges), so that sums of their products are exact in float32."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed, device), device=device,
                      dtype=torch.int32)
    return (t.to(torch.float32) * (2.0 ** pow2_scale)).to(dtype)


def e4m3_integer_grid(shape, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """E4M3 codes (uint8) of integers uniform in [lo, hi] (exact for |x| <= 16)."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed, device), device=device,
                      dtype=torch.int32)
    return t.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def e4m3_normal(shape, std: float, seed: int, device="cpu"):
    """N(0, std) drawn in float32, divided by a power-of-two per-tensor scale
    that brings the largest magnitude to at most 448 (the largest finite E4M3
    value), and cast to E4M3 (nearest even).  Returns (codes as uint8, scale)."""
    t = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32) * std
    amax = float(t.abs().max()) if t.numel() else 0.0
    scale = 2.0 ** int(np.ceil(np.log2(amax / 448.0))) if amax > 0 else 1.0
    return (t / scale).to(torch.float8_e4m3fn).view(torch.uint8), scale


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (on the CPU)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


def layer_seed(base: int, layer: int, step: int, what: int) -> int:
    """A distinct seed per (workload seed, layer, step, tensor kind)."""
    return (base * 1_000_003 + layer * 10_007 + step * 101 + what) & 0x7FFFFFFF
