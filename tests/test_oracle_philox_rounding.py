"""Pins for the oracle's Philox4x32-10, bf16 rounding and stochastic rounding.

Philox is checked against an independent implementation: Triton's
``tl.philox`` evaluated on the CPU by Triton's interpreter.  Round-to-nearest
bf16 is checked against torch's float32 -> bfloat16 cast.  Stochastic rounding
is checked against a hand-worked fixture (tests/golden/sr_bf16.json), exact
unbiasedness over all 2^16 random values, and the explainer's dead-zone claim
(Technical Summary §2, "Precision and Fidelity").
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import philox, rounding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def _k(c_ptr, out_ptr, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + i * 4 + 0)
    c1 = tl.load(c_ptr + i * 4 + 1)
    c2 = tl.load(c_ptr + i * 4 + 2)
    c3 = tl.load(c_ptr + i * 4 + 3)
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + i * 4 + 0, a)
    tl.store(out_ptr + i * 4 + 1, b)
    tl.store(out_ptr + i * 4 + 2, c)
    tl.store(out_ptr + i * 4 + 3, d)

req = json.loads(sys.stdin.read())
res = []
for seed, ctrs in req:
    c = torch.tensor(np.array(ctrs, dtype=np.uint32).view(np.int32))
    out = torch.zeros_like(c)
    _k[(1,)](c, out, seed, N=c.shape[0])
    res.append(out.numpy().view(np.uint32).tolist())
print(json.dumps(res))
"""


def _triton_philox(requests):
    pytest.importorskip("triton")
    proc = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(requests),
                          capture_output=True, text=True, timeout=300)
    if proc.returncode != 0:
        pytest.skip("Triton interpreter unavailable: " + proc.stderr.strip().splitlines()[-1])
    return json.loads(proc.stdout.strip().splitlines()[-1])


def test_philox_matches_triton_interpreter():
    rng = np.random.default_rng(7)
    seeds = [0, 1, 0x123456789ABCDEF0, (1 << 64) - 1 >> 1, 20260623]
    requests = []
    for s in seeds:
        ctrs = rng.integers(0, 2 ** 32, size=(8, 4), dtype=np.uint64).astype(np.uint32)
        ctrs[0] = 0
        ctrs[1] = [0xFFFFFFFF] * 4
        requests.append([s, ctrs.tolist()])
    got = _triton_philox(requests)
    for (s, ctrs), ref in zip(requests, got):
        mine = philox.philox4x32_10(np.array(ctrs, dtype=np.uint32), s & 0xFFFFFFFF, s >> 32)
        assert np.array_equal(mine, np.array(ref, dtype=np.uint32)), hex(s)


def test_sr_random16_uses_the_counter_layout():
    # element idx -> counter (idx>>3, step), word (idx&7)>>1, half idx&1
    seed, step = 0xDEADBEEF12345678, 7
    idx = np.arange(64, dtype=np.int64) + (1 << 33)
    r = philox.sr_random16(idx, seed, step)
    assert r.max() <= 0xFFFF
    for base in range(0, 64, 8):
        g = int(idx[base] >> 3)
        ctr = np.array([[g & 0xFFFFFFFF, g >> 32, step, 0]], dtype=np.uint32)
        words = philox.philox4x32_10(ctr, seed & 0xFFFFFFFF, seed >> 32)[0]
        halves = [int(w) >> (16 * h) & 0xFFFF for w in words for h in (0, 1)]
        assert r[base:base + 8].tolist() == halves


def test_sr_random16_is_uniform():
    r = philox.sr_random16(np.arange(1 << 18, dtype=np.int64), 99, 3)
    counts = np.bincount(r >> 12, minlength=16)  # 16 bins of the top 4 bits
    expected = r.size / 16
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 50.0  # 15 dof; p ~ 1e-5


def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(3.0),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1e-40, 1.00390625,
                  1.01171875, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rounding.bf16_bits_rne(x), ref)


def test_bf16_rne_nan_is_canonical():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    assert rounding.bf16_bits_rne(x).tolist() == [0x7FC0, 0x7FC0]


def test_sr_golden_fixture():
    with open(os.path.join(GOLDEN, "sr_bf16.json")) as f:
        cases = json.load(f)["cases"]
    for xb, rb, want in cases:
        x = np.array([int(xb, 16)], dtype=np.uint32).view(np.float32)
        got = rounding.bf16_bits_stochastic(x, np.array([int(rb, 16)], dtype=np.uint32))
        assert int(got[0]) == int(want, 16), (xb, rb)


def test_sr_is_exactly_unbiased_over_all_random_values():
    rng = np.random.default_rng(3)
    xs = (rng.standard_normal(200) * 10.0).astype(np.float32)
    r = np.arange(1 << 16, dtype=np.uint32)
    for x in xs:
        b = rounding.bf16_bits_stochastic(np.full(r.shape, x, dtype=np.float32), r)
        mean = rounding.bf16_bits_to_f32(b).astype(np.float64).mean()
        assert mean == pytest.approx(float(x), rel=0, abs=abs(float(x)) * 1e-12)


def test_sr_escapes_the_bf16_dead_zone():
    """A sub-ULP update below 1.0 vanishes under round-to-nearest, but its
    expectation survives stochastic rounding keyed by Philox (§2 dead zone)."""
    x = np.float32(1.0) - np.float32(1e-4)
    assert rounding.bf16_bits_rne(np.array([x]))[0] == 0x3F80  # RNE: exactly 1.0
    n = 1 << 16
    r16 = philox.sr_random16(np.arange(n, dtype=np.int64), 20260623, 1)
    vals = rounding.bf16_bits_to_f32(
        rounding.bf16_bits_stochastic(np.full(n, x, dtype=np.float32), r16)).astype(np.float64)
    # values are 1 - 2^-8 (prob p) or 1.0; p = (1 - x) / 2^-8
    p = (1.0 - float(x)) / 2 ** -8
    sigma = np.sqrt(p * (1 - p) / n) * 2 ** -8
    assert abs(vals.mean() - float(x)) < 4 * sigma


def test_sr_round_up_probability_matches_fraction():
    rng = np.random.default_rng(11)
    n = 1 << 15
    for frac_bits in (0x1000, 0x5555, 0xC000):
        u = np.uint32(0x40490000 | frac_bits)  # 3.14..., fixed dropped bits
        x = np.full(n, u, dtype=np.uint32).view(np.float32)
        r16 = philox.sr_random16(rng.integers(0, 1 << 40, size=n), 5, 2)
        up = (rounding.bf16_bits_stochastic(x, r16) == 0x404A).mean()
        p = frac_bits / 65536
        assert abs(up - p) < 4 * np.sqrt(p * (1 - p) / n)
