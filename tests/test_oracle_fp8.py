"""Pins for the oracle's E4M3 decoding and FP8 weight gradient (oracle/fp8.py):
torch's float8_e4m3fn (an independent implementation) on all 256 codes, the
format's landmarks, and a brute-force exact sum."""

from fractions import Fraction

import numpy as np
import torch

from oracle import fp8


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8.e4m3_bits_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all(), np.argwhere(~same)[:5]
    assert np.array_equal(np.signbit(ours[~np.isnan(ours)]), np.signbit(ref[~np.isnan(ref)]))


def test_landmarks():
    d = fp8.e4m3_bits_to_f32(np.array([0x38, 0x7E, 0x01, 0x08, 0x7F, 0xFF, 0x80, 0xB8], np.uint8))
    assert d[0] == 1.0 and d[1] == 448.0 and d[2] == 2.0 ** -9 and d[3] == 2.0 ** -6
    assert np.isnan(d[4]) and np.isnan(d[5])
    assert d[6] == 0.0 and np.signbit(d[6]) and d[7] == -1.0


def test_weight_gradient_is_the_exact_scaled_sum():
    rng = np.random.default_rng(3)
    T, N, K = 7, 3, 5
    xt = rng.integers(0, 256, (K, T)).astype(np.uint8)
    dyt = rng.integers(0, 256, (N, T)).astype(np.uint8)
    xt[(xt & 0x7F) == 0x7F] = 0x38  # no NaN codes
    dyt[(dyt & 0x7F) == 0x7F] = 0x40
    sx, sdy = 0.375, 3.0e-4
    g = fp8.weight_gradient_fp8(xt, dyt, sx, sdy)
    X = fp8.e4m3_bits_to_f32(xt)
    dY = fp8.e4m3_bits_to_f32(dyt)
    c = np.float32(Fraction(float(np.float32(sx))) * Fraction(float(np.float32(sdy))))
    for n in range(N):
        for k in range(K):
            s = sum(Fraction(float(dY[n, t])) * Fraction(float(X[k, t])) for t in range(T))
            want = np.float32(np.float32(s) * c)  # each product rounded once to float32
            assert g[n, k] == want, (n, k, g[n, k], want)
