// Per-element arithmetic of the FORGE step: the eight elementwise rules,
// Philox4x32-10, bf16 stochastic rounding and the block-64 INT8 state code.
//
// Every floating-point operation is written with an explicit round-to-nearest
// intrinsic (__fmul_rn, __fadd_rn, __fsub_rn, __fdiv_rn, __fsqrt_rn), so no
// multiply-add contraction or approximate division can change a result: the
// same per-element sequence runs in the fused epilogue and in the standalone
// optimizer kernel, and each rule is one fixed sequence of IEEE float32
// operations (the order is given next to each rule).
//
// Method: "FORGE: Fused On-Register Gradient Elimination" (gist.science
// explainer), Technical Summary §2 "Precision and Fidelity" (FP32 gradient,
// stochastic rounding of BF16 weights, INT8 states in blocks of 64) and §3
// "Generality" (the eight rules).
#pragma once

#include <cstdint>

#include "common.h"

namespace forge {
namespace dev {

__device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float dvd(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ float sqr(float a) { return __fsqrt_rn(a); }

// sign with sign(+-0) = +0 and NaN passed through.
__device__ __forceinline__ float sign0(float c) {
  return c > 0.f ? 1.f : (c < 0.f ? -1.f : (c == 0.f ? 0.f : c));
}

// One step of rule KIND on one element.  w: current weight (fp32 value),
// g: fp32 gradient, s1/s2: dequantised states (updated in place).
// Orders (each operation rounded):
//   AdamW  m = b1*m + omb1*g;  v = b2*v + omb2*(g*g);  d = sqrt(v)*inv_sqrt_c2 + eps;
//          w = w*decay - step_size*(m/d)
//   NAdam  g += l2*w;  m, v as AdamW;  d = sqrt(v*inv_c2) + eps;
//          w = w - coef_g*(g/d);  w = w - coef_m*(m/d)
//   RAdam  g += l2*w;  m, v as AdamW;  rectified: d = sqrt(v) + eps;
//          w = w - step_size*((m*sqrt_c2)/d);  otherwise w = w - step_size*m
//   Lion   c = b1*m + omb1*g;  w = w*decay - lr*sign(c);  m = b2*m + omb2*g
//   RMSprop g += l2*w;  v = alpha*v + oma*(g*g);  w = w - lr*(g/(sqrt(v) + eps))
//   AdaGrad g += l2*w;  v = v + g*g;  w = w - lr*(g/(sqrt(v) + eps))
//   SGD    g += l2*w;  w = w - lr*g
//   SGD-m  g += l2*w;  b = mom*b + g;  w = w - lr*b
template <int KIND>
__device__ __forceinline__ void rule(float& w, float g, float& s1, float& s2,
                                     const OptScalars& sc) {
  if (KIND != kAdamW && KIND != kLion) {
    if (sc.l2 != 0.f) g = add(g, mul(sc.l2, w));
  }
  if (KIND == kAdamW || KIND == kNAdam || KIND == kRAdam) {
    const float m = add(mul(sc.b1, s1), mul(sc.omb1, g));
    const float v = add(mul(sc.b2, s2), mul(sc.omb2, mul(g, g)));
    if (KIND == kAdamW) {
      const float d = add(mul(sqr(v), sc.inv_sqrt_c2), sc.eps);
      w = sub(mul(w, sc.decay), mul(sc.step_size, dvd(m, d)));
    } else if (KIND == kNAdam) {
      const float d = add(sqr(mul(v, sc.inv_c2)), sc.eps);
      w = sub(w, mul(sc.coef_g, dvd(g, d)));
      w = sub(w, mul(sc.coef_m, dvd(m, d)));
    } else {
      if (sc.rectified) {
        const float d = add(sqr(v), sc.eps);
        w = sub(w, mul(sc.step_size, dvd(mul(m, sc.sqrt_c2), d)));
      } else {
        w = sub(w, mul(sc.step_size, m));
      }
    }
    s1 = m;
    s2 = v;
  } else if (KIND == kLion) {
    const float c = add(mul(sc.b1, s1), mul(sc.omb1, g));
    w = sub(mul(w, sc.decay), mul(sc.lr, sign0(c)));
    s1 = add(mul(sc.b2, s1), mul(sc.omb2, g));
  } else if (KIND == kRMSprop) {
    const float v = add(mul(sc.alpha, s2), mul(sc.oma, mul(g, g)));
    w = sub(w, mul(sc.lr, dvd(g, add(sqr(v), sc.eps))));
    s2 = v;
  } else if (KIND == kAdaGrad) {
    const float v = add(s2, mul(g, g));
    w = sub(w, mul(sc.lr, dvd(g, add(sqr(v), sc.eps))));
    s2 = v;
  } else if (KIND == kSGD) {
    w = sub(w, mul(sc.lr, g));
  } else {  // kSGDMomentum
    const float b = add(mul(sc.mom, s1), g);
    w = sub(w, mul(sc.lr, b));
    s1 = b;
  }
}

// ------------------------------------------------------------------ Philox

// Philox4x32 with 10 rounds (Salmon et al., SC'11): per round, the 32x32->64
// products of counter words 0 and 2 with two odd multipliers; the key is
// bumped by the Weyl constants before every round after the first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The 4 random words covering elements 8*grp .. 8*grp+7 of a weight matrix.
__device__ __forceinline__ uint4 sr_words(uint64_t grp, uint64_t seed, uint64_t step) {
  const uint4 ctr = make_uint4(static_cast<uint32_t>(grp), static_cast<uint32_t>(grp >> 32),
                               static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32));
  return philox4x32_10(ctr, static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

// The same words with the ten rounds' keys formed ahead (round_keys[2r],
// round_keys[2r + 1] = the key after r bumps), e.g. once per launch.
__device__ __forceinline__ uint4 sr_words_rk(uint64_t grp, uint64_t step, const uint32_t* round_keys) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  uint4 c = make_uint4(static_cast<uint32_t>(grp), static_cast<uint32_t>(grp >> 32),
                       static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32));
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(kM0, c.x), lo0 = kM0 * c.x;
    const uint32_t hi1 = __umulhi(kM1, c.z), lo1 = kM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ round_keys[2 * r], lo1, hi0 ^ c.w ^ round_keys[2 * r + 1], lo0);
  }
  return c;
}

// 16 random bits of element j (0..7) of a group.
__device__ __forceinline__ uint32_t sr_bits(const uint4& r, int j) {
  const uint32_t w = (j >> 1) == 0 ? r.x : (j >> 1) == 1 ? r.y : (j >> 1) == 2 ? r.z : r.w;
  return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// fp32 -> bf16 bits by stochastic rounding: add the 16 random bits to the
// fp32 pattern and keep the upper half.  NaN -> 0x7FC0, +-Inf kept.
__device__ __forceinline__ uint32_t bf16_sr(float x, uint32_t r16) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t mag = u & 0x7FFFFFFFu;
  if (mag > 0x7F800000u) return 0x7FC0u;
  if (mag == 0x7F800000u) return u >> 16;
  return (u + r16) >> 16;  // largest finite 0xFF7FFFFF + 0xFFFF does not wrap
}

__device__ __forceinline__ float bf16_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// fp32 -> bf16 bits, round to nearest, ties to even (BF16 moments).  NaN ->
// 0x7FC0; a value past the largest finite bf16 rounds to Inf.
__device__ __forceinline__ uint32_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;  // no wrap: at most 0xFF800000 + 0x8000
}

// ------------------------------------------------------------------ INT8 code

// Value of one code of a block with absmax `a`: code * (a / 127) or (a / 255).
template <bool SIGNED>
__device__ __forceinline__ float dequant(int code, float a) {
  const float s = dvd(a, SIGNED ? 127.f : 255.f);
  return mul(static_cast<float>(code), s);
}

// Code of x in a block with absmax `a` (s = a/127 or a/255): clamp(rint(x/s)),
// 0 when a == 0 or x/s is NaN.
template <bool SIGNED>
__device__ __forceinline__ int quant(float x, float a) {
  if (a == 0.f) return 0;
  const float s = dvd(a, SIGNED ? 127.f : 255.f);
  const float r = dvd(x, s);
  if (r != r) return 0;
  float q = rintf(r);
  q = fminf(fmaxf(q, SIGNED ? -127.f : 0.f), SIGNED ? 127.f : 255.f);
  return static_cast<int>(q);
}

// quant<SIGNED>(x, a) with the block's step s = a/127 (or a/255) and its
// reciprocal inv = RN(1/s) formed once per block: the same code, mostly
// without the division.  y = RN(x * inv) = (x/s)(1 + e1)(1 + e2) with
// |e1|, |e2| <= 2^-24, so |y - x/s| <= 2^-23 (1 + 2^-25) |x/s| < 1.6e-5 for
// |x/s| <= 128, and RN(x/s) lies within 2^-24 * 128 < 7.7e-6 of x/s: y and
// RN(x/s) round to the same integer unless a half-integer lies within
// 2.4e-5 of y.  There (and whenever inv is not finite) the quotient is
// formed exactly as in quant; elsewhere rint(y) is the code.
template <bool SIGNED>
__device__ __forceinline__ int quant_recip(float x, float a, float s, float inv) {
  if (a == 0.f) return 0;
  const float y = mul(x, inv);
  const float fr = __fsub_rn(y, floorf(y));  // exact for |y| < 2^23
  const float r = (fabsf(__fsub_rn(fr, 0.5f)) <= 3.0e-5f || !(fabsf(inv) <= 3.0e38f)) ? dvd(x, s) : y;
  if (r != r) return 0;
  float q = rintf(r);
  q = fminf(fmaxf(q, SIGNED ? -127.f : 0.f), SIGNED ? 127.f : 255.f);
  return static_cast<int>(q);
}

// The fused epilogue's INT8 arithmetic, written to keep off the conversion
// unit (int <-> float casts and floor/rint run there at a fraction of the FP32
// rate); every function gives the same values as the definitions above.
//
// Code k (0..3) of a word of four packed codes, as a float: the byte placed
// under the exponent of 2^23 (bit pattern 0x4B0000cc) is 2^23 + c exactly, so
// one subtraction gives c.  Signed codes are flipped to c + 128 first.
template <bool SIGNED>
__device__ __forceinline__ float code_f32(uint32_t word, int k) {
  const uint32_t biased = __byte_perm(SIGNED ? (word ^ 0x80808080u) : word, 0x4B000000u, 0x7440u | k);
  return __fsub_rn(__uint_as_float(biased), SIGNED ? 8388736.f : 8388608.f);
}

// clamp(rint(y)) as an integer, NaN -> 0: adding 1.5 * 2^23 rounds any |y| <
// 2^22 to an integer (nearest even) held in the low mantissa bits.  `near`
// reports a y within 3e-5 of a half-integer (see quant_recip), where the
// rounding of y and of the exact quotient may differ.  CLAMP = false is for
// y = x * RN(1/s) with a finite reciprocal and |x| <= absmax: then s >=
// 3.3e-39, whose relative spacing is below 5e-7, so |y| <= 127.0001 (255.0002
// unsigned, where x >= 0) and the clamp would never change the rounded code.
constexpr float kShifter = 12582912.f;
template <bool SIGNED, bool CLAMP = true>
__device__ __forceinline__ int code_round(float y, bool& near) {
  const float yc = CLAMP ? fminf(fmaxf(y, SIGNED ? -127.f : 0.f), SIGNED ? 127.f : 255.f) : y;
  const float t = __fadd_rn(yc, kShifter);
  near = fabsf(__fsub_rn(yc, __fsub_rn(t, kShifter))) >= 0.49997f;
  const int k = static_cast<int>(__float_as_uint(t) - 0x4B400000u);
  return (y == y) ? k : 0;
}

// code_round<SIGNED, false> without its NaN test, for a caller that forms all
// codes of a group again from the exact quotient (code_round) whenever one
// reports `redo`: the comparison is written so that a NaN y (and an infinite
// one) reports it.  Returns the bit pattern of y + 1.5 * 2^23, whose low byte
// is the code (two's complement for a negative one) that code_round<SIGNED,
// false> gives for every other y: 1.5 * 2^23 has a zero low byte.
template <bool SIGNED>
__device__ __forceinline__ uint32_t code_round_fast(float y, bool& redo) {
  const float t = __fadd_rn(y, kShifter);
  redo = !(fabsf(__fsub_rn(y, __fsub_rn(t, kShifter))) < 0.49997f);
  return __float_as_uint(t);
}

// Running absmax that never takes a NaN (NaN > a is false).
__device__ __forceinline__ float absmax_acc(float a, float x) {
  const float ax = fabsf(x);
  return ax > a ? ax : a;
}

}  // namespace dev
}  // namespace forge
