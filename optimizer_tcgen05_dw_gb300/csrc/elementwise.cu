// Elementwise kernels: the standalone optimizer step of the unfused schedule,
// the INT8 state quantiser/dequantiser, and dX for fp32 master weights.
//
// The optimizer step runs exactly the per-element arithmetic of the fused
// epilogue (optim.cuh) on a gradient read from global memory -- the
// "separate optimizer kernel launch" the FORGE explainer's Technical Summary
// §4 ("Throughput") names as the cost the fused step removes.
//
// Layout of work: each thread owns 8 consecutive elements of a row (one
// Philox call, 16/32-byte vector accesses; consecutive threads own
// consecutive groups, so a warp touches 256 contiguous elements).  For INT8
// states the qblock/8 threads of a block (4, 8, 16 or 32 lanes for blocks of
// 32, 64, 128 or 256) share the block's absmax through warp shuffles.
#include <cuda_bf16.h>

#include "launch.h"
#include "optim.cuh"

namespace forge {

namespace {

constexpr int kElemThreads = 256;

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Max over the `lanes` lanes (a power of two up to 32) of an aligned lane
// group; all 32 lanes call it.
__device__ __forceinline__ float group_max(float a, int lanes) {
  for (int o = 1; o < lanes; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  return a;
}

template <bool SIGNED>
__device__ __forceinline__ void load_codes8(const void* base, int64_t e0, float a, float (&v)[8]) {
  const uint2 c = *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(base) + e0);
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
    const int code = SIGNED ? static_cast<int>(static_cast<int8_t>(b)) : static_cast<int>(b);
    v[j] = dev::dequant<SIGNED>(code, a);
  }
}

template <bool SIGNED>
__device__ __forceinline__ void store_codes8(void* base, int64_t e0, float a, const float (&v)[8]) {
  uint32_t w[2] = {0u, 0u};
  const float st = dev::dvd(a, SIGNED ? 127.f : 255.f), inv = dev::dvd(1.f, st);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w[j >> 2] |= (static_cast<uint32_t>(dev::quant_recip<SIGNED>(v[j], a, st, inv)) & 0xFFu) << (8 * (j & 3));
  *reinterpret_cast<uint2*>(static_cast<uint8_t*>(base) + e0) = make_uint2(w[0], w[1]);
}

__device__ __forceinline__ void load_bf16x8(const void* base, int64_t e0, float (&v)[8]) {
  const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + e0);
  const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = dev::bf16_to_f32(w[j] & 0xFFFFu);
    v[2 * j + 1] = dev::bf16_to_f32(w[j] >> 16);
  }
}

__device__ __forceinline__ void store_bf16x8_rne(void* base, int64_t e0, const float (&v)[8]) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) o[j] = dev::bf16_rne(v[2 * j]) | (dev::bf16_rne(v[2 * j + 1]) << 16);
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + e0) = make_uint4(o[0], o[1], o[2], o[3]);
}

template <int KIND, int WDT, int SDT>
__device__ __forceinline__ void opt_group(int64_t gid, bool active, const ElemParams& p) {
  const int64_t e0 = gid * 8;
  float g[8], w[8], s1[8], s2[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) { g[j] = 0.f; w[j] = 0.f; s1[j] = 0.f; s2[j] = 0.f; }
  // block index (rows hold K/qblock whole blocks)
  const int64_t sidx = SDT == kSInt8 ? e0 / p.qblock : 0;
  if (active) {
    if (p.dW != nullptr) load8(p.dW + e0, g);
    if (WDT == kWBf16) {
      const uint4 wb = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.W) + e0);
      const uint32_t wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[2 * j] = dev::bf16_to_f32(wv[j] & 0xFFFFu);
        w[2 * j + 1] = dev::bf16_to_f32(wv[j] >> 16);
      }
    } else {
      load8(static_cast<const float*>(p.W) + e0, w);
    }
    if (SDT == kSInt8) {
      if (uses_s1(KIND)) load_codes8<true>(p.s1, e0, p.s1_scale[sidx], s1);
      if (uses_s2(KIND)) load_codes8<false>(p.s2, e0, p.s2_scale[sidx], s2);
    } else if (SDT == kSBf16) {
      if (uses_s1(KIND)) load_bf16x8(p.s1, e0, s1);
      if (uses_s2(KIND)) load_bf16x8(p.s2, e0, s2);
    } else {
      if (uses_s1(KIND)) load8(static_cast<const float*>(p.s1) + e0, s1);
      if (uses_s2(KIND)) load8(static_cast<const float*>(p.s2) + e0, s2);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) dev::rule<KIND>(w[j], g[j], s1[j], s2[j], p.sc);
    if (WDT == kWBf16) {
      const uint4 r = dev::sr_words((static_cast<uint64_t>(e0) >> 3) + p.sr_base, p.seed, p.step);
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = dev::bf16_sr(w[2 * j], dev::sr_bits(r, 2 * j)) |
               (dev::bf16_sr(w[2 * j + 1], dev::sr_bits(r, 2 * j + 1)) << 16);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.W) + e0) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      store8(static_cast<float*>(p.W) + e0, w);
    }
    if (SDT == kSFp32) {
      if (uses_s1(KIND)) store8(static_cast<float*>(p.s1) + e0, s1);
      if (uses_s2(KIND)) store8(static_cast<float*>(p.s2) + e0, s2);
    } else if (SDT == kSBf16) {
      if (uses_s1(KIND)) store_bf16x8_rne(p.s1, e0, s1);
      if (uses_s2(KIND)) store_bf16x8_rne(p.s2, e0, s2);
    }
  }
  if (SDT == kSInt8) {
    // new block absmax over the 8 threads of this block (inactive threads
    // belong to inactive blocks and contribute nothing)
    float n1 = 0.f, n2 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      n1 = dev::absmax_acc(n1, s1[j]);
      n2 = dev::absmax_acc(n2, s2[j]);
    }
    if (uses_s1(KIND)) n1 = group_max(n1, p.qblock / 8);
    if (uses_s2(KIND)) n2 = group_max(n2, p.qblock / 8);
    if (active) {
      const bool leader = (gid & (p.qblock / 8 - 1)) == 0;
      if (uses_s1(KIND)) {
        store_codes8<true>(p.s1, e0, n1, s1);
        if (leader) p.s1_scale[sidx] = n1;
      }
      if (uses_s2(KIND)) {
        store_codes8<false>(p.s2, e0, n2, s2);
        if (leader) p.s2_scale[sidx] = n2;
      }
    }
  }
}

template <int WDT, int SDT>
__global__ void __launch_bounds__(kElemThreads) opt_step_kernel(const ElemParams p) {
  const int64_t groups = p.N * p.K / 8;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x - lane;
       base < groups; base += stride) {
    const int64_t gid = base + lane;
    const bool active = gid < groups;
    switch (p.sc.kind) {
      case kAdamW: opt_group<kAdamW, WDT, SDT>(gid, active, p); break;
      case kNAdam: opt_group<kNAdam, WDT, SDT>(gid, active, p); break;
      case kRAdam: opt_group<kRAdam, WDT, SDT>(gid, active, p); break;
      case kLion: opt_group<kLion, WDT, SDT>(gid, active, p); break;
      case kRMSprop: opt_group<kRMSprop, WDT, SDT>(gid, active, p); break;
      case kAdaGrad: opt_group<kAdaGrad, WDT, SDT>(gid, active, p); break;
      case kSGD: opt_group<kSGD, WDT, SDT>(gid, active, p); break;
      default: opt_group<kSGDMomentum, WDT, SDT>(gid, active, p); break;
    }
  }
}

template <bool SIGNED>
__global__ void __launch_bounds__(kElemThreads) quantize_kernel(const ElemParams p) {
  const int64_t groups = p.N * p.K / 8;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x - lane;
       base < groups; base += stride) {
    const int64_t gid = base + lane;
    const bool active = gid < groups;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
    if (active) load8(p.dW + gid * 8, v);
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) a = dev::absmax_acc(a, v[j]);
    a = group_max(a, p.qblock / 8);
    if (active) {
      store_codes8<SIGNED>(p.s1, gid * 8, a, v);
      if ((gid & (p.qblock / 8 - 1)) == 0) p.s1_scale[gid * 8 / p.qblock] = a;
    }
  }
}

template <bool SIGNED>
__global__ void __launch_bounds__(kElemThreads) dequantize_kernel(const ElemParams p) {
  const int64_t groups = p.N * p.K / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gid < groups;
       gid += stride) {
    float v[8];
    load_codes8<SIGNED>(p.s1, gid * 8, p.s1_scale[gid * 8 / p.qblock], v);
    store8(static_cast<float*>(p.W) + gid * 8, v);
  }
}

// 16-byte asynchronous copy global -> shared (cp.async, L1 bypassed); with
// `valid` false the destination is zero-filled and nothing is read.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// W rounded to its nearest bf16 (ties to even) and widened back, with integer
// operations: the same value as __float2bfloat16_rn for every finite and
// infinite W (a NaN stays a NaN).
__device__ __forceinline__ float round_to_bf16(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return __uint_as_float(u | 0x00400000u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return __uint_as_float(u & 0xFFFF0000u);
}

// dX[t, k] = sum_n dY[t, n] * bf16(W[n, k]) with fp32 accumulation.  A block
// of 256 threads owns a TM x TK output tile; SPLIT groups of threads share
// it, group g taking n = 32 s + g (32 / SPLIT) ... of each 32-n slice s (the
// groups' sums are added at the end, in group order); a thread keeps 4 x 4
// outputs (rows ty + (TM / 4) i, columns 4 tx + j).  Slices stream through a
// 3-deep ring in shared memory filled with asynchronous copies, so two slices
// are in flight while the block multiplies the third.  Each slice's weights
// are rounded to bf16 once, in place, when it lands (not once per use).
// Within a group each output sums its products in ascending n (one fused
// multiply-add each).  64 x 64 tiles for grids that fill the GPU; 32 x 32
// tiles split four ways give small layers four times as many blocks.
//
// The block lets a dependent grid launch at once (programmatic dependent
// launch): the FORGE step that follows on the stream starts its main loop
// while dX runs, and waits for this grid before its first weight write.
constexpr int kDgStages = 3;
template <int TM, int TK, int SPLIT>
__global__ void __launch_bounds__(256) dgrad_fp32w_kernel(const __nv_bfloat16* __restrict__ dY,
                                                          const float* __restrict__ W,
                                                          __nv_bfloat16* __restrict__ dX,
                                                          int64_t T, int64_t N, int64_t K) {
  constexpr int kGroup = (TM / 4) * (TK / 4);  // threads per group
  constexpr int kNPer = 32 / SPLIT;            // n per group and slice
  static_assert(kGroup * SPLIT == 256, "256 threads per block");
  static_assert((SPLIT - 1) * TM * TK <= kDgStages * 32 * TK, "the partial sums reuse the weight ring");
  __shared__ __align__(16) uint16_t sA[kDgStages][TM][40];  // [stage][t][n]: dY bits, 80-byte rows
  __shared__ __align__(16) float sB[kDgStages][32][TK];     // [stage][n][k]: W
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = static_cast<int>(threadIdx.x);
  const int grp = tid / kGroup, lt = tid % kGroup;
  const int tx = lt % (TK / 4), ty = lt / (TK / 4);
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * TM, k0 = static_cast<int64_t>(blockIdx.x) * TK;
  const int64_t slices = (N + 31) / 32;
  // slice `sl` into stage `st`: dY rows of 32 n (four 16-byte pieces each),
  // W rows of TK k (TK / 4 pieces each); N and K are multiples of 8, so a
  // piece is wholly inside or wholly outside the matrix
  auto load = [&](int64_t sl, int st) {
    if (sl < slices) {
      const int64_t n0 = sl * 32;
      for (int c = tid; c < TM * 4; c += 256) {
        const int row = c >> 2, ch = c & 3;
        const int64_t t = t0 + row, n = n0 + ch * 8;
        const bool ok = t < T && n < N;
        cp_async16(&sA[st][row][ch * 8], ok ? static_cast<const void*>(dY + t * N + n) : dY, ok);
      }
#pragma unroll
      for (int c = tid; c < 8 * TK; c += 256) {
        const int nr = c / (TK / 4), kc = c % (TK / 4);
        const int64_t n = n0 + nr, k = k0 + kc * 4;
        const bool ok = n < N && k < K;
        cp_async16(&sB[st][nr][kc * 4], ok ? static_cast<const void*>(W + n * K + k) : W, ok);
      }
    }
    cp_async_commit();  // an empty group past the last slice keeps the counting uniform
  };
  float acc[4][4] = {};
#pragma unroll
  for (int st = 0; st < kDgStages - 1; ++st) load(st, st);
  for (int64_t sl = 0; sl < slices; ++sl) {
    cp_async_wait<kDgStages - 2>();  // slice sl has landed (this thread's pieces)
    __syncthreads();                 // ... everyone's; and slice sl - 1 is no longer read
    const int st = static_cast<int>(sl % kDgStages);
#pragma unroll
    for (int e = tid; e < 32 * TK; e += 256) {  // the slice's 32 x TK weights, each once
      float& x = sB[st][e / TK][e % TK];
      x = round_to_bf16(x);
    }
    __syncthreads();
    load(sl + kDgStages - 1, static_cast<int>((sl + kDgStages - 1) % kDgStages));
#pragma unroll 4
    for (int q = 0; q < kNPer; ++q) {
      const int nn = grp * kNPer + q;
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        a[i] = __uint_as_float(static_cast<uint32_t>(sA[st][ty + (TM / 4) * i][nn]) << 16);
      const float4 wv = *reinterpret_cast<const float4*>(&sB[st][nn][tx * 4]);
      w[0] = wv.x;
      w[1] = wv.y;
      w[2] = wv.z;
      w[3] = wv.w;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(a[i], w[j], acc[i][j]);
    }
  }
  cp_async_wait<0>();
  if constexpr (SPLIT > 1) {  // groups 1.. hand their sums to group 0 through the weight ring
    __syncthreads();          // every thread is done with the ring
    float* part = &sB[0][0][0];
    if (grp > 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          part[((grp - 1) * TM + ty + (TM / 4) * i) * TK + tx * 4 + j] = acc[i][j];
    }
    __syncthreads();
    if (grp > 0) return;
#pragma unroll
    for (int g = 1; g < SPLIT; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += part[((g - 1) * TM + ty + (TM / 4) * i) * TK + tx * 4 + j];
  }
  const int64_t k = k0 + tx * 4;
  if (k >= K) return;  // K % 8 == 0: columns k .. k + 3 are all inside or all outside
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + ty + (TM / 4) * i;
    if (t >= T) continue;
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[i][0]))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[i][1]))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[i][2]))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[i][3]))) << 16);
    *reinterpret_cast<uint2*>(dX + t * K + k) = make_uint2(lo, hi);
  }
}

int elem_grid(int64_t groups, int num_sms) {
  const int64_t want = (groups + kElemThreads - 1) / kElemThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_opt_step(int wdt, int sdt, const ElemParams& p, int num_sms, cudaStream_t s) {
  const int grid = elem_grid(p.N * p.K / 8, num_sms);
  if (wdt == kWBf16) {
    if (sdt == kSInt8) opt_step_kernel<kWBf16, kSInt8><<<grid, kElemThreads, 0, s>>>(p);
    else if (sdt == kSBf16) opt_step_kernel<kWBf16, kSBf16><<<grid, kElemThreads, 0, s>>>(p);
    else opt_step_kernel<kWBf16, kSFp32><<<grid, kElemThreads, 0, s>>>(p);
  } else {
    if (sdt == kSInt8) opt_step_kernel<kWFp32, kSInt8><<<grid, kElemThreads, 0, s>>>(p);
    else if (sdt == kSBf16) opt_step_kernel<kWFp32, kSBf16><<<grid, kElemThreads, 0, s>>>(p);
    else opt_step_kernel<kWFp32, kSFp32><<<grid, kElemThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize(const ElemParams& p, int num_sms, cudaStream_t s) {
  const int grid = elem_grid(p.N * p.K / 8, num_sms);
  if (p.is_signed) quantize_kernel<true><<<grid, kElemThreads, 0, s>>>(p);
  else quantize_kernel<false><<<grid, kElemThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const ElemParams& p, int num_sms, cudaStream_t s) {
  const int grid = elem_grid(p.N * p.K / 8, num_sms);
  if (p.is_signed) dequantize_kernel<true><<<grid, kElemThreads, 0, s>>>(p);
  else dequantize_kernel<false><<<grid, kElemThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dgrad_fp32w(const void* dY, const float* W, void* dX, int64_t T, int64_t N,
                               int64_t K, int num_sms, cudaStream_t s) {
  const auto* y = static_cast<const __nv_bfloat16*>(dY);
  auto* x = static_cast<__nv_bfloat16*>(dX);
  if (((K + 63) / 64) * ((T + 63) / 64) >= num_sms) {
    const dim3 grid(static_cast<unsigned>((K + 63) / 64), static_cast<unsigned>((T + 63) / 64));
    dgrad_fp32w_kernel<64, 64, 1><<<grid, 256, 0, s>>>(y, W, x, T, N, K);
  } else {
    const dim3 grid(static_cast<unsigned>((K + 31) / 32), static_cast<unsigned>((T + 31) / 32));
    dgrad_fp32w_kernel<32, 32, 4><<<grid, 256, 0, s>>>(y, W, x, T, N, K);
  }
  return cudaGetLastError();
}

}  // namespace forge
