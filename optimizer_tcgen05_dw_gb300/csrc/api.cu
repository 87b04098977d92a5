// The C ABI of libforge (declared in include/forge.h): argument checks,
// per-step optimizer scalars, TMA tensor maps, and kernel launches.
//
// Nothing here allocates device memory: every buffer is the caller's.  The
// library's only device state is one status word per device and the
// one-launch step's dX-completion counters (below), both static.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "forge.h"
#include "common.h"
#include "launch.h"

namespace forge {

// Device-side status word: 0 = OK, otherwise the first error a kernel saw.
__device__ uint32_t g_device_status;

// Per column block of W, the dX tiles of the current one-launch step whose
// MMAs have finished; cleared on the stream before each such launch.  Steps
// launched concurrently on different streams of one device would share
// them, so the one-launch path is taken only while the caller keeps its
// steps on one device ordered (forge.h, forge_set_step_fusion).
__device__ uint32_t g_dx_done[kMaxDxBlocks + 2];  // + the residency gate's two words

// Scratch of forge_linear_bwd_step_static alone: that entry point's own
// dX-completion counters for the one-launch step, one word per 256-column
// block of W (1024 words: K up to 262144), and the residency gate's two words.
// Static device memory, so the entry point never allocates; cleared on the
// caller's stream before each launch that uses it.
constexpr int kStaticScratchWords = 1024;
static __device__ __align__(256) uint32_t g_static_scratch[kStaticScratchWords + 2];

namespace {

thread_local char g_msg[512] = "";

forge_status_t fail(forge_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

forge_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(FORGE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int32_t> g_skip_loads{0};
std::atomic<int32_t> g_step_fusion{1};

// ---------------------------------------------------------------- per device

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int num_sms = 0;
  uint32_t* status = nullptr;
  uint32_t* dx_done = nullptr;
  uint32_t* static_scratch = nullptr;  // g_static_scratch on this device
  int step_pairs[kNumKernelSdt] = {};  // resident one-launch-step pairs, by kernel state dtype
  int cc_major = 0, cc_minor = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

forge_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FORGE_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_ready[dev]) {
    DeviceInfo d;
    if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    void* sym = nullptr;
    if ((e = cudaGetSymbolAddress(&sym, g_device_status)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    d.status = static_cast<uint32_t*>(sym);
    if ((e = cudaGetSymbolAddress(&sym, g_dx_done)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(dX counters)");
    d.dx_done = static_cast<uint32_t*>(sym);
    if ((e = cudaGetSymbolAddress(&sym, g_static_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    d.static_scratch = static_cast<uint32_t*>(sym);
    if (d.cc_major == 10 && d.cc_minor == 3) {
      d.step_pairs[kSFp32] = step_max_pairs(kSFp32);
      d.step_pairs[kSInt8] = step_max_pairs(kSInt8);
      d.step_pairs[kSBf16] = step_max_pairs(kSBf16);
      d.step_pairs[kSInt8W] = step_max_pairs(kSInt8W);
      d.step_pairs[kSInt8X] = step_max_pairs(kSInt8X);
      d.step_pairs[kSInt8WX] = step_max_pairs(kSInt8WX);
    }
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  *out = g_dev[dev];
  return FORGE_OK;
}

// ---------------------------------------------------------------- tensor maps

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

forge_status_t encode_fn(EncodeFn* fn) {
  static std::once_flag once;
  static EncodeFn cached = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeFn>(p);
  });
  if (cached == nullptr) {
    return err != cudaSuccess ? cuda_fail(err, "cuTensorMapEncodeTiled lookup")
                              : fail(FORGE_ERR_CUDA, "cuTensorMapEncodeTiled not available");
  }
  *fn = cached;
  return FORGE_OK;
}

// A 2-D row-major tensor [outer x inner] of `esize`-byte elements, read and
// written in boxes of box_outer rows x box_inner elements with the given
// shared-memory swizzle; out-of-range elements read as 0 and are not written.
forge_status_t tensor_map(CUtensorMap* m, const void* base, CUtensorMapDataType dtype, int esize,
                          int64_t inner, int64_t outer, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle) {
  EncodeFn fn;
  forge_status_t st = encode_fn(&fn);
  if (st != FORGE_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * static_cast<cuuint64_t>(esize)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FORGE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld]", static_cast<int>(r),
                static_cast<long long>(outer), static_cast<long long>(inner));
  return FORGE_OK;
}

// An MN-major GEMM operand stored [rows x cols] (bf16, cols % 64 == 0) seen as
// a 3-D tensor (64 columns, rows, cols/64 column blocks), so one box of
// {64, box_rows, blocks} lands in shared memory as `blocks` consecutive
// 128-byte-swizzled atoms of box_rows x 64: a whole stage operand per copy.
forge_status_t mn_major_3d_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows,
                               uint32_t box_rows, uint32_t blocks) {
  EncodeFn fn;
  forge_status_t st = encode_fn(&fn);
  if (st != FORGE_OK) return st;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, blocks};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FORGE_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d) for [%lld x %lld]",
                static_cast<int>(r), static_cast<long long>(rows), static_cast<long long>(cols));
  return FORGE_OK;
}

// The weight-gradient operands dY [T x N] (A, 128 columns per tile) and
// X [T x K] (B, 256 columns per tile): 3-D single-copy maps when N and K are
// multiples of 64, else 2-D maps of one 64-column block per copy.
forge_status_t wgrad_maps(const forge_linear_t* lin, int bk, CUtensorMap* ma, CUtensorMap* mb,
                          int32_t* op3d);

// GEMM operands: bf16, 64-element (128-byte) rows, 128-byte swizzle.
forge_status_t bf16_map(CUtensorMap* m, const void* base, int64_t inner, int64_t outer,
                        uint32_t box_inner, uint32_t box_outer) {
  return tensor_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, box_inner, box_outer,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

forge_status_t wgrad_maps(const forge_linear_t* lin, int bk, CUtensorMap* ma, CUtensorMap* mb,
                          int32_t* op3d) {
  forge_status_t st;
  if (lin->N % 64 == 0 && lin->K % 64 == 0) {
    *op3d = 1;
    if ((st = mn_major_3d_map(ma, lin->dY, lin->N, lin->T, bk, kTileM / 64)) != FORGE_OK) return st;
    return mn_major_3d_map(mb, lin->X, lin->K, lin->T, bk, kTileN / 2 / 64);  // half of B per CTA
  }
  *op3d = 0;
  if ((st = bf16_map(ma, lin->dY, lin->N, lin->T, 64, bk)) != FORGE_OK) return st;
  return bf16_map(mb, lin->X, lin->K, lin->T, 64, bk);
}

// INT8 states: the absmax block width of a state dtype (0 if not INT8).
int qblock_of(int32_t s_dtype) {
  switch (s_dtype) {
    case FORGE_STATE_INT8_B32: return 32;
    case FORGE_STATE_INT8_B64: return 64;
    case FORGE_STATE_INT8_B128: return 128;
    case FORGE_STATE_INT8_B256: return 256;
    default: return 0;
  }
}

// The kernels' state dtype (every INT8 block width is kSInt8; the block width
// travels in the parameters).
int base_sdt(int32_t s_dtype) { return qblock_of(s_dtype) != 0 ? kSInt8 : s_dtype; }

// Maps of the state tiles the bf16-weight epilogue stages through shared
// memory: fp32 states in 32-column boxes (128-byte rows, 128-byte swizzle),
// INT8 codes in 64-column boxes and bf16 states in 32-column boxes (64-byte
// rows, 64-byte swizzle); 128 rows each.  A rule that keeps no such state gets a copy of `other` (unused).
forge_status_t state_maps(const forge_state_t* st, int kind, int64_t N, int64_t K,
                          const CUtensorMap& other, CUtensorMap* m1, CUtensorMap* m2) {
  *m1 = other;
  *m2 = other;
  const bool int8 = qblock_of(st->s_dtype) != 0;
  const void* bufs[2] = {st->s1, st->s2};
  const bool used[2] = {uses_s1(kind), uses_s2(kind)};
  CUtensorMap* maps[2] = {m1, m2};
  for (int i = 0; i < 2; ++i) {
    if (!used[i]) continue;
    forge_status_t r =
        int8 ? tensor_map(maps[i], bufs[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, N, 64, kTileM,
                          CU_TENSOR_MAP_SWIZZLE_64B)
        : st->s_dtype == FORGE_STATE_BF16
             ? tensor_map(maps[i], bufs[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, 32, kTileM,
                          CU_TENSOR_MAP_SWIZZLE_64B)
             : tensor_map(maps[i], bufs[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, K, N, 32, kTileM,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != FORGE_OK) return r;
  }
  return FORGE_OK;
}

// The state dtype the tensor-core kernel is instantiated for: INT8 states
// over a short reduction (T <= kStageWeightsMaxT) with bf16 weights take the
// epilogue that stages the weights too; INT8 blocks other than 64 the
// variants that read the block width from the parameters.
int kernel_sdt(const forge_state_t* st, int64_t T) {
  const int qb = qblock_of(st->s_dtype);
  if (qb != 0 && st->w_dtype == FORGE_W_BF16_SR) {
    const bool staged = T <= kStageWeightsMaxT;
    if (qb == 64) return staged ? kSInt8W : kSInt8;
    return staged ? kSInt8WX : kSInt8X;
  }
  return base_sdt(st->s_dtype);
}

// log2 of an INT8 block width (0 when not INT8).
int qshift_of(int32_t s_dtype) {
  const int qb = qblock_of(s_dtype);
  int sh = 0;
  while (qb > 0 && (1 << sh) < qb) ++sh;
  return sh;
}

// The bf16 weights in 64-column x 128-row boxes (128-byte swizzle), for the
// kSInt8W epilogue.  Otherwise a copy of `other` (unused).
forge_status_t weight_map(const forge_state_t* st, int sdt, int64_t N, int64_t K, const CUtensorMap& other,
                          CUtensorMap* mw) {
  *mw = other;
  if (sdt == kSInt8W || sdt == kSInt8WX) return bf16_map(mw, st->W, K, N, 64, kTileM);
  return FORGE_OK;
}

// Philox4x32-10 round keys of `seed`: the key, bumped by the Weyl constants
// before each round after the first.
void philox_round_keys(uint64_t seed, uint32_t* rk) {
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    rk[2 * r] = k0;
    rk[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// ---------------------------------------------------------------- scalars

// Per-step scalars of each rule, in double from the float hyper-parameters,
// rounded once to float (the formulas of the published methods; see optim.cuh
// for the per-element order).
OptScalars make_scalars(int kind, const forge_hparams_t& hp, int64_t step) {
  OptScalars s;
  std::memset(&s, 0, sizeof(s));
  s.kind = kind;
  const double lr = hp.lr, b1 = hp.beta1, b2 = hp.beta2, eps = hp.eps, wd = hp.weight_decay;
  const double t = static_cast<double>(step);
  s.l2 = static_cast<float>(wd);
  s.lr = static_cast<float>(lr);
  s.eps = static_cast<float>(eps);
  s.b1 = static_cast<float>(b1);
  s.b2 = static_cast<float>(b2);
  s.omb1 = static_cast<float>(1.0 - b1);
  s.omb2 = static_cast<float>(1.0 - b2);
  switch (kind) {
    case kAdamW: {
      const double c1 = 1.0 - std::pow(b1, t), c2 = 1.0 - std::pow(b2, t);
      s.decay = static_cast<float>(1.0 - lr * wd);
      s.step_size = static_cast<float>(lr / c1);
      s.inv_sqrt_c2 = static_cast<float>(1.0 / std::sqrt(c2));
      break;
    }
    case kNAdam: {
      // mu_i = b1 (1 - 0.5 * 0.96^(0.004 i)); product of mu_1..mu_t
      const double c2 = 1.0 - std::pow(b2, t);
      auto mu = [&](int64_t i) { return b1 * (1.0 - 0.5 * std::pow(0.96, static_cast<double>(i) * 0.004)); };
      double prod = 1.0;
      for (int64_t i = 1; i <= step; ++i) prod *= mu(i);
      const double mu_t = mu(step), mu_next = mu(step + 1);
      const double prod_next = prod * mu_next;
      s.inv_c2 = static_cast<float>(1.0 / c2);
      s.coef_g = static_cast<float>(lr * (1.0 - mu_t) / (1.0 - prod));
      s.coef_m = static_cast<float>(lr * mu_next / (1.0 - prod_next));
      break;
    }
    case kRAdam: {
      const double c1 = 1.0 - std::pow(b1, t), c2 = 1.0 - std::pow(b2, t);
      const double rho_inf = 2.0 / (1.0 - b2) - 1.0;
      const double rho_t = rho_inf - 2.0 * t * std::pow(b2, t) / c2;
      s.sqrt_c2 = static_cast<float>(std::sqrt(c2));
      if (rho_t > 5.0) {
        const double r = std::sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf /
                                   ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t));
        s.rectified = 1;
        s.step_size = static_cast<float>(lr * r / c1);
      } else {
        s.rectified = 0;
        s.step_size = static_cast<float>(lr / c1);
      }
      break;
    }
    case kLion:
      s.decay = static_cast<float>(1.0 - lr * wd);
      break;
    case kRMSprop:
      s.alpha = hp.alpha;
      s.oma = static_cast<float>(1.0 - static_cast<double>(hp.alpha));
      break;
    case kSGDMomentum:
      s.mom = hp.momentum;
      break;
    default:
      break;
  }
  return s;
}

// ---------------------------------------------------------------- checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

forge_status_t check_state(const forge_state_t* st, int kind, int64_t N, int64_t K) {
  if (st == nullptr) return fail(FORGE_ERR_INVALID_ARG, "state is NULL");
  if (st->w_dtype != FORGE_W_FP32 && st->w_dtype != FORGE_W_BF16_SR)
    return fail(FORGE_ERR_INVALID_ARG, "w_dtype %d", st->w_dtype);
  if (st->s_dtype != FORGE_STATE_FP32 && st->s_dtype != FORGE_STATE_BF16 && qblock_of(st->s_dtype) == 0)
    return fail(FORGE_ERR_INVALID_ARG, "s_dtype %d", st->s_dtype);
  if (N * K > 0 && (st->W == nullptr || !aligned16(st->W)))
    return fail(FORGE_ERR_INVALID_ARG, "W must be a non-NULL 16-byte aligned device pointer");
  const int qb = qblock_of(st->s_dtype);
  const bool int8 = qb != 0;
  if (int8 && K % qb != 0)
    return fail(FORGE_ERR_INVALID_ARG, "INT8 states in blocks of %d need K %% %d == 0 (K=%lld)", qb, qb,
                (long long)K);
  if (int8 && K % 64 != 0)
    return fail(FORGE_ERR_INVALID_ARG, "INT8 states need K %% 64 == 0 (K=%lld)", (long long)K);
  if (N * K == 0) return FORGE_OK;
  if (uses_s1(kind)) {
    if (st->s1 == nullptr || !aligned16(st->s1))
      return fail(FORGE_ERR_INVALID_ARG, "rule %d needs s1 (16-byte aligned)", kind);
    if (int8 && st->s1_scale == nullptr) return fail(FORGE_ERR_INVALID_ARG, "INT8 s1 needs s1_scale");
  }
  if (uses_s2(kind)) {
    if (st->s2 == nullptr || !aligned16(st->s2))
      return fail(FORGE_ERR_INVALID_ARG, "rule %d needs s2 (16-byte aligned)", kind);
    if (int8 && st->s2_scale == nullptr) return fail(FORGE_ERR_INVALID_ARG, "INT8 s2 needs s2_scale");
  }
  return FORGE_OK;
}

forge_status_t check_linear(const forge_linear_t* lin, bool need_x) {
  if (lin == nullptr) return fail(FORGE_ERR_INVALID_ARG, "lin is NULL");
  if (lin->T < 0 || lin->N < 0 || lin->K < 0)
    return fail(FORGE_ERR_INVALID_ARG, "negative shape T=%lld N=%lld K=%lld", (long long)lin->T,
                (long long)lin->N, (long long)lin->K);
  if (lin->N % 8 != 0 || lin->K % 8 != 0)
    return fail(FORGE_ERR_INVALID_ARG, "N and K must be multiples of 8 (N=%lld K=%lld)",
                (long long)lin->N, (long long)lin->K);
  if (lin->T > (int64_t{1} << 31) - 1 || lin->N > (int64_t{1} << 31) - 1 || lin->K > (int64_t{1} << 31) - 1)
    return fail(FORGE_ERR_UNSUPPORTED, "dimensions must fit in 31 bits");
  if (lin->T > 0 && lin->N > 0) {
    if (lin->dY == nullptr || !aligned16(lin->dY)) return fail(FORGE_ERR_INVALID_ARG, "dY must be 16-byte aligned");
    if (need_x && lin->K > 0 && (lin->X == nullptr || !aligned16(lin->X)))
      return fail(FORGE_ERR_INVALID_ARG, "X must be 16-byte aligned");
  }
  if (lin->dX != nullptr && !aligned16(lin->dX)) return fail(FORGE_ERR_INVALID_ARG, "dX must be 16-byte aligned");
  return FORGE_OK;
}

forge_status_t check_hp(int32_t kind, const forge_hparams_t* hp, int64_t step) {
  if (kind < FORGE_ADAMW || kind > FORGE_SGD_MOMENTUM) return fail(FORGE_ERR_INVALID_ARG, "opt_kind %d", kind);
  if (hp == nullptr) return fail(FORGE_ERR_INVALID_ARG, "hparams is NULL");
  if (step < 1) return fail(FORGE_ERR_INVALID_ARG, "step must be >= 1 (got %lld)", (long long)step);
  return FORGE_OK;
}

void fill_tiles(GemmParams& p, int64_t M, int64_t Ncols, int64_t red, int bk = kBlockK) {
  p.M = static_cast<int32_t>(M);
  p.Ncols = static_cast<int32_t>(Ncols);
  p.num_kb = static_cast<int32_t>((red + bk - 1) / bk);
  p.tiles_m = static_cast<int32_t>((M + 2 * kTileM - 1) / (2 * kTileM));  // 256-row pair tiles
  p.tiles_n = static_cast<int32_t>((Ncols + kTileN - 1) / kTileN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.num_units = p.num_tiles;
  p.split_from = p.num_tiles;
}

// A last partial wave of pair tiles (R = num_tiles % pairs of them) runs as
// 2R column halves when they fit one wave, so that it takes half as long; a
// layer of at most pairs / 2 tiles (wider than 128 columns) runs every tile as
// two halves on twice the pairs.  Either way a pair holds at most one half
// unit, its last.  Only for the staged epilogue without dX tiles.
void split_tail(GemmParams& p, int pairs) {
  const int F = p.num_tiles, R = F % pairs;
  if (F > pairs && R > 0 && 2 * R <= pairs) {
    p.split_from = F - R;
    p.num_units = F + R;
  } else if (F > 0 && 2 * F <= pairs && p.Ncols > kTileN / 2) {
    p.split_from = 0;
    p.num_units = 2 * F;
  }
}

// Clusters of two CTAs, at most one CTA per SM, at most one pair per unit.
int grid_for(const GemmParams& p, const DeviceInfo& d) {
  const int pairs = d.num_sms / 2;
  return 2 * (p.num_units < pairs ? p.num_units : pairs);
}

forge_status_t launch_dgrad(const forge_linear_t* lin, const void* W, int32_t w_dtype, cudaStream_t s,
                            const DeviceInfo& d) {
  const int64_t T = lin->T, N = lin->N, K = lin->K;
  if (T == 0 || K == 0) return FORGE_OK;
  cudaError_t e;
  if (N == 0) {  // empty reduction: dX = 0
    if ((e = cudaMemsetAsync(lin->dX, 0, static_cast<size_t>(T * K * 2), s)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync(dX)");
    return FORGE_OK;
  }
  if (w_dtype == FORGE_W_FP32) {
    if ((e = launch_dgrad_fp32w(lin->dY, static_cast<const float*>(W), lin->dX, T, N, K, d.num_sms, s)) !=
        cudaSuccess)
      return cuda_fail(e, "dX (fp32 weights) launch");
    return FORGE_OK;
  }
  CUtensorMap ma, mb;
  forge_status_t st;
  if ((st = bf16_map(&ma, lin->dY, N, T, 64, kTileM)) != FORGE_OK) return st;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if (K % 64 == 0) {
    p.op3d = 1;
    if ((st = mn_major_3d_map(&mb, W, K, N, kBlockK, kTileN / 2 / 64)) != FORGE_OK) return st;
  } else if ((st = bf16_map(&mb, W, K, N, 64, kBlockK)) != FORGE_OK) {
    return st;
  }
  fill_tiles(p, T, K, N);
  p.out = lin->dX;
  p.status = d.status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.skip_loads = g_skip_loads.load();
  if ((e = launch_tc_plain(kModeDgrad, ma, mb, p, grid_for(p, d), s)) != cudaSuccess)
    return cuda_fail(e, "dX launch");
  return FORGE_OK;
}

// Deal the one-launch step's dX tiles over `pairs` so that the largest
// per-pair work (dX tiles plus dW tiles) is smallest.  dW tiles go
// round-robin: the first num_tiles % pairs pairs get one more ("heavy").  A
// dW tile costs about c = 1.1 T / N dX tiles (reductions over T and N, plus
// its optimizer epilogue).  The kernel deals dx_rounds rounds to every pair
// and the rest round-robin to the pairs from dx_heavy on.  Candidates: all
// full rounds with the few left-over tiles on the last pairs (away from the
// heavy ones), or fewer rounds with the rest on the light pairs; the
// smallest modelled maximum wins.
void balance_dx(GemmParams& p, int pairs, int64_t T, int64_t N) {
  const int D = p.dx_tiles, F = p.num_tiles;
  const int heavy = F % pairs, fl = F / pairs;
  const double c = 1.1 * static_cast<double>(T) / static_cast<double>(N);
  const int full = D / pairs, ex = D % pairs;
  // full rounds; the ex left-over tiles on pairs pairs-ex .. pairs-1
  double best = full + fl * c;
  if (ex > 0) best = std::max(best, full + 1 + fl * c);
  if (heavy > 0) best = std::max(best, full + (fl + 1) * c);
  if (ex > 0 && heavy > pairs - ex) best = std::max(best, full + 1 + (fl + 1) * c);
  p.dx_rounds = full;
  p.dx_heavy = pairs - ex;
  if (heavy == 0) return;
  const int nl = pairs - heavy;
  for (int r = full; r >= 0; --r) {  // r rounds, the rest on the light pairs
    const int rem = D - r * pairs;
    const double load = std::max(r + (rem + nl - 1) / nl + fl * c, r + (fl + 1) * c);
    if (load + 1e-9 < best) {
      best = load;
      p.dx_rounds = r;
      p.dx_heavy = heavy;
    }
  }
}

// dX and the FORGE step in one persistent launch (bf16 weights; N and K
// multiples of 64; T > 0): dX tiles over (T, K) reducing over N, then dW
// tiles over (N, K) reducing over T.
forge_status_t launch_step(const forge_linear_t* lin, const forge_state_t* state, int32_t opt_kind,
                           const OptScalars& sc, int64_t step, uint64_t seed, uint64_t sr_base,
                           cudaStream_t s, const DeviceInfo& d, uint32_t* counters = nullptr) {
  const int64_t T = lin->T, N = lin->N, K = lin->K;
  forge_status_t st;
  CUtensorMap ma, mb, mda, mdb, m1, m2, mdx, mw;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = wgrad_maps(lin, kFusedBlockK, &ma, &mb, &p.op3d)) != FORGE_OK) return st;
  if ((st = bf16_map(&mda, lin->dY, N, T, 64, kTileM)) != FORGE_OK) return st;
  if ((st = mn_major_3d_map(&mdb, state->W, K, N, kFusedBlockK, kTileN / 2 / 64)) != FORGE_OK) return st;
  if ((st = state_maps(state, opt_kind, N, K, ma, &m1, &m2)) != FORGE_OK) return st;
  if ((st = bf16_map(&mdx, lin->dX, K, T, 64, kTileM)) != FORGE_OK) return st;
  const int sdt = kernel_sdt(state, T);
  if ((st = weight_map(state, sdt, N, K, ma, &mw)) != FORGE_OK) return st;
  fill_tiles(p, N, K, T, kFusedBlockK);
  p.W = state->W; p.s1 = state->s1; p.s2 = state->s2;
  p.s1_scale = state->s1_scale; p.s2_scale = state->s2_scale;
  p.sc = sc;
  p.qblock = qblock_of(state->s_dtype);
  p.qshift = qshift_of(state->s_dtype);
  p.seed = seed;
  philox_round_keys(seed, p.round_keys);
  p.step = static_cast<uint64_t>(step);
  p.sr_base = sr_base;
  p.status = d.status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.skip_loads = g_skip_loads.load();
  p.dx_rows = static_cast<int32_t>(T);
  p.dx_tiles_m = static_cast<int32_t>((T + 2 * kTileM - 1) / (2 * kTileM));
  p.dx_tiles = p.dx_tiles_m * p.tiles_n;
  p.dx_num_kb = static_cast<int32_t>((N + kFusedBlockK - 1) / kFusedBlockK);
  p.dx_done = counters != nullptr ? counters : d.dx_done;
  p.dx_target = static_cast<uint32_t>(2 * p.dx_tiles_m);
  cudaError_t e;
  // the per-column-block counters and the residency gate's two words
  if ((e = cudaMemsetAsync(p.dx_done, 0, static_cast<size_t>(p.tiles_n + 2) * sizeof(uint32_t), s)) != cudaSuccess)
    return cuda_fail(e, "clearing the dX counters");
  // Every pair must be resident at once (dW tiles wait for other pairs' dX
  // tiles): at most the occupancy limit, at most one pair per tile.
  const int pairs = std::min(std::min(d.num_sms / 2, d.step_pairs[sdt]), p.num_tiles + p.dx_tiles);
  balance_dx(p, pairs, T, N);
  if ((e = launch_tc_step(sdt, ma, mb, mda, mdb, m1, m2, mdx, mw, p, 2 * pairs, s)) !=
      cudaSuccess)
    return cuda_fail(e, "one-launch step");
  return FORGE_OK;
}

forge_status_t check_device(const DeviceInfo& d) {
  if (d.cc_major != 10 || d.cc_minor != 3)
    return fail(FORGE_ERR_UNSUPPORTED, "libforge is built for sm_103a; device is sm_%d%d", d.cc_major, d.cc_minor);
  return FORGE_OK;
}

// forge_linear_bwd_step on rows [row_offset, row_offset + N) of a matrix with
// K columns: the stochastic-rounding counter takes the element's index in the
// whole matrix, (row_offset + n) * K + k.
forge_status_t bwd_step(const forge_linear_t* lin, const forge_state_t* state, int32_t opt_kind,
                        const forge_hparams_t* hp, int64_t step, uint64_t seed, int64_t row_offset,
                        void* stream) {
  forge_status_t st;
  if ((st = check_linear(lin, true)) != FORGE_OK) return st;
  if ((st = check_hp(opt_kind, hp, step)) != FORGE_OK) return st;
  if ((st = check_state(state, opt_kind, lin->N, lin->K)) != FORGE_OK) return st;
  if (lin->N == 0 || lin->K == 0) return FORGE_OK;
  if (state->s_dtype == FORGE_STATE_BF16 && state->w_dtype == FORGE_W_FP32 && lin->T > 0)
    return fail(FORGE_ERR_UNSUPPORTED, "bf16 moments need bf16 weights in the fused step");
  if (state->w_dtype == FORGE_W_FP32 && lin->T > 0 && qblock_of(state->s_dtype) != 0 &&
      qblock_of(state->s_dtype) != 64)
    return fail(FORGE_ERR_UNSUPPORTED, "INT8 blocks other than 64 need bf16 weights in the fused step");
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  if ((st = check_device(d)) != FORGE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const OptScalars sc = make_scalars(opt_kind, *hp, step);
  const uint64_t sr_base = static_cast<uint64_t>(row_offset) * static_cast<uint64_t>(lin->K) / 8u;
  // One launch for dX and the FORGE step (bf16 weights, 64-aligned N and K):
  // the dX tiles first, each dW tile's update after the dX tiles that read its
  // weights.
  if (lin->dX != nullptr && lin->T > 0 && state->w_dtype == FORGE_W_BF16_SR && lin->N % 64 == 0 &&
      lin->K % 64 == 0 && (lin->K + kTileN - 1) / kTileN <= kMaxDxBlocks && g_step_fusion.load() &&
      d.step_pairs[kernel_sdt(state, lin->T)] > 0)
    return launch_step(lin, state, opt_kind, sc, step, seed, sr_base, s, d);
  // 1. dX from the pre-update weights, enqueued first on the same stream.
  if (lin->dX != nullptr && (st = launch_dgrad(lin, state->W, state->w_dtype, s, d)) != FORGE_OK) return st;
  cudaError_t e;
  if (lin->T == 0) {
    // No tokens: the gradient is exactly zero; apply the rule to it.
    ElemParams ep;
    std::memset(&ep, 0, sizeof(ep));
    ep.W = state->W; ep.s1 = state->s1; ep.s2 = state->s2;
    ep.s1_scale = state->s1_scale; ep.s2_scale = state->s2_scale;
    ep.N = lin->N; ep.K = lin->K; ep.sc = sc; ep.seed = seed; ep.step = static_cast<uint64_t>(step);
    ep.sr_base = sr_base;
    ep.qblock = qblock_of(state->s_dtype);
    if ((e = launch_opt_step(state->w_dtype, base_sdt(state->s_dtype), ep, d.num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "optimizer launch (T = 0)");
    return FORGE_OK;
  }
  // 2. the fused weight-gradient + optimizer pass.
  const int bk = state->w_dtype == FORGE_W_BF16_SR ? kFusedBlockK : kBlockK;
  CUtensorMap ma, mb;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = wgrad_maps(lin, bk, &ma, &mb, &p.op3d)) != FORGE_OK) return st;
  fill_tiles(p, lin->N, lin->K, lin->T, bk);
  p.W = state->W; p.s1 = state->s1; p.s2 = state->s2;
  p.s1_scale = state->s1_scale; p.s2_scale = state->s2_scale;
  p.sc = sc;
  p.qblock = qblock_of(state->s_dtype);
  p.qshift = qshift_of(state->s_dtype);
  p.seed = seed;
  philox_round_keys(seed, p.round_keys);
  p.step = static_cast<uint64_t>(step);
  p.sr_base = sr_base;
  p.status = d.status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.skip_loads = g_skip_loads.load();
  CUtensorMap m1 = ma, m2 = ma, mw = ma, mbh = mb;
  // the staged epilogue (states through shared memory by TMA): bf16 weights,
  // or fp32 weights with fp32 states
  if (state->w_dtype == FORGE_W_BF16_SR ||
      (state->w_dtype == FORGE_W_FP32 && state->s_dtype == FORGE_STATE_FP32)) {
    if ((st = state_maps(state, opt_kind, lin->N, lin->K, ma, &m1, &m2)) != FORGE_OK ||
        (st = weight_map(state, kernel_sdt(state, lin->T), lin->N, lin->K, ma, &mw)) != FORGE_OK)
      return st;
    if (p.qblock != 256) split_tail(p, d.num_sms / 2);  // a 256-column block spans both halves
    if (p.split_from < p.num_tiles && p.op3d &&  // half units load one 64-column block of X
        (st = mn_major_3d_map(&mbh, lin->X, lin->K, lin->T, bk, 1)) != FORGE_OK)
      return st;
  }
  // after the fp32-weight dX kernel the step may start at once: its epilogue
  // waits for dX (which reads the weights it overwrites) before any write
  const bool after_dx = lin->dX != nullptr && state->w_dtype == FORGE_W_FP32 && lin->N > 0;
  if ((e = launch_tc_fused(state->w_dtype, kernel_sdt(state, lin->T), ma, mb, mbh, m1, m2, mw, p,
                           grid_for(p, d), s, after_dx)) != cudaSuccess)
    return cuda_fail(e, "fused step launch");
  return FORGE_OK;
}

}  // namespace
}  // namespace forge

using namespace forge;

extern "C" {

forge_status_t forge_linear_bwd_step(const forge_linear_t* lin, const forge_state_t* state,
                                     int32_t opt_kind, const forge_hparams_t* hp, int64_t step,
                                     uint64_t seed, void* stream) {
  g_msg[0] = '\0';
  return bwd_step(lin, state, opt_kind, hp, step, seed, 0, stream);
}

forge_status_t forge_linear_bwd_step_shard(const forge_linear_t* lin, const forge_state_t* state,
                                           int32_t opt_kind, const forge_hparams_t* hp, int64_t step,
                                           uint64_t seed, int64_t row_offset, void* stream) {
  g_msg[0] = '\0';
  if (row_offset < 0) return fail(FORGE_ERR_INVALID_ARG, "row_offset must be >= 0 (got %lld)", (long long)row_offset);
  if (lin != nullptr && row_offset > (int64_t{1} << 31) - 1 - lin->N)
    return fail(FORGE_ERR_UNSUPPORTED, "row_offset + N must fit in 31 bits");
  return bwd_step(lin, state, opt_kind, hp, step, seed, row_offset, stream);
}

forge_status_t forge_linear_bwd_step_static(const forge_linear_t* lin, const forge_state_t* state,
                                            int32_t opt_kind, const forge_hparams_t* hp,
                                            int64_t step, uint64_t seed, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if ((st = check_linear(lin, true)) != FORGE_OK) return st;
  if ((st = check_hp(opt_kind, hp, step)) != FORGE_OK) return st;
  if ((st = check_state(state, opt_kind, lin->N, lin->K)) != FORGE_OK) return st;
  const bool one_launch = lin->dX != nullptr && lin->T > 0 && lin->N > 0 && lin->K > 0 &&
                          state->w_dtype == FORGE_W_BF16_SR && lin->N % 64 == 0 && lin->K % 64 == 0;
  if (!one_launch)  // no scratch needed: the regular entry point's two-launch form
    return forge_linear_bwd_step(lin, state, opt_kind, hp, step, seed, stream);
  const int64_t blocks = (lin->K + kTileN - 1) / kTileN;
  if (blocks > kStaticScratchWords)
    return fail(FORGE_ERR_UNSUPPORTED, "K = %lld needs %lld scratch counters; the static scratch holds %d",
                static_cast<long long>(lin->K), static_cast<long long>(blocks), kStaticScratchWords);
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  if ((st = check_device(d)) != FORGE_OK) return st;
  if (d.step_pairs[kernel_sdt(state, lin->T)] <= 0)  // the one launch cannot be resident: no scratch
    return forge_linear_bwd_step(lin, state, opt_kind, hp, step, seed, stream);  // two launches
  return launch_step(lin, state, opt_kind, make_scalars(opt_kind, *hp, step), step, seed, 0,
                     static_cast<cudaStream_t>(stream), d, d.static_scratch);
}

forge_status_t forge_linear_bwd_step_fp8(const forge_linear_fp8_t* lin, const forge_state_t* state,
                                         int32_t opt_kind, const forge_hparams_t* hp, int64_t step,
                                         uint64_t seed, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if (lin == nullptr) return fail(FORGE_ERR_INVALID_ARG, "lin is NULL");
  const int64_t T = lin->T, N = lin->N, K = lin->K;
  if (T < 0 || N < 0 || K < 0)
    return fail(FORGE_ERR_INVALID_ARG, "negative shape T=%lld N=%lld K=%lld", (long long)T, (long long)N,
                (long long)K);
  if (N % 8 != 0 || K % 8 != 0)
    return fail(FORGE_ERR_INVALID_ARG, "N and K must be multiples of 8 (N=%lld K=%lld)", (long long)N,
                (long long)K);
  if (T % 16 != 0) return fail(FORGE_ERR_INVALID_ARG, "FP8 operands need T %% 16 == 0 (T=%lld)", (long long)T);
  if (T > (int64_t{1} << 31) - 1 || N > (int64_t{1} << 31) - 1 || K > (int64_t{1} << 31) - 1)
    return fail(FORGE_ERR_UNSUPPORTED, "dimensions must fit in 31 bits");
  if (T > 0 && N > 0 && K > 0) {
    if (lin->Xt == nullptr || !aligned16(lin->Xt)) return fail(FORGE_ERR_INVALID_ARG, "Xt must be 16-byte aligned");
    if (lin->dYt == nullptr || !aligned16(lin->dYt)) return fail(FORGE_ERR_INVALID_ARG, "dYt must be 16-byte aligned");
  }
  const double c = static_cast<double>(lin->x_scale) * static_cast<double>(lin->dy_scale);
  if (!std::isfinite(lin->x_scale) || !std::isfinite(lin->dy_scale) || !std::isfinite(static_cast<float>(c)))
    return fail(FORGE_ERR_INVALID_ARG, "FP8 scales and their product must be finite floats");
  if ((st = check_hp(opt_kind, hp, step)) != FORGE_OK) return st;
  if ((st = check_state(state, opt_kind, N, K)) != FORGE_OK) return st;
  if (state->w_dtype != FORGE_W_BF16_SR)
    return fail(FORGE_ERR_UNSUPPORTED, "the FP8 step stages bf16 weights (w_dtype must be FORGE_W_BF16_SR)");
  if (N == 0 || K == 0) return FORGE_OK;
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  if ((st = check_device(d)) != FORGE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const OptScalars sc = make_scalars(opt_kind, *hp, step);
  cudaError_t e;
  if (T == 0) {  // no tokens: the rule on a zero gradient
    ElemParams ep;
    std::memset(&ep, 0, sizeof(ep));
    ep.W = state->W; ep.s1 = state->s1; ep.s2 = state->s2;
    ep.s1_scale = state->s1_scale; ep.s2_scale = state->s2_scale;
    ep.N = N; ep.K = K; ep.sc = sc; ep.seed = seed; ep.step = static_cast<uint64_t>(step);
    ep.qblock = qblock_of(state->s_dtype);
    if ((e = launch_opt_step(state->w_dtype, base_sdt(state->s_dtype), ep, d.num_sms, s)) != cudaSuccess)
      return cuda_fail(e, "optimizer launch (T = 0)");
    return FORGE_OK;
  }
  // A = dY^T [N x T] and B = X^T [K x T], token-contiguous: K-major operands,
  // 128 tokens (bytes) by 128 rows per box.
  CUtensorMap ma, mb, m1, m2, mw;
  if ((st = tensor_map(&ma, lin->dYt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, T, N, kFp8BlockK, kTileM,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FORGE_OK)
    return st;
  if ((st = tensor_map(&mb, lin->Xt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, T, K, kFp8BlockK, kTileN / 2,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FORGE_OK)
    return st;
  if ((st = state_maps(state, opt_kind, N, K, ma, &m1, &m2)) != FORGE_OK) return st;
  const int sdt = kernel_sdt(state, T);
  if ((st = weight_map(state, sdt, N, K, ma, &mw)) != FORGE_OK) return st;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  fill_tiles(p, N, K, T, kFp8BlockK);
  p.qblock = qblock_of(state->s_dtype);
  p.qshift = qshift_of(state->s_dtype);
  if (p.qblock != 256) split_tail(p, d.num_sms / 2);  // a 256-column block spans both halves
  CUtensorMap mbh = mb;
  if (p.split_from < p.num_tiles &&  // half units load 64 rows of X^T
      (st = tensor_map(&mbh, lin->Xt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, T, K, kFp8BlockK, kTileN / 4,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != FORGE_OK)
    return st;
  p.W = state->W; p.s1 = state->s1; p.s2 = state->s2;
  p.s1_scale = state->s1_scale; p.s2_scale = state->s2_scale;
  p.sc = sc;
  p.seed = seed;
  philox_round_keys(seed, p.round_keys);
  p.step = static_cast<uint64_t>(step);
  p.status = d.status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.skip_loads = g_skip_loads.load();
  p.gscale = static_cast<float>(c);
  if ((e = launch_tc_fp8(sdt, ma, mb, mbh, m1, m2, mw, p, grid_for(p, d), s)) != cudaSuccess)
    return cuda_fail(e, "FP8 step launch");
  return FORGE_OK;
}

void forge_set_step_fusion(int32_t enable) { g_step_fusion.store(enable != 0 ? 1 : 0); }

forge_status_t forge_linear_dgrad(const forge_linear_t* lin, const void* W, int32_t w_dtype, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if ((st = check_linear(lin, false)) != FORGE_OK) return st;
  if (w_dtype != FORGE_W_FP32 && w_dtype != FORGE_W_BF16_SR) return fail(FORGE_ERR_INVALID_ARG, "w_dtype %d", w_dtype);
  if (lin->T == 0 || lin->K == 0) return FORGE_OK;
  if (lin->dX == nullptr) return fail(FORGE_ERR_INVALID_ARG, "dX is NULL");
  if (lin->N > 0 && (W == nullptr || !aligned16(W))) return fail(FORGE_ERR_INVALID_ARG, "W must be 16-byte aligned");
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  if ((st = check_device(d)) != FORGE_OK) return st;
  return launch_dgrad(lin, W, w_dtype, static_cast<cudaStream_t>(stream), d);
}

forge_status_t forge_unfused_wgrad(const forge_linear_t* lin, float* dW, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if ((st = check_linear(lin, true)) != FORGE_OK) return st;
  if (lin->N == 0 || lin->K == 0) return FORGE_OK;
  if (dW == nullptr || !aligned16(dW)) return fail(FORGE_ERR_INVALID_ARG, "dW must be a 16-byte aligned device pointer");
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  if ((st = check_device(d)) != FORGE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (lin->T == 0) {
    if ((e = cudaMemsetAsync(dW, 0, static_cast<size_t>(lin->N * lin->K * 4), s)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync(dW)");
    return FORGE_OK;
  }
  CUtensorMap ma, mb;
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = wgrad_maps(lin, kWgradBlockK, &ma, &mb, &p.op3d)) != FORGE_OK) return st;
  fill_tiles(p, lin->N, lin->K, lin->T, kWgradBlockK);
  p.out = dW;
  p.status = d.status;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.skip_loads = g_skip_loads.load();
  if ((e = launch_tc_plain(kModeWgradStore, ma, mb, p, grid_for(p, d), s)) != cudaSuccess)
    return cuda_fail(e, "wgrad launch");
  return FORGE_OK;
}

forge_status_t forge_unfused_opt_step(const float* dW, const forge_state_t* state, int64_t N, int64_t K,
                                      int32_t opt_kind, const forge_hparams_t* hp, int64_t step,
                                      uint64_t seed, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if (N < 0 || K < 0 || K % 8 != 0) return fail(FORGE_ERR_INVALID_ARG, "need N >= 0 and K %% 8 == 0");
  if ((st = check_hp(opt_kind, hp, step)) != FORGE_OK) return st;
  if ((st = check_state(state, opt_kind, N, K)) != FORGE_OK) return st;
  if (N == 0 || K == 0) return FORGE_OK;
  if (dW != nullptr && !aligned16(dW)) return fail(FORGE_ERR_INVALID_ARG, "dW must be 16-byte aligned");
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  ElemParams ep;
  std::memset(&ep, 0, sizeof(ep));
  ep.dW = dW;
  ep.W = state->W; ep.s1 = state->s1; ep.s2 = state->s2;
  ep.s1_scale = state->s1_scale; ep.s2_scale = state->s2_scale;
  ep.N = N; ep.K = K;
  ep.sc = make_scalars(opt_kind, *hp, step);
  ep.seed = seed;
  ep.step = static_cast<uint64_t>(step);
  ep.qblock = qblock_of(state->s_dtype);
  cudaError_t e = launch_opt_step(state->w_dtype, base_sdt(state->s_dtype), ep, d.num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "optimizer launch");
  return FORGE_OK;
}

static forge_status_t quant_common(const void* a, const void* b, const float* absmax, int64_t rows,
                                   int64_t cols, int32_t block = 64) {
  if (block != 32 && block != 64 && block != 128 && block != 256)
    return fail(FORGE_ERR_INVALID_ARG, "block must be 32, 64, 128 or 256 (got %d)", block);
  if (rows < 0 || cols < 0 || cols % 64 != 0 || cols % block != 0)
    return fail(FORGE_ERR_INVALID_ARG, "need cols %% 64 == 0 and cols %% block == 0");
  if (rows * cols == 0) return FORGE_OK;
  if (a == nullptr || b == nullptr || absmax == nullptr || !aligned16(a) || !aligned16(b))
    return fail(FORGE_ERR_INVALID_ARG, "NULL or misaligned pointer");
  return FORGE_OK;
}

forge_status_t forge_quantize_state_block(const float* x, void* codes, float* absmax, int64_t rows,
                                          int64_t cols, int32_t is_signed, int32_t block, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if ((st = quant_common(x, codes, absmax, rows, cols, block)) != FORGE_OK) return st;
  if (rows * cols == 0) return FORGE_OK;
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  ElemParams ep;
  std::memset(&ep, 0, sizeof(ep));
  ep.dW = x; ep.s1 = codes; ep.s1_scale = absmax; ep.N = rows; ep.K = cols; ep.is_signed = is_signed ? 1 : 0;
  ep.qblock = block;
  cudaError_t e = launch_quantize(ep, d.num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return FORGE_OK;
}

forge_status_t forge_dequantize_state_block(const void* codes, const float* absmax, float* x, int64_t rows,
                                            int64_t cols, int32_t is_signed, int32_t block, void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  if ((st = quant_common(x, codes, absmax, rows, cols, block)) != FORGE_OK) return st;
  if (rows * cols == 0) return FORGE_OK;
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  ElemParams ep;
  std::memset(&ep, 0, sizeof(ep));
  ep.W = x; ep.s1 = const_cast<void*>(codes); ep.s1_scale = const_cast<float*>(absmax);
  ep.N = rows; ep.K = cols; ep.is_signed = is_signed ? 1 : 0;
  ep.qblock = block;
  cudaError_t e = launch_dequantize(ep, d.num_sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
  return FORGE_OK;
}

forge_status_t forge_quantize_state(const float* x, void* codes, float* absmax, int64_t rows, int64_t cols,
                                    int32_t is_signed, void* stream) {
  return forge_quantize_state_block(x, codes, absmax, rows, cols, is_signed, 64, stream);
}

forge_status_t forge_dequantize_state(const void* codes, const float* absmax, float* x, int64_t rows,
                                      int64_t cols, int32_t is_signed, void* stream) {
  return forge_dequantize_state_block(codes, absmax, x, rows, cols, is_signed, 64, stream);
}

forge_status_t forge_get_device_status(void* stream) {
  g_msg[0] = '\0';
  forge_status_t st;
  DeviceInfo d;
  if ((st = device_info(&d)) != FORGE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  if ((e = cudaMemcpy(&word, d.status, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read status word");
  if (word != 0) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(d.status, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear status word");
    if (word == kStatusTimeout) return fail(FORGE_ERR_TIMEOUT, "a pipeline wait in a kernel expired");
    return fail(FORGE_ERR_DEVICE, "device status %u", word);
  }
  return FORGE_OK;
}

forge_status_t forge_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 ? 2000000000ull : ns);
  return FORGE_OK;
}

forge_status_t forge_debug_skip_loads(int32_t enable) {
  g_skip_loads.store(enable ? 1 : 0);
  return FORGE_OK;
}

const char* forge_status_string(forge_status_t status) {
  switch (status) {
    case FORGE_OK: return "FORGE_OK";
    case FORGE_ERR_INVALID_ARG: return "FORGE_ERR_INVALID_ARG: invalid argument";
    case FORGE_ERR_UNSUPPORTED: return "FORGE_ERR_UNSUPPORTED: unsupported request";
    case FORGE_ERR_CUDA: return "FORGE_ERR_CUDA: CUDA runtime error";
    case FORGE_ERR_TIMEOUT: return "FORGE_ERR_TIMEOUT: device-side wait expired";
    case FORGE_ERR_DEVICE: return "FORGE_ERR_DEVICE: device-side error";
  }
  return "unknown forge_status_t";
}

const char* forge_last_error_message(void) { return g_msg; }

int32_t forge_abi_version(void) { return FORGE_ABI_VERSION; }

}  // extern "C"
