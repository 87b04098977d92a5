// The tensor-core kernel behind the fused step (alone, or in one launch with
// dX), the unfused wgrad pass and dX.
//
// FORGE (gist.science explainer), Technical Summary §2 "Core Mechanism": for
// each tile of W the partial products of dY and X are accumulated in FP32,
// the optimizer is applied to the finished tile at once, the gradient tile is
// discarded, and only the updated weights and moments are written back.
//
// GB300 design: clusters of two CTAs (one per SM), persistent over output
// tiles of 256 x 256; the pair runs tcgen05 with .cta_group::2, CTA r holding
// rows [128 r, 128 r + 128) of the tile in its tensor memory.
//   warp 0      one lane of each CTA issues TMA loads of its half of the
//               operands (its 128 rows of A, its 128 columns of B) into a
//               STG-deep shared-memory ring (128-byte swizzle); both halves
//               complete on the leader CTA's "full" mbarrier;
//   warp 1      allocates 512 tensor-memory columns (collectively with the
//               peer); in the leader one lane issues tcgen05.mma (M=256,
//               N=256, K=16, bf16 -> fp32; K=32 for E4M3) into one of two
//               TMEM accumulators,
//               so the MMAs of tile i+1 overlap the epilogue of tile i, and
//               multicasts its commits to both CTAs' "empty" / "tmem full"
//               barriers;
//   warps 2..   the epilogue of each CTA: tcgen05.ld pulls its 128 rows of
//               the finished fp32 tile into registers (one TMEM lane = one
//               output row), then runs the optimizer on it (FORGE), or stores
//               it as fp32 (unfused pass 1) or bf16 (dX); the epilogue warps
//               of both CTAs release the accumulator on the leader's barrier.
//               Plain modes and fp32 weights: warps 2..9 (direct stores).
//               The FORGE step with bf16 weights: warps 2..17 compute, warp
//               18 stages the optimizer states through shared memory with
//               TMA (with INT8 states over a short reduction, the weights
//               too; in the one-launch step it also stores the dX tiles that
//               run first in the same launch).
// Work units: whole tiles, except that in the FORGE step without dX a last
// partial wave (fewer tiles than half the pairs) runs as 128-column halves
// (N = 128 MMAs, half-width B boxes), each pair taking at most one as its
// last unit, so that wave takes half as long.
// Operand layouts (all 128-byte swizzled atoms of 8 rows x 128 bytes):
//   wgrad  A = dY^T tile [128 n x BK t] per CTA: dY is [T x N] with n
//          contiguous, so A is MN-major: two 64-wide column atoms BK*128
//          bytes apart (LBO), 8-row token groups 1 KiB apart (SBO).
//          B = X tile [128 k x BK t] per CTA, MN-major, two atoms.
//   dgrad  A = dY tile [128 t x 64 n], K-major (n contiguous); B = W tile
//          [128 k x 64 n] per CTA, MN-major.
//   FP8    the FORGE step from E4M3 codes stored token-contiguous: A = dY^T
//          tile [128 n x 128 t], B = X^T tile [128 k x 128 t] per CTA, both
//          K-major (one 128-byte row per output row and stage); tcgen05
//          kind::f8f6f4, K = 32 per instruction; the epilogue multiplies the
//          FP32 sum by the product of the two per-tensor scales.
// Every wait is bounded (GemmParams::wait_limit_ns): on expiry the CTA records
// a timeout in the status word, all roles stop, in-flight copies and MMAs are
// drained (again bounded), tensor memory is released and the CTA returns.
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "common.h"
#include "optim.cuh"
#include "ptx.cuh"

namespace forge {

struct SharedState {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t mma_done;
  uint64_t epi_full[2];     // staged epilogue chunk landed (TMA epilogue only)
  uint32_t tmem_base;
  int32_t abort;
};

// Per-instantiation layout (per CTA).  The FORGE step with bf16 weights
// stages its optimizer-state tiles through shared memory with TMA (two 32 KiB
// chunk buffers) next to a 5-stage operand ring; the other modes use a
// deeper ring.  A stage holds 128 rows of A and 128 columns of B (half of the
// pair's 256): 32 KiB at 64 tokens.
constexpr int kEpiBufBytes = 32768;
// INT8 states stage the bf16 weight chunk too (see StagedGeom).  With the
// method's block of 64 the buffer holds codes and weights only (32 KiB: the
// block absmax is exchanged inside the weight region, each thread loads its
// own old scale), so the ring keeps all five stages; the other block widths
// need two more small regions (a larger buffer) and give up one stage.
constexpr int kEpiBufBytesW = 37888;
__host__ __device__ constexpr bool stages_weights(int sdt) { return sdt == kSInt8W || sdt == kSInt8WX; }
__host__ __device__ constexpr bool compact_int8(int sdt) { return sdt == kSInt8W; }
constexpr int kEpiBarrier = 1;       // named barrier of the epilogue warps
constexpr int kEpiInnerBarrier = 2;  // the staged epilogue's compute warps only
constexpr int kPairM = 2 * kTileM;  // rows of a pair tile

template <int MODE, int WDT, int SDT = kSFp32>
struct KCfg {
  static constexpr bool kFp8 = (MODE == kModeFusedFp8);
  // the staged epilogue: every FORGE step with bf16 weights, and the fused
  // step with fp32 weights and fp32 states
  static constexpr bool kTmaEpi =
      ((MODE == kModeFusedOpt || MODE == kModeStep || kFp8) && WDT == kWBf16) ||
      (MODE == kModeFusedOpt && WDT == kWFp32 && SDT == kSFp32);
  static constexpr bool kStageW = kTmaEpi && stages_weights(SDT);
  static constexpr int kBK =
      kFp8 ? kFp8BlockK
           : (kTmaEpi ? kFusedBlockK : (MODE == kModeWgradStore ? kWgradBlockK : kBlockK));  // tokens per stage
  static constexpr int kStg =
      kTmaEpi ? (kStageW && !compact_int8(SDT) ? kFusedStages - 1 : kFusedStages)
              : (MODE == kModeWgradStore ? kWgradStages : kStages);
  static constexpr int kEsz = kFp8 ? 1 : 2;           // operand element bytes
  static constexpr int kA = kTileM * kBK * kEsz;       // bytes of A per stage (this CTA's 128 rows)
  static constexpr int kB = (kTileN / 2) * kBK * kEsz; // bytes of B per stage (this CTA's 128 columns)
  static constexpr int kEpiBuf = kStageW && !compact_int8(SDT) ? kEpiBufBytesW : kEpiBufBytes;
  static constexpr int kEpiBytes = kTmaEpi ? 2 * kEpiBuf : 0;
  static constexpr int kSmem = kStg * (kA + kB) + kEpiBytes + 512 + 1024;
  // TMA warp, MMA warp, epilogue warps (four per 32-lane quarter of TMEM in the
  // staged epilogue, two in the plain ones).
  static constexpr int kEpiWarps = kTmaEpi ? kNumEpiWarpsStaged : kNumEpiWarps;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + (kTmaEpi ? 1 : 0));  // + the I/O warp
};
static_assert(sizeof(SharedState) <= 512, "shared state region");
static_assert(KCfg<kModeFusedOpt, kWBf16>::kStg <= 8 && KCfg<kModeWgradStore, kWBf16>::kStg <= 8 &&
                  kStages <= 8, "barrier arrays");
static_assert(KCfg<kModeWgradStore, kWBf16>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeFusedOpt, kWBf16>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeDgrad, kWBf16>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeFusedFp8, kWBf16>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeStep, kWBf16, kSInt8W>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeFusedFp8, kWBf16, kSInt8W>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeStep, kWBf16, kSInt8WX>::kSmem <= 232448, "dynamic shared memory limit");
static_assert(KCfg<kModeFusedFp8, kWBf16, kSInt8WX>::kSmem <= 232448, "dynamic shared memory limit");

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting
// or the wait expired (the first expiry records the timeout).
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                             SharedState* ss, bool honour_abort = true) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *reinterpret_cast<volatile int32_t*>(&ss->abort)) return false;
    if (ptx::global_timer_ns() - t0 > p.wait_limit_ns) {
      *reinterpret_cast<volatile int32_t*>(&ss->abort) = 1;
      atomicCAS(p.status, 0u, static_cast<uint32_t>(kStatusTimeout));
      return false;
    }
  }
}

// Tile order: groups of kRasterGroup consecutive column tiles, row-major
// inside a group.  The ~num_SMs tiles in flight at once then cover a compact
// (num_SMs / 8) x 8 rectangle, so each wave streams a small set of operand
// column blocks from HBM instead of every column block of one operand.
constexpr int kRasterGroup = 8;

__device__ __forceinline__ void tile_coords_of(int tile, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int span = tiles_m * kRasterGroup;
  const int grp = tile / span;
  const int first_n = grp * kRasterGroup;
  const int width = min(kRasterGroup, tiles_n - first_n);
  const int local = tile - grp * span;
  tm = local / width;
  tn = first_n + (local - tm * width);
}
__device__ __forceinline__ void tile_coords(int tile, const GemmParams& p, int& tm, int& tn) {
  tile_coords_of(tile, p.tiles_m, p.tiles_n, tm, tn);
}

// Unit u of the weight tiles (see GemmParams::split_from): its tile and, for
// a half unit, which 128-column half (0 or 1); -1 for a whole tile.
__device__ __forceinline__ void unit_coords(int u, const GemmParams& p, int& tm, int& tn, int& half) {
  const bool split = u >= p.split_from;
  half = split ? ((u - p.split_from) & 1) : -1;
  tile_coords(split ? p.split_from + ((u - p.split_from) >> 1) : u, p, tm, tn);
}

// ------------------------------------------------------------------ roles

// Tile index of the pair's i-th tile, and the CTA's rank in the pair.
__device__ __forceinline__ int pair_id() { return static_cast<int>(blockIdx.x) >> 1; }
__device__ __forceinline__ int num_pairs() { return static_cast<int>(gridDim.x) >> 1; }

// One-launch step: a pair first runs its dX tiles, then its dW tiles
// pair_id(), pair_id() + num_pairs(), ...  The dX tiles are dealt in rounds,
// one per pair for the first dx_rounds rounds, then round-robin over the
// pairs from dx_heavy on (those with one dW tile fewer), so the pairs' work
// comes out about even; consecutive tiles run side by side in every round.
__device__ __forceinline__ int my_dx_tiles(const GemmParams& p) {
  int n = p.dx_rounds;
  if (pair_id() >= p.dx_heavy) {
    const int nl = num_pairs() - p.dx_heavy, lr = pair_id() - p.dx_heavy;
    const int rem = p.dx_tiles - p.dx_rounds * num_pairs();
    n += rem > lr ? (rem - 1 - lr) / nl + 1 : 0;
  }
  return n;
}
__device__ __forceinline__ void dx_tile_coords(int i, const GemmParams& p, int& tm, int& tn) {
  const int d = i < p.dx_rounds
                    ? i * num_pairs() + pair_id()
                    : p.dx_rounds * num_pairs() + (i - p.dx_rounds) * (num_pairs() - p.dx_heavy) +
                          (pair_id() - p.dx_heavy);
  tile_coords_of(d, p.dx_tiles_m, p.tiles_n, tm, tn);
}

template <int MODE, int STG, int BK>
__device__ void producer_role(const CUtensorMap* mA, const CUtensorMap* mB, const CUtensorMap* mDA,
                              const CUtensorMap* mDB, const GemmParams& p, uint8_t* smA,
                              uint8_t* smB, SharedState* ss, uint32_t rank) {
  constexpr int kEsz = MODE == kModeFusedFp8 ? 1 : 2;
  constexpr int kA = kTileM * BK * kEsz, kB = (kTileN / 2) * BK * kEsz;
  uint32_t it = 0;
  uint32_t issued_mask = 0;
  uint32_t last_parity = 0;  // bit s: parity of the last phase armed on full[s]
  const uint32_t full0 = ptx::mapa(ptx::smem_addr(&ss->full[0]), 0);  // the leader's barriers
  if (!p.skip_loads) {
    if (MODE == kModeStep) {  // the dX tiles: A = dY (K-major), B = W (MN-major)
      const int ndx = my_dx_tiles(p);
      for (int i = 0; i < ndx; ++i) {
        int tm, tn;
        dx_tile_coords(i, p, tm, tn);
        const int m0 = tm * kPairM + static_cast<int>(rank) * kTileM;
        const int n0 = tn * kTileN + static_cast<int>(rank) * (kTileN / 2);
        for (int kb = 0; kb < p.dx_num_kb; ++kb, ++it) {
          const int s = static_cast<int>(it % STG);
          const uint32_t ph = (it / STG) & 1u;
          if (!bounded_wait(&ss->empty[s], ph ^ 1u, p, ss)) goto drain;
          const uint32_t bar = full0 + static_cast<uint32_t>(s) * 8u;
          if (rank == 0) ptx::mbar_arrive_expect_tx(&ss->full[s], 2u * (kA + kB));
          ptx::tma_load_2d_pair(mDA, bar, smA + s * kA, kb * BK, m0);
          ptx::tma_load_3d_pair(mDB, bar, smB + s * kB, 0, kb * BK, n0 / 64);
          issued_mask |= 1u << s;
          last_parity = (last_parity & ~(1u << s)) | (ph << s);
        }
      }
    }
    for (int u = pair_id(); u < p.num_units; u += num_pairs()) {
      int tm, tn, half;
      unit_coords(u, p, tm, tn, half);
      const int m0 = tm * kPairM + static_cast<int>(rank) * kTileM;  // this CTA's A rows
      // this CTA's B columns: 128 of a whole tile, 64 of a half unit (whose B
      // boxes come from the half-width map, passed as mDB)
      const int n0 = half < 0 ? tn * kTileN + static_cast<int>(rank) * (kTileN / 2)
                              : tn * kTileN + half * (kTileN / 2) + static_cast<int>(rank) * (kTileN / 4);
      const uint32_t bytes = half < 0 ? 2u * (kA + kB) : 2u * (kA + kB / 2);
      for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
        const int s = static_cast<int>(it % STG);
        const uint32_t ph = (it / STG) & 1u;
        if (!bounded_wait(&ss->empty[s], ph ^ 1u, p, ss)) goto drain;
        const uint32_t bar = full0 + static_cast<uint32_t>(s) * 8u;
        if (rank == 0) ptx::mbar_arrive_expect_tx(&ss->full[s], bytes);
        uint8_t* a = smA + s * kA;
        uint8_t* b = smB + s * kB;
        if (MODE == kModeFusedFp8) {  // dY^T and X^T, token-contiguous: one 128 x 128-byte box each
          ptx::tma_load_2d_pair(mA, bar, a, kb * BK, m0);
          ptx::tma_load_2d_pair(half < 0 ? mB : mDB, bar, b, kb * BK, n0);
          issued_mask |= 1u << s;
          last_parity = (last_parity & ~(1u << s)) | (ph << s);
          continue;
        }
        if (MODE == kModeDgrad) {
          ptx::tma_load_2d_pair(mA, bar, a, kb * BK, m0);
        } else if (p.op3d) {  // [2 column blocks][BK rows][64 columns] in one copy
          ptx::tma_load_3d_pair(mA, bar, a, 0, kb * BK, m0 / 64);
        } else {
          ptx::tma_load_2d_pair(mA, bar, a, m0, kb * BK);
          ptx::tma_load_2d_pair(mA, bar, a + 64 * BK * 2, m0 + 64, kb * BK);
        }
        if (p.op3d) {
          ptx::tma_load_3d_pair(half < 0 ? mB : mDB, bar, b, 0, kb * BK, n0 / 64);
        } else {
          ptx::tma_load_2d_pair(mB, bar, b, n0, kb * BK);
          if (half < 0) ptx::tma_load_2d_pair(mB, bar, b + 64 * BK * 2, n0 + 64, kb * BK);
        }
        issued_mask |= 1u << s;
        last_parity = (last_parity & ~(1u << s)) | (ph << s);
      }
    }
  }
drain:
  // Every issued copy lands before the pair can exit (already true unless a
  // consumer gave up early).  The leader's full barriers count both CTAs'
  // copies; the peer's copies are covered by the leader's drain and the
  // cluster barrier at the end of the kernel.
  if (rank == 0)
    for (int s = 0; s < STG; ++s)
      if (issued_mask & (1u << s)) bounded_wait(&ss->full[s], (last_parity >> s) & 1u, p, ss, false);
}

// Leader CTA only.
template <int MODE, int STG, int BK>
__device__ void mma_role(const GemmParams& p, uint8_t* smA, uint8_t* smB, SharedState* ss) {
  constexpr bool kFp8 = MODE == kModeFusedFp8;
  constexpr int kA = kTileM * BK * (kFp8 ? 1 : 2), kB = (kTileN / 2) * BK * (kFp8 ? 1 : 2);
  uint32_t it = 0;
  int local = 0;
  // One tile into accumulator local & 1: num_kb stages; A K-major (dX: dY) or
  // MN-major (dW: dY^T); B MN-major.  False if the CTA is aborting.
  auto run_tile = [&](int num_kb, bool a_kmajor, int n_cols) -> bool {
    const int acc = local & 1;
    const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
    if (!bounded_wait(&ss->tmem_empty[acc], aph ^ 1u, p, ss)) return false;
    ptx::tc_fence_after();
    const uint32_t idesc = kFp8       ? ptx::idesc_e4m3_f32(kPairM, n_cols)
                           : a_kmajor ? ptx::idesc_bf16_f32(kPairM, n_cols, false, true)
                                      : ptx::idesc_bf16_f32(kPairM, n_cols, true, true);
    const uint32_t d_tmem = ss->tmem_base + static_cast<uint32_t>(acc * kTileN);
    for (int kb = 0; kb < num_kb; ++kb, ++it) {
      const int s = static_cast<int>(it % STG);
      const uint32_t ph = (it / STG) & 1u;
      if (!bounded_wait(&ss->full[s], ph, p, ss)) return false;
      ptx::tc_fence_after();
      const uint32_t a0 = ptx::smem_addr(smA + s * kA);
      const uint32_t b0 = ptx::smem_addr(smB + s * kB);
      if constexpr (kFp8) {
        // Both operands K-major: 32 E4M3 = 32 B of each 128-byte swizzle row
        // per instruction, 8-row groups 1 KiB apart.
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk)
          ptx::mma_e4m3_pair(d_tmem, ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024),
                             ptx::smem_desc_sw128(b0 + kk * 32, 16, 1024), idesc,
                             (kb | kk) != 0 ? 1u : 0u);
        ptx::mma_commit_pair_multicast(&ss->empty[s], 0x3);
        continue;
      }
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        // MN-major: 16 reduction rows = two 8-row groups of 128 B -> +2 KiB;
        // atoms of 64 columns x BK rows sit BK*128 bytes apart (LBO).
        // K-major: 16 bf16 = 32 B inside the 128-byte swizzle row.
        const uint64_t adesc = a_kmajor ? ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024)
                                        : ptx::smem_desc_sw128(a0 + kk * 2048, BK * 128, 1024);
        const uint64_t bdesc = ptx::smem_desc_sw128(b0 + kk * 2048, BK * 128, 1024);
        ptx::mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      ptx::mma_commit_pair_multicast(&ss->empty[s], 0x3);  // frees the stage in both CTAs
    }
    ptx::mma_commit_pair_multicast(&ss->tmem_full[acc], 0x3);  // accumulator complete
    ++local;
    return true;
  };
  if (MODE == kModeStep) {
    const int ndx = my_dx_tiles(p);
    for (int i = 0; i < ndx; ++i)
      if (!run_tile(p.dx_num_kb, true, kTileN)) goto done;
  }
  for (int u = pair_id(); u < p.num_units; u += num_pairs())  // a half unit: N = 128
    if (!run_tile(p.num_kb, MODE == kModeDgrad, u < p.split_from ? kTileN : kTileN / 2)) goto done;
done:
  // Tensor memory may be released only after every issued MMA has finished.
  ptx::mma_commit_pair_multicast(&ss->mma_done, 0x1);
  bounded_wait(&ss->mma_done, 0u, p, ss, false);
}

// ------------------------------------------------------------------ epilogues

// W / state traffic of the epilogue touches each line once (read, then
// written back): keep it out of L1 and mark it evict-first in L2, so it does
// not displace the operand tiles the main loop re-reads from L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

__device__ __forceinline__ void st_stream(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
               ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void ld8f(const float* p, float (&v)[8], uint64_t pol) {
  const uint4 a = ld_stream(p, pol), b = ld_stream(p + 4, pol);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
  v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

__device__ __forceinline__ void st8f(float* p, const float (&v)[8], uint64_t pol) {
  st_stream(p, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3])), pol);
  st_stream(p + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                              __float_as_uint(v[6]), __float_as_uint(v[7])), pol);
}

__device__ __forceinline__ void ld8bf16(const uint16_t* p, float (&w)[8], uint64_t pol) {
  const uint4 wb = ld_stream(p, pol);
  const uint32_t wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    w[2 * j] = dev::bf16_to_f32(wv[j] & 0xFFFFu);
    w[2 * j + 1] = dev::bf16_to_f32(wv[j] >> 16);
  }
}

// 8 consecutive elements e0..e0+7 of one row of W (e0 % 8 == 0), fp32 or no
// state: load, apply the rule, round, store.
template <int KIND, int WDT>
__device__ __forceinline__ void group8_fp32state(const float* g, int64_t e0, const GemmParams& p,
                                                 uint64_t pol) {
  float w[8], s1[8], s2[8];
  if (WDT == kWBf16) ld8bf16(static_cast<const uint16_t*>(p.W) + e0, w, pol);
  else ld8f(static_cast<const float*>(p.W) + e0, w, pol);
  if (uses_s1(KIND)) ld8f(static_cast<const float*>(p.s1) + e0, s1, pol);
  if (uses_s2(KIND)) ld8f(static_cast<const float*>(p.s2) + e0, s2, pol);
#pragma unroll
  for (int j = 0; j < 8; ++j) dev::rule<KIND>(w[j], g[j], s1[j], s2[j], p.sc);
  if (WDT == kWBf16) {
    const uint4 r = dev::sr_words_rk((static_cast<uint64_t>(e0) >> 3) + p.sr_base, p.step, p.round_keys);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = dev::bf16_sr(w[2 * j], dev::sr_bits(r, 2 * j)) |
             (dev::bf16_sr(w[2 * j + 1], dev::sr_bits(r, 2 * j + 1)) << 16);
    st_stream(static_cast<uint16_t*>(p.W) + e0, make_uint4(o[0], o[1], o[2], o[3]), pol);
  } else {
    st8f(static_cast<float*>(p.W) + e0, w, pol);
  }
  if (uses_s1(KIND)) st8f(static_cast<float*>(p.s1) + e0, s1, pol);
  if (uses_s2(KIND)) st8f(static_cast<float*>(p.s2) + e0, s2, pol);
}

template <int KIND, int WDT>
__device__ __forceinline__ void epi_fused_fp32state(uint32_t tbase, int64_t row, int colbase,
                                                    bool row_ok, const GemmParams& p) {
  const int64_t K = p.Ncols;
  const uint64_t pol = evict_first_policy();
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float g[32];
    ptx::tmem_ld_32x32b_x32(tbase + c * 32, g);
    if (!row_ok) continue;
    const int col0 = colbase + c * 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (col0 + q * 8 < K) group8_fp32state<KIND, WDT>(g + q * 8, row * K + col0 + q * 8, p, pol);
    }
  }
}

// Byte j of a 64-byte code block held in 16 words.
__device__ __forceinline__ int code_at(const uint32_t (&c)[16], int j, bool is_signed) {
  const uint32_t b = (c[j >> 2] >> (8 * (j & 3))) & 0xFFu;
  return is_signed ? static_cast<int>(static_cast<int8_t>(b)) : static_cast<int>(b);
}

// One INT8 block of 64 elements of one row (the thread owns the whole block):
// pass 1 finds the new absmax of each state, pass 2 recomputes the same
// element results, writes W, and quantises the states with the new absmax.
template <int KIND, int WDT>
__device__ __forceinline__ void epi_fused_int8_block(uint32_t tblock, int64_t row, int col0,
                                                     bool ok, const GemmParams& p) {
  const int64_t K = p.Ncols;
  const int64_t e_blk = row * K + col0;
  const int64_t sidx = row * (K / 64) + col0 / 64;
  uint32_t c1[16], c2[16];
  float a1 = 0.f, a2 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) { c1[i] = 0u; c2[i] = 0u; }
  if (ok) {
    if (uses_s1(KIND)) {
      const uint4* q = reinterpret_cast<const uint4*>(static_cast<const int8_t*>(p.s1) + e_blk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = q[i];
        c1[4 * i] = v.x; c1[4 * i + 1] = v.y; c1[4 * i + 2] = v.z; c1[4 * i + 3] = v.w;
      }
      a1 = p.s1_scale[sidx];
    }
    if (uses_s2(KIND)) {
      const uint4* q = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.s2) + e_blk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = q[i];
        c2[4 * i] = v.x; c2[4 * i + 1] = v.y; c2[4 * i + 2] = v.z; c2[4 * i + 3] = v.w;
      }
      a2 = p.s2_scale[sidx];
    }
  }
  const bool need_w_for_state = (KIND != kAdamW && KIND != kLion) && p.sc.l2 != 0.f;
  float n1 = 0.f, n2 = 0.f;  // new absmax
  // ---- pass 1: new states, absmax only
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float g[32];
    ptx::tmem_ld_32x32b_x32(tblock + half * 32, g);
    if (!ok) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float w[8];
      const int64_t e0 = e_blk + half * 32 + q * 8;
      if (need_w_for_state) {
        if (WDT == kWBf16) {
          const uint4 wb = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.W) + e0);
          const uint32_t wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            w[2 * j] = dev::bf16_to_f32(wv[j] & 0xFFFFu);
            w[2 * j + 1] = dev::bf16_to_f32(wv[j] >> 16);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) w[j] = static_cast<const float*>(p.W)[e0 + j];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = half * 32 + q * 8 + j;
        float s1 = uses_s1(KIND) ? dev::dequant<true>(code_at(c1, jj, true), a1) : 0.f;
        float s2 = uses_s2(KIND) ? dev::dequant<false>(code_at(c2, jj, false), a2) : 0.f;
        float wj = w[j];
        dev::rule<KIND>(wj, g[q * 8 + j], s1, s2, p.sc);
        if (uses_s1(KIND)) n1 = dev::absmax_acc(n1, s1);
        if (uses_s2(KIND)) n2 = dev::absmax_acc(n2, s2);
      }
    }
  }
  // ---- pass 2: recompute, write W, quantise states
  uint32_t o1[16], o2[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) { o1[i] = 0u; o2[i] = 0u; }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float g[32];
    ptx::tmem_ld_32x32b_x32(tblock + half * 32, g);
    if (!ok) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float w[8];
      const int64_t e0 = e_blk + half * 32 + q * 8;
      if (WDT == kWBf16) {
        const uint4 wb = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.W) + e0);
        const uint32_t wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          w[2 * j] = dev::bf16_to_f32(wv[j] & 0xFFFFu);
          w[2 * j + 1] = dev::bf16_to_f32(wv[j] >> 16);
        }
      } else {
        const float4* wp = reinterpret_cast<const float4*>(static_cast<const float*>(p.W) + e0);
        const float4 a = wp[0], b = wp[1];
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = half * 32 + q * 8 + j;
        float s1 = uses_s1(KIND) ? dev::dequant<true>(code_at(c1, jj, true), a1) : 0.f;
        float s2 = uses_s2(KIND) ? dev::dequant<false>(code_at(c2, jj, false), a2) : 0.f;
        dev::rule<KIND>(w[j], g[q * 8 + j], s1, s2, p.sc);
        if (uses_s1(KIND))
          o1[jj >> 2] |= (static_cast<uint32_t>(dev::quant<true>(s1, n1)) & 0xFFu) << (8 * (jj & 3));
        if (uses_s2(KIND))
          o2[jj >> 2] |= (static_cast<uint32_t>(dev::quant<false>(s2, n2)) & 0xFFu) << (8 * (jj & 3));
      }
      if (WDT == kWBf16) {
        const uint4 r = dev::sr_words_rk((static_cast<uint64_t>(e0) >> 3) + p.sr_base, p.step, p.round_keys);
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = dev::bf16_sr(w[2 * j], dev::sr_bits(r, 2 * j)) |
                 (dev::bf16_sr(w[2 * j + 1], dev::sr_bits(r, 2 * j + 1)) << 16);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.W) + e0) =
            make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        float4* wp = reinterpret_cast<float4*>(static_cast<float*>(p.W) + e0);
        wp[0] = make_float4(w[0], w[1], w[2], w[3]);
        wp[1] = make_float4(w[4], w[5], w[6], w[7]);
      }
    }
  }
  if (!ok) return;
  if (uses_s1(KIND)) {
    uint4* q = reinterpret_cast<uint4*>(static_cast<int8_t*>(p.s1) + e_blk);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = make_uint4(o1[4 * i], o1[4 * i + 1], o1[4 * i + 2], o1[4 * i + 3]);
    p.s1_scale[sidx] = n1;
  }
  if (uses_s2(KIND)) {
    uint4* q = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.s2) + e_blk);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = make_uint4(o2[4 * i], o2[4 * i + 1], o2[4 * i + 2], o2[4 * i + 3]);
    p.s2_scale[sidx] = n2;
  }
}

template <int KIND, int WDT, int SDT>
__device__ __forceinline__ void epi_fused(uint32_t tbase, int64_t row, int colbase, bool row_ok,
                                          const GemmParams& p) {
  if (SDT == kSInt8) {
#pragma unroll 1
    for (int blk = 0; blk < 2; ++blk) {
      const int col0 = colbase + blk * 64;
      epi_fused_int8_block<KIND, WDT>(tbase + blk * 64, row, col0, row_ok && col0 < p.Ncols, p);
    }
  } else {
    epi_fused_fp32state<KIND, WDT>(tbase, row, colbase, row_ok, p);
  }
}

template <int WDT, int SDT>
__device__ __forceinline__ void epi_fused_dispatch(uint32_t tbase, int64_t row, int colbase,
                                                   bool row_ok, const GemmParams& p) {
  switch (p.sc.kind) {
    case kAdamW: epi_fused<kAdamW, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    case kNAdam: epi_fused<kNAdam, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    case kRAdam: epi_fused<kRAdam, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    case kLion: epi_fused<kLion, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    case kRMSprop: epi_fused<kRMSprop, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    case kAdaGrad: epi_fused<kAdaGrad, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    case kSGD: epi_fused<kSGD, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
    default: epi_fused<kSGDMomentum, WDT, SDT>(tbase, row, colbase, row_ok, p); break;
  }
}

// fp32 store of the accumulator (unfused pass 1) or bf16 store (dX).
template <int MODE>
__device__ __forceinline__ void epi_store(uint32_t tbase, int64_t row, int colbase, bool row_ok,
                                          const GemmParams& p) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float g[32];
    ptx::tmem_ld_32x32b_x32(tbase + c * 32, g);
    if (!row_ok) continue;
    const int col0 = colbase + c * 32;
    if (MODE == kModeWgradStore) {
      float* out = static_cast<float*>(p.out) + row * static_cast<int64_t>(p.Ncols);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (col0 + q * 4 < p.Ncols)
          *reinterpret_cast<float4*>(out + col0 + q * 4) =
              make_float4(g[4 * q], g[4 * q + 1], g[4 * q + 2], g[4 * q + 3]);
    } else {
      uint16_t* out = static_cast<uint16_t*>(p.out) + row * static_cast<int64_t>(p.Ncols);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (col0 + q * 8 >= p.Ncols) continue;
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(g[8 * q + 2 * j], g[8 * q + 2 * j + 1]);
          o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(out + col0 + q * 8) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// L2 prefetch of the (up to) 128 columns from `col0` of row `row` of W and of
// the states the rule reads: one request per 128-byte line, no registers held.
__device__ __forceinline__ void prefetch_l2(const void* base, int64_t byte0, int64_t bytes) {
  const char* b = static_cast<const char*>(base) + byte0;
  for (int64_t o = 0; o < bytes; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(b + o));
}
template <int WDT, int SDT>
__device__ __forceinline__ void prefetch_row_l2(int64_t row, int col0, const GemmParams& p) {
  const int64_t K = p.Ncols;
  const int64_t n = min(static_cast<int64_t>(128), K - col0);
  const int64_t e0 = row * K + col0;
  prefetch_l2(p.W, e0 * (WDT == kWBf16 ? 2 : 4), n * (WDT == kWBf16 ? 2 : 4));
  const int esz = SDT == kSInt8 ? 1 : (SDT == kSBf16 ? 2 : 4);
  const bool u1 = uses_s1(p.sc.kind), u2 = uses_s2(p.sc.kind);
  if (u1) prefetch_l2(p.s1, e0 * esz, n * esz);
  if (u2) prefetch_l2(p.s2, e0 * esz, n * esz);
}

template <int MODE, int WDT, int SDT>
__device__ void epilogue_role(const GemmParams& p, SharedState* ss, int warp, int lane,
                              uint32_t rank) {
  const int quarter = warp & 3;           // TMEM lanes this warp may access
  const int half = (warp - 2) >> 2;       // which 128 of the 256 columns
  const int r = quarter * 32 + lane;
  int local = 0;
  const uint32_t empty0 = ptx::mapa(ptx::smem_addr(&ss->tmem_empty[0]), 0);
  for (int tile = pair_id(); tile < p.num_tiles; tile += num_pairs(), ++local) {
    const int acc = local & 1;
    const uint32_t aph = (static_cast<uint32_t>(local) >> 1) & 1u;
    int tm, tn;
    tile_coords(tile, p, tm, tn);
    const int64_t row = static_cast<int64_t>(tm) * kPairM + rank * kTileM + r;
    const int colbase = tn * kTileN + half * 128;
    const bool row_ok = row < p.M;
    // While the tile's main loop runs, pull this thread's weights and states
    // into L2, so the epilogue's loads (one round trip per 8 elements) hit.
    if (MODE == kModeFusedOpt && row_ok && colbase < p.Ncols) prefetch_row_l2<WDT, SDT>(row, colbase, p);
    // One thread waits; the others block on the named barrier, which also
    // hands every warp the same verdict, so warps stay converged for the
    // .sync.aligned tensor-memory loads that follow.
    bool ok = true;
    if (warp == 2 && lane == 0) ok = bounded_wait(&ss->tmem_full[acc], aph, p, ss);
    if (ptx::bar_red_or(kEpiBarrier, 32 * kNumEpiWarps, !ok)) break;
    if (MODE == kModeFusedOpt && local == 0) ptx::grid_dep_wait();  // before the first write
    ptx::tc_fence_after();
    const uint32_t tbase = ss->tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(acc * kTileN + half * 128);
    if (MODE == kModeFusedOpt)
      epi_fused_dispatch<WDT, SDT>(tbase, row, colbase, row_ok, p);
    else
      epi_store<MODE>(tbase, row, colbase, row_ok, p);
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(empty0 + static_cast<uint32_t>(acc) * 8u);
  }
}

// ------------------------------------------------------------------ TMA-staged epilogue

// Byte offset of 16-byte chunk c of row r in a box of 64-byte rows stored with
// the 64-byte swizzle, and of 128-byte rows with the 128-byte swizzle (the
// layouts the tensor-memory accelerator writes).  Eight consecutive rows
// reading the same logical chunk hit eight different bank groups.
__device__ __forceinline__ uint32_t sw64(int r, int c) {
  return static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void unpack_bf16x8(uint4 v, float* w) {
  const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    w[2 * j] = dev::bf16_to_f32(a[j] & 0xFFFFu);
    w[2 * j + 1] = dev::bf16_to_f32(a[j] >> 16);
  }
}

// Eight weights to bf16 by stochastic rounding (dev::bf16_sr), packed in
// pairs.  When all eight are finite (w * 0 is then 0; an infinite or NaN w
// makes the sum NaN), each is its bit pattern plus its 16 random bits, upper
// half kept: the two halves of a word come from one byte permutation.
__device__ __forceinline__ uint4 pack_sr_bf16x8(const float* w, uint4 rnd) {
  float probe = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) probe = __fmaf_rn(w[j], 0.f, probe);
  const uint32_t rw[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  uint32_t o[4];
  if (probe == probe) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = __byte_perm(__float_as_uint(w[2 * j]) + (rw[j] & 0xFFFFu),
                         __float_as_uint(w[2 * j + 1]) + (rw[j] >> 16), 0x7632u);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = dev::bf16_sr(w[2 * j], dev::sr_bits(rnd, 2 * j)) |
             (dev::bf16_sr(w[2 * j + 1], dev::sr_bits(rnd, 2 * j + 1)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// FP8 operands: the accumulated sum of E4M3 code products times the product
// of the two per-tensor scales is the gradient.
__device__ __forceinline__ void scale_grad(float (&g)[8], const GemmParams& p) {
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = __fmul_rn(g[j], p.gscale);
}

// fp32 states: a chunk is 128 rows x 32 columns (m and v 16 KiB each in
// shared memory); this thread owns 8 columns of row r (two 16-byte chunks of
// each state), starting at element e0.  Its 8 bf16 weights come in and go out
// in registers (`wv`).
template <int KIND, bool SCALE>
__device__ __forceinline__ void epi_chunk_fp32(uint32_t taddr, uint8_t* buf, int r, int sub,
                                               int64_t e0, uint4& wv, const GemmParams& p) {
  constexpr int kOffS1 = 0, kOffS2 = 16384;
  float g[8], w[8], s1[8], s2[8];
  uint32_t gr[8];
  ptx::tmem_ld_issue(taddr, gr);  // the gradient arrives while the states are read
  unpack_bf16x8(wv, w);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (uses_s1(KIND)) {
      const float4 x = *reinterpret_cast<const float4*>(buf + kOffS1 + sw128(r, 2 * sub + i));
      s1[4 * i] = x.x; s1[4 * i + 1] = x.y; s1[4 * i + 2] = x.z; s1[4 * i + 3] = x.w;
    } else {
      s1[4 * i] = s1[4 * i + 1] = s1[4 * i + 2] = s1[4 * i + 3] = 0.f;
    }
    if (uses_s2(KIND)) {
      const float4 x = *reinterpret_cast<const float4*>(buf + kOffS2 + sw128(r, 2 * sub + i));
      s2[4 * i] = x.x; s2[4 * i + 1] = x.y; s2[4 * i + 2] = x.z; s2[4 * i + 3] = x.w;
    } else {
      s2[4 * i] = s2[4 * i + 1] = s2[4 * i + 2] = s2[4 * i + 3] = 0.f;
    }
  }
  // the rounding bits depend on the element index only: their ten dependent
  // rounds overlap the wait for the gradient
  const uint4 rnd = dev::sr_words_rk((static_cast<uint64_t>(e0) >> 3) + p.sr_base, p.step, p.round_keys);
  ptx::tmem_wait_ld(gr);
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = __uint_as_float(gr[j]);
  if (SCALE) scale_grad(g, p);
#pragma unroll
  for (int j = 0; j < 8; ++j) dev::rule<KIND>(w[j], g[j], s1[j], s2[j], p.sc);
  wv = pack_sr_bf16x8(w, rnd);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (uses_s1(KIND))
      *reinterpret_cast<float4*>(buf + kOffS1 + sw128(r, 2 * sub + i)) =
          make_float4(s1[4 * i], s1[4 * i + 1], s1[4 * i + 2], s1[4 * i + 3]);
    if (uses_s2(KIND))
      *reinterpret_cast<float4*>(buf + kOffS2 + sw128(r, 2 * sub + i)) =
          make_float4(s2[4 * i], s2[4 * i + 1], s2[4 * i + 2], s2[4 * i + 3]);
  }
}

// fp32 states and fp32 weights: as epi_chunk_fp32, with the thread's 8 fp32
// weights in registers (`wv`, two 16-byte words) written back unrounded.
template <int KIND>
__device__ __forceinline__ void epi_chunk_fp32w(uint32_t taddr, uint8_t* buf, int r, int sub,
                                                uint4 (&wv)[2], const GemmParams& p) {
  constexpr int kOffS1 = 0, kOffS2 = 16384;
  float g[8], w[8], s1[8], s2[8];
  uint32_t gr[8];
  ptx::tmem_ld_issue(taddr, gr);  // the gradient arrives while the states are read
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    w[4 * i] = __uint_as_float(wv[i].x); w[4 * i + 1] = __uint_as_float(wv[i].y);
    w[4 * i + 2] = __uint_as_float(wv[i].z); w[4 * i + 3] = __uint_as_float(wv[i].w);
    if (uses_s1(KIND)) {
      const float4 x = *reinterpret_cast<const float4*>(buf + kOffS1 + sw128(r, 2 * sub + i));
      s1[4 * i] = x.x; s1[4 * i + 1] = x.y; s1[4 * i + 2] = x.z; s1[4 * i + 3] = x.w;
    } else {
      s1[4 * i] = s1[4 * i + 1] = s1[4 * i + 2] = s1[4 * i + 3] = 0.f;
    }
    if (uses_s2(KIND)) {
      const float4 x = *reinterpret_cast<const float4*>(buf + kOffS2 + sw128(r, 2 * sub + i));
      s2[4 * i] = x.x; s2[4 * i + 1] = x.y; s2[4 * i + 2] = x.z; s2[4 * i + 3] = x.w;
    } else {
      s2[4 * i] = s2[4 * i + 1] = s2[4 * i + 2] = s2[4 * i + 3] = 0.f;
    }
  }
  ptx::tmem_wait_ld(gr);
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = __uint_as_float(gr[j]);
#pragma unroll
  for (int j = 0; j < 8; ++j) dev::rule<KIND>(w[j], g[j], s1[j], s2[j], p.sc);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    wv[i] = make_uint4(__float_as_uint(w[4 * i]), __float_as_uint(w[4 * i + 1]), __float_as_uint(w[4 * i + 2]),
                       __float_as_uint(w[4 * i + 3]));
    if (uses_s1(KIND))
      *reinterpret_cast<float4*>(buf + kOffS1 + sw128(r, 2 * sub + i)) =
          make_float4(s1[4 * i], s1[4 * i + 1], s1[4 * i + 2], s1[4 * i + 3]);
    if (uses_s2(KIND))
      *reinterpret_cast<float4*>(buf + kOffS2 + sw128(r, 2 * sub + i)) =
          make_float4(s2[4 * i], s2[4 * i + 1], s2[4 * i + 2], s2[4 * i + 3]);
  }
}

// bf16 states: a chunk is 128 rows x 32 columns (m and v 8 KiB each in
// shared memory, 64-byte rows with the 64-byte swizzle); this thread owns 8
// columns of row r (16 bytes of each state), starting at element e0.  The
// rule runs on the widened moments; the new ones are rounded to nearest even.
template <int KIND, bool SCALE>
__device__ __forceinline__ void epi_chunk_bf16s(uint32_t taddr, uint8_t* buf, int r, int sub,
                                                int64_t e0, uint4& wv, const GemmParams& p) {
  constexpr int kOffS1 = 0, kOffS2 = 8192;
  float g[8], w[8], s1[8], s2[8];
  uint32_t gr[8];
  ptx::tmem_ld_issue(taddr, gr);  // the gradient arrives while the states are read
  unpack_bf16x8(wv, w);
  if (uses_s1(KIND)) unpack_bf16x8(*reinterpret_cast<const uint4*>(buf + kOffS1 + sw64(r, sub)), s1);
  if (uses_s2(KIND)) unpack_bf16x8(*reinterpret_cast<const uint4*>(buf + kOffS2 + sw64(r, sub)), s2);
  const uint4 rnd = dev::sr_words_rk((static_cast<uint64_t>(e0) >> 3) + p.sr_base, p.step, p.round_keys);
  ptx::tmem_wait_ld(gr);
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = __uint_as_float(gr[j]);
  if (SCALE) scale_grad(g, p);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (!uses_s1(KIND)) s1[j] = 0.f;
    if (!uses_s2(KIND)) s2[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) dev::rule<KIND>(w[j], g[j], s1[j], s2[j], p.sc);
  wv = pack_sr_bf16x8(w, rnd);
  uint32_t o1[4], o2[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    o1[j] = dev::bf16_rne(s1[2 * j]) | (dev::bf16_rne(s1[2 * j + 1]) << 16);
    o2[j] = dev::bf16_rne(s2[2 * j]) | (dev::bf16_rne(s2[2 * j + 1]) << 16);
  }
  if (uses_s1(KIND))
    *reinterpret_cast<uint4*>(buf + kOffS1 + sw64(r, sub)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  if (uses_s2(KIND))
    *reinterpret_cast<uint4*>(buf + kOffS2 + sw64(r, sub)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
}

// INT8 states: a chunk is 128 rows x 64 columns (codes 8 KiB per state in
// shared memory); this thread owns 16 columns (a quarter) of row r, its 16
// bf16 weights in registers (`wv`).  The new block absmax of a 64-column block
// combines the four quarters through shared memory, of a 32-column block the
// two quarters it spans; blocks of 128 or 256 columns span several chunks and
// arrive found already (wide1, wide2: int8_wide_absmax).  The weights use the
// new float32 moments, then the moments are quantised with the new absmax.
// CMP (compact layout): the exchange region is the start of the weight region,
// free only once every compute thread has taken its weights into registers
// (a barrier before the exchange) and until the first weights are written
// back (a barrier after it).
template <int KIND, bool SCALE, bool CMP = false>
__device__ __forceinline__ void epi_chunk_int8(uint32_t taddr, uint8_t* buf, int r, int sub,
                                               int64_t e0, uint4 (&wv)[2], float a1, float a2,
                                               float* n1_out, float* n2_out, int nthreads,
                                               int qb, float wide1, float wide2,
                                               const GemmParams& p) {
  constexpr int kOffS1 = 0, kOffS2 = 8192, kOffAmax = 16384;
  float m[16], v[16];  // the new moments stay live until the block absmax is known
  uint32_t gr[16];
  ptx::tmem_ld_issue(taddr, gr);  // the gradient arrives while the codes are read
  const uint4 c1 = uses_s1(KIND) ? *reinterpret_cast<const uint4*>(buf + kOffS1 + sw64(r, sub))
                                 : make_uint4(0, 0, 0, 0);
  const uint4 c2 = uses_s2(KIND) ? *reinterpret_cast<const uint4*>(buf + kOffS2 + sw64(r, sub))
                                 : make_uint4(0, 0, 0, 0);
  const uint32_t q1[4] = {c1.x, c1.y, c1.z, c1.w}, q2[4] = {c2.x, c2.y, c2.z, c2.w};
  const float sd1 = dev::dvd(a1, 127.f), sd2 = dev::dvd(a2, 255.f);  // old code steps
  float n1 = 0.f, n2 = 0.f;
  // the rounding bits of the 16 weights, ahead of the gradient wait
  const uint64_t grp = (static_cast<uint64_t>(e0) >> 3) + p.sr_base;
  const uint4 rnd0 = dev::sr_words_rk(grp, p.step, p.round_keys);
  const uint4 rnd1 = dev::sr_words_rk(grp + 1, p.step, p.round_keys);
  ptx::tmem_wait_ld(gr);
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // two halves of 8 columns: gradient and weights
    float g[8], w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = __uint_as_float(gr[8 * h + i]);
    if (SCALE) scale_grad(g, p);
    unpack_bf16x8(wv[h], w);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 8 * h + i;
      m[j] = uses_s1(KIND) ? dev::mul(dev::code_f32<true>(q1[j >> 2], j & 3), sd1) : 0.f;
      v[j] = uses_s2(KIND) ? dev::mul(dev::code_f32<false>(q2[j >> 2], j & 3), sd2) : 0.f;
      dev::rule<KIND>(w[i], g[i], m[j], v[j], p.sc);
      if (uses_s1(KIND)) n1 = fmaxf(n1, fabsf(m[j]));  // = absmax_acc: n1 is never NaN
      if (uses_s2(KIND)) n2 = fmaxf(n2, fabsf(v[j]));
    }
    wv[h] = pack_sr_bf16x8(w, h == 0 ? rnd0 : rnd1);
  }
  if (qb > 64) {  // the block spans chunks: its absmax was found ahead
    n1 = wide1;
    n2 = wide2;
  } else {
    float* amax = reinterpret_cast<float*>(buf + kOffAmax);  // [state][quarter][row]
    if (CMP) ptx::bar_sync(kEpiInnerBarrier, nthreads);  // every thread's weights are read
    amax[(0 * 4 + sub) * 128 + r] = n1;
    amax[(1 * 4 + sub) * 128 + r] = n2;
    ptx::bar_sync(kEpiInnerBarrier, nthreads);
    const int o0 = qb == 32 ? (sub & 2) : 0, on = qb == 32 ? 2 : 4;  // quarters of the block
#pragma unroll 1
    for (int o = o0; o < o0 + on; ++o) {
      n1 = fmaxf(n1, amax[(0 * 4 + o) * 128 + r]);
      n2 = fmaxf(n2, amax[(1 * 4 + o) * 128 + r]);
    }
    if (CMP) ptx::bar_sync(kEpiInnerBarrier, nthreads);  // read by all before weights return
  }
  // New codes (dev::quant_recip's rule): round x * (1/s) with the shifter;
  // the few near a half-integer or not finite, and every code of a block
  // whose reciprocal is not finite, are redone from the exact quotient x / s
  // (a branch that is rarely taken).
  uint32_t o1[4] = {0u, 0u, 0u, 0u}, o2[4] = {0u, 0u, 0u, 0u};
  const float st1 = dev::dvd(n1, 127.f), st2 = dev::dvd(n2, 255.f);  // code steps
  const float iv1 = dev::dvd(1.f, st1), iv2 = dev::dvd(1.f, st2);
  const bool bad1 = !(fabsf(iv1) <= 3.0e38f), bad2 = !(fabsf(iv2) <= 3.0e38f);
  // The sixteen codes are formed branch-free; if any lies near a rounding
  // boundary (rare) all sixteen are formed again from the exact quotient,
  // which gives the others' codes unchanged.
  auto codes = [&](const float (&x)[16], float st, float inv, bool bad, uint32_t (&o)[4], auto sgn) {
    constexpr bool S = decltype(sgn)::value;
    uint32_t k[16];  // the low byte of each is the code
    bool any = bad;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      bool nr;
      k[i] = dev::code_round_fast<S>(dev::mul(x[i], inv), nr);
      any |= nr;
    }
    if (any) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        bool nr;
        k[i] = static_cast<uint32_t>(dev::code_round<S>(dev::dvd(x[i], st), nr));
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)  // four codes per word, byte i = code 4q + i
      o[q] = __byte_perm(__byte_perm(k[4 * q], k[4 * q + 1], 0x0040u),
                         __byte_perm(k[4 * q + 2], k[4 * q + 3], 0x0040u), 0x5410u);
  };
  if (uses_s1(KIND)) codes(m, st1, iv1, bad1, o1, std::true_type{});
  if (uses_s2(KIND)) codes(v, st2, iv2, bad2, o2, std::false_type{});
  if (n1 == 0.f) o1[0] = o1[1] = o1[2] = o1[3] = 0u;  // a zero block keeps zero codes
  if (n2 == 0.f) o2[0] = o2[1] = o2[2] = o2[3] = 0u;
  if (uses_s1(KIND))
    *reinterpret_cast<uint4*>(buf + kOffS1 + sw64(r, sub)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  if (uses_s2(KIND))
    *reinterpret_cast<uint4*>(buf + kOffS2 + sw64(r, sub)) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  *n1_out = n1;
  *n2_out = n2;
}

// INT8 states with blocks wider than a chunk (qb = 128 or 256 columns): the
// new absmax of each block of this thread's row in the unit (a pair tile's
// 256 columns, or a 128-column half), found before its chunks are quantised.
// The thread forms the new moments of its 16 columns of each of the unit's
// `nch` chunks with the arithmetic of epi_chunk_int8, reading the old codes,
// scales and (for rules whose moments depend on the weights) weights straight
// from global memory, all still unchanged; the four column quarters of a row
// then combine their maxima in shared memory (`amax`, 1024 floats of the
// chunk's buffer).  The results go to the first 512 floats of both buffers'
// regions (`amax` and `amax_other`), [state][block b of the unit][row]: two
// blocks of 128 in a whole unit, else one.
template <int KIND, bool SCALE>
__device__ __forceinline__ void int8_wide_absmax(uint32_t tunit, int64_t row, int col0, int nch, int r,
                                                 int sub, int qs, float* amax, float* amax_other,
                                                 int nthreads, const GemmParams& p) {
  const int64_t K = p.Ncols;
  const bool need_w = (KIND != kAdamW && KIND != kLion) && p.sc.l2 != 0.f;
  float l1a = 0.f, l1b = 0.f, l2a = 0.f, l2b = 0.f;  // blocks 0 and 1 of the unit
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    const int col = col0 + c * 64 + sub * 16;
    uint32_t gr[16];
    ptx::tmem_ld_issue(tunit + static_cast<uint32_t>(c * 64 + sub * 16), gr);
    uint4 q1 = make_uint4(0, 0, 0, 0), q2 = make_uint4(0, 0, 0, 0), w0 = q1, w1 = q1;
    float a1 = 0.f, a2 = 0.f;
    if (row < p.M && col < K) {
      const int64_t e0 = row * K + col, sidx = row * (K >> qs) + (col >> qs);
      if (uses_s1(KIND)) {
        q1 = *reinterpret_cast<const uint4*>(static_cast<const int8_t*>(p.s1) + e0);
        a1 = p.s1_scale[sidx];
      }
      if (uses_s2(KIND)) {
        q2 = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.s2) + e0);
        a2 = p.s2_scale[sidx];
      }
      if (need_w) {
        w0 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.W) + e0);
        w1 = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.W) + e0 + 8);
      }
    }
    ptx::tmem_wait_ld(gr);
    const uint32_t c1[4] = {q1.x, q1.y, q1.z, q1.w}, c2[4] = {q2.x, q2.y, q2.z, q2.w};
    const float sd1 = dev::dvd(a1, 127.f), sd2 = dev::dvd(a2, 255.f);
    float n1 = 0.f, n2 = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float g[8], w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = __uint_as_float(gr[8 * h + i]);
      if (SCALE) scale_grad(g, p);
      unpack_bf16x8(h == 0 ? w0 : w1, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = 8 * h + i;
        float m = uses_s1(KIND) ? dev::mul(dev::code_f32<true>(c1[j >> 2], j & 3), sd1) : 0.f;
        float v = uses_s2(KIND) ? dev::mul(dev::code_f32<false>(c2[j >> 2], j & 3), sd2) : 0.f;
        dev::rule<KIND>(w[i], g[i], m, v, p.sc);
        if (uses_s1(KIND)) n1 = fmaxf(n1, fabsf(m));
        if (uses_s2(KIND)) n2 = fmaxf(n2, fabsf(v));
      }
    }
    const bool second = ((c * 64) >> qs) != 0;  // the unit's block this chunk lies in: 0 or 1
    if (second) {
      l1b = fmaxf(l1b, n1);
      l2b = fmaxf(l2b, n2);
    } else {
      l1a = fmaxf(l1a, n1);
      l2a = fmaxf(l2a, n2);
    }
  }
  const int nblk = ((nch * 64) >> qs) > 1 ? 2 : 1;
  float f1a = 0.f, f1b = 0.f, f2a = 0.f, f2b = 0.f;
#pragma unroll 1
  for (int b = 0; b < nblk; ++b) {
    amax[(0 * 4 + sub) * 128 + r] = b == 0 ? l1a : l1b;
    amax[(1 * 4 + sub) * 128 + r] = b == 0 ? l2a : l2b;
    ptx::bar_sync(kEpiInnerBarrier, nthreads);
    float m1 = 0.f, m2 = 0.f;
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      m1 = fmaxf(m1, amax[(0 * 4 + o) * 128 + r]);
      m2 = fmaxf(m2, amax[(1 * 4 + o) * 128 + r]);
    }
    ptx::bar_sync(kEpiInnerBarrier, nthreads);  // read by all before the region is written again
    if (b == 0) {
      f1a = m1;
      f2a = m2;
    } else {
      f1b = m1;
      f2b = m2;
    }
  }
  if (sub == 0) {  // one quarter publishes its row's results in both buffers
    float* dst[2] = {amax, amax_other};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      dst[i][(0 * 2 + 0) * 128 + r] = f1a;
      dst[i][(0 * 2 + 1) * 128 + r] = f1b;
      dst[i][(1 * 2 + 0) * 128 + r] = f2a;
      dst[i][(1 * 2 + 1) * 128 + r] = f2b;
    }
  }
  ptx::bar_sync(kEpiInnerBarrier, nthreads);  // published before any quarter reads them
}

// Chunk geometry of the staged FORGE epilogue for one state dtype.  A chunk
// is 128 rows x kCC columns of the CTA's 128 x 256 half of a pair tile:
// fp32 states 32 columns (m and v 16 KiB each in shared memory), bf16 states
// 32 columns (8 KiB each), INT8 states 64 columns (one code block per row;
// 8 KiB of codes per state).
template <int KIND, int SDT>
struct StagedGeom {
  static constexpr bool U1 = uses_s1(KIND), U2 = uses_s2(KIND);
  static constexpr bool I8 = (SDT == kSInt8 || SDT == kSInt8W || SDT == kSInt8X || SDT == kSInt8WX);
  // INT8 block width: the method's 64, compiled in, or (0) read from the
  // parameters (32, 128 or 256)
  static constexpr int QB = (SDT == kSInt8 || SDT == kSInt8W) ? 64 : 0;
  static constexpr bool BF = (SDT == kSBf16);
  static constexpr int kCC = I8 ? 64 : 32;
  static constexpr int kChunks = kTileN / kCC;
  static constexpr int kOffS1 = 0;
  static constexpr int kOffS2 = (I8 || BF) ? 8192 : 16384;
  static constexpr uint32_t kStateBytes = (I8 || BF) ? 8192u : 16384u;
  static constexpr uint32_t kTx = (U1 ? kStateBytes : 0u) + (U2 ? kStateBytes : 0u);
  static constexpr int kWPerThread = kCC / 4;  // bf16 weights per thread and chunk (8 or 16)
  // kSInt8W, kSInt8WX: the chunk's bf16 weights (128 rows x 128 bytes,
  // 128-byte swizzle) are staged by TMA as well.  With INT8 states the old
  // scales of the next chunk are handed from the quarter that loads them to
  // the other three (kOffOld), and the block absmax is exchanged at kOffAmax;
  // except in the compact layout (kSInt8W: CMP), where the weights follow the
  // codes at 16384, the absmax exchange uses the weight region once every
  // compute thread holds its weights in registers, and each thread loads its
  // own old scale.
  static constexpr bool WST = stages_weights(SDT);
  static constexpr bool CMP = compact_int8(SDT);
  static constexpr int kOffAmax = 16384, kOffOld = 20480, kOffW = CMP ? 16384 : 21504;
  static constexpr int kBuf = WST && !CMP ? kEpiBufBytesW : kEpiBufBytes;
  static constexpr uint32_t kTxAll = kTx + (WST ? 16384u : 0u);
  static constexpr int kNC = 32 * kNumEpiWarpsStaged;  // compute threads
  static constexpr int kNB = kNC + 32;                 // compute threads + the I/O warp
};

// The pair's tiles in order, and the origin of each in this CTA: its first W
// row and first column.  The origins of the tile in hand and of the next one
// are kept, found once per tile (tile_coords divides): chunk j and the chunk
// j + 1 prefetched ahead of it always lie in one of the two.
// Units are whole tiles (kChunks chunks) or, for a pair's last unit only,
// 128-column halves (kChunks / 2 chunks): chunk j belongs to unit j / kChunks,
// and `total` counts the pair's chunks.
template <int kChunks>
struct TileWalk {
  int cur_tile = 0, cur_row0 = 0, cur_col0 = 0, nxt_row0 = 0, nxt_col0 = 0;
  int my_tiles = 0, total = 0;
  __device__ __forceinline__ void origin(int i, const GemmParams& p, uint32_t rank, int& row0,
                                         int& col0) const {
    int tm, tn, half;
    unit_coords(pair_id() + i * num_pairs(), p, tm, tn, half);
    row0 = tm * kPairM + static_cast<int>(rank) * kTileM;
    col0 = tn * kTileN + (half > 0 ? kTileN / 2 : 0);
  }
  __device__ __forceinline__ void init(const GemmParams& p, uint32_t rank) {
    my_tiles = p.num_units > pair_id() ? (p.num_units - 1 - pair_id()) / num_pairs() + 1 : 0;
    total = my_tiles * kChunks;
    if (my_tiles > 0 && pair_id() + (my_tiles - 1) * num_pairs() >= p.split_from) total -= kChunks / 2;
    if (my_tiles > 0) origin(0, p, rank, cur_row0, cur_col0);
    if (my_tiles > 1) origin(1, p, rank, nxt_row0, nxt_col0);
  }
  // Tile `local` (> 0) becomes the one in hand.
  __device__ __forceinline__ void advance(int local, const GemmParams& p, uint32_t rank) {
    cur_tile = local;
    cur_row0 = nxt_row0;
    cur_col0 = nxt_col0;
    if (local + 1 < my_tiles) origin(local + 1, p, rank, nxt_row0, nxt_col0);
  }
  __device__ __forceinline__ void where(int j, int kCC, int& row0, int& col0) const {
    const bool next = (j / kChunks) != cur_tile;
    row0 = next ? nxt_row0 : cur_row0;
    col0 = (next ? nxt_col0 : cur_col0) + (j % kChunks) * kCC;
  }
};

// Bounded wait until a grid-wide counter reaches `target` (acquire).  False if
// the CTA is aborting or the wait expired (the expiry is recorded).
__device__ __forceinline__ bool bounded_wait_count(const uint32_t* cnt, uint32_t target,
                                                   const GemmParams& p, SharedState* ss) {
  if (ptx::ld_acquire_gpu(cnt) >= target) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  while (true) {
    __nanosleep(256);
    if (ptx::ld_acquire_gpu(cnt) >= target) return true;
    if (*reinterpret_cast<volatile int32_t*>(&ss->abort)) return false;
    if (ptx::global_timer_ns() - t0 > p.wait_limit_ns) {
      *reinterpret_cast<volatile int32_t*>(&ss->abort) = 1;
      atomicCAS(p.status, 0u, static_cast<uint32_t>(kStatusTimeout));
      return false;
    }
  }
}

// The one-launch step's residency gate, passed by each CTA's I/O thread before
// its first weight tile: no weight or state of the launch is written unless
// every CTA of the launch is running (a dW tile waits for dX tiles of other
// pairs, which a pair that never started would never finish).  Each CTA adds
// one to `started` (dx_done[tiles_n]) when it starts; the first thread to see
// all of them there writes the decision "go" (1) to dx_done[tiles_n + 1], the
// first whose wait expires writes "stop" (2); one compare-and-swap settles it,
// so every CTA of the launch acts on the same decision.  On "stop" the launch
// ends with a timeout in the status word and W, the states and the scales as
// they were (only dX, an output, was written).
__device__ __forceinline__ bool residency_gate(const GemmParams& p, SharedState* ss) {
  const uint32_t* started = p.dx_done + p.tiles_n;
  uint32_t* decision = p.dx_done + p.tiles_n + 1;
  const uint64_t t0 = ptx::global_timer_ns();
  while (true) {
    const uint32_t d = ptx::ld_acquire_gpu(decision);
    if (d == 1u) return true;
    if (d == 2u) {
      *reinterpret_cast<volatile int32_t*>(&ss->abort) = 1;
      atomicCAS(p.status, 0u, static_cast<uint32_t>(kStatusTimeout));
      return false;
    }
    if (ptx::ld_acquire_gpu(started) >= gridDim.x) {
      atomicCAS(decision, 0u, 1u);
    } else if (*reinterpret_cast<volatile int32_t*>(&ss->abort)) {
      return false;
    } else if (ptx::global_timer_ns() - t0 > p.wait_limit_ns) {
      atomicCAS(decision, 0u, 2u);
    } else {
      __nanosleep(256);
    }
  }
}

// One dX tile of the one-launch step, by a compute warp: 64 columns
// (sub*64..) of TMEM lane row r, rounded to bf16 (nearest even) and written
// to row r of `box`, a 128-row x 64-column bf16 box in shared memory laid out
// with the 128-byte swizzle, from where the I/O thread stores it with TMA.
__device__ __forceinline__ void epi_dx_stage(uint32_t taddr, uint8_t* box, int r) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float g[32];
    ptx::tmem_ld_32x32b_x32(taddr + c * 32, g);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(g[8 * q + 2 * j], g[8 * q + 2 * j + 1]);
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(box + sw128(r, 4 * c + q)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// The I/O warp of the FORGE epilogue (bf16 weights).  Its lane 0 moves the
// optimizer states: before the compute warps start chunk j it waits for the
// accumulator (first chunk of a tile) and for chunk j's staged states; while
// they work on chunk j it waits until the bulk stores of chunk j-1 have read
// their buffer and issues the TMA loads of chunk j+1 into it; after they have
// written chunk j back to shared memory it issues chunk j's TMA stores.  None
// of its waits sits between two chunks of the compute warps.  In the
// one-launch step (STEP) the pair's dX tiles come first: for each it waits
// for the accumulator, then counts the tile done in its column block (its
// MMAs, and so its reads of the weights, are complete); before a dW tile's
// first chunk it waits until all dX tiles of the tile's column block are
// counted, so no weight is written while a dX tile may still read it.
template <int KIND, int SDT, int MODE>
__device__ void epilogue_io_role(const CUtensorMap* mS1, const CUtensorMap* mS2,
                                 const CUtensorMap* mDX, const CUtensorMap* mW, const GemmParams& p,
                                 SharedState* ss, uint8_t* epi, int lane, uint32_t rank) {
  using G = StagedGeom<KIND, SDT>;
  constexpr bool STEP = MODE == kModeStep;
  TileWalk<G::kChunks> walk;
  walk.init(p, rank);
  const int total = walk.total;
  const bool io = (lane == 0);
  // Weight/state lines are touched once per step: evict-first in L2, so they
  // do not displace the operand tiles the main loop re-reads from L2.
  const uint64_t pol = evict_first_policy();
  auto issue = [&](int j) {
    int row0, col0;
    walk.where(j, G::kCC, row0, col0);
    uint8_t* buf = epi + (j & 1) * G::kBuf;
    uint64_t* bar = &ss->epi_full[j & 1];
    ptx::mbar_arrive_expect_tx(bar, G::kTxAll);
    if (G::U1) ptx::tma_load_2d_hint(mS1, bar, buf + G::kOffS1, col0, row0, pol);
    if (G::U2) ptx::tma_load_2d_hint(mS2, bar, buf + G::kOffS2, col0, row0, pol);
    if (G::WST) ptx::tma_load_2d_hint(mW, bar, buf + G::kOffW, col0, row0, pol);
  };
  auto store_at = [&](int j, int row0, int col0) {
    const uint8_t* buf = epi + (j & 1) * G::kBuf;
    if (G::U1) ptx::tma_store_2d_hint(mS1, buf + G::kOffS1, col0, row0, pol);
    if (G::U2) ptx::tma_store_2d_hint(mS2, buf + G::kOffS2, col0, row0, pol);
    if (G::WST) ptx::tma_store_2d_hint(mW, buf + G::kOffW, col0, row0, pol);
    ptx::bulk_commit_group();
  };
  int issued = 0, consumed = 0, local = -1;
  bool aborted = false;
  if (STEP) {  // the dX tiles: staged in both epilogue buffers, stored with TMA
    const int ndx = my_dx_tiles(p);
    for (int i = 0; i < ndx; ++i) {
      ++local;
      bool ok = true;
      int tm, tn;
      dx_tile_coords(i, p, tm, tn);
      if (io) {
        ptx::bulk_wait_group_read0();  // the previous dX tile's stores have read the staging
        ok = bounded_wait(&ss->tmem_full[local & 1], (static_cast<uint32_t>(local) >> 1) & 1u, p, ss);
      }
      if (io && ok) ptx::red_release_gpu_add(p.dx_done + tn, 1u);
      if (ptx::bar_red_or(kEpiBarrier, G::kNB, !ok)) {
        aborted = true;
        break;
      }
      ptx::bar_sync(kEpiBarrier, G::kNB);  // the compute warps have staged the tile
      if (io) {
        const int row0 = tm * kPairM + static_cast<int>(rank) * kTileM;
        const int col0 = tn * kTileN;
        if (row0 < p.dx_rows) {
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (col0 + 64 * b < p.Ncols) ptx::tma_store_2d(mDX, epi + b * 16384, col0 + 64 * b, row0);
        }
        ptx::bulk_commit_group();
      }
    }
    if (io) ptx::bulk_wait_group_read0();  // the buffers are free for the weight tiles' states
  }
  const int first = local + 1;  // accumulator index of the first dW tile
  // Waits until chunk j may start: its tile's accumulator (first chunk of a
  // tile) and its staged states.  False if a wait failed.
  auto ready = [&](int j) -> bool {
    bool ok = true;
    if (j % G::kChunks == 0) {
      ++local;
      if (local > first) walk.advance(local - first, p, rank);
      if (io) ok = bounded_wait(&ss->tmem_full[local & 1], (static_cast<uint32_t>(local) >> 1) & 1u, p, ss);
      if (STEP && io && ok && local == first) ok = residency_gate(p, ss);
      if (STEP && io && ok) ok = bounded_wait_count(p.dx_done + walk.cur_col0 / kTileN, p.dx_target, p, ss);
    }
    if (io && ok) ok = bounded_wait(&ss->epi_full[j & 1], (static_cast<uint32_t>(j) >> 1) & 1u, p, ss);
    return ok;
  };
  // The barriers release the compute warps into a chunk (ordering their
  // tensor- and shared-memory reads after the waits above) or stop everyone;
  // inside a tile one barrier both ends chunk j and starts chunk j + 1.  At
  // the end of a tile the compute warps free the accumulator between two
  // barriers, so the next tile's MMAs never wait for the tile after it.
  bool stop = aborted || total == 0;
  if (!stop) {
    if (io) {
      issue(0);
      issued = 1;
      if (MODE == kModeFusedOpt) ptx::grid_dep_wait();  // before the first store
    }
    stop = ptx::bar_red_or(kEpiBarrier, G::kNB, !ready(0));
    if (!stop) consumed = 1;
  }
  for (int j = 0; j < total && !stop; ++j) {
    int srow, scol;
    walk.where(j, G::kCC, srow, scol);  // chunk j's origin, before the walk moves on
    const bool more = j + 1 < total;
    if (io && more) {
      ptx::bulk_wait_group_read0();  // chunk j-1's stores have read buffer (j+1)&1
      issue(j + 1);
      issued = j + 2;
    }
    if (more && (j + 1) % G::kChunks != 0) {
      stop = ptx::bar_red_or(kEpiBarrier, G::kNB, !ready(j + 1));
      if (io) store_at(j, srow, scol);
    } else {
      ptx::bar_sync(kEpiBarrier, G::kNB);  // chunk j is back in shared memory
      if (io) store_at(j, srow, scol);
      if (more) stop = ptx::bar_red_or(kEpiBarrier, G::kNB, !ready(j + 1));
    }
    if (!stop && more) consumed = j + 2;
  }
  if (io) {
    ptx::bulk_wait_group0();
    for (int j = consumed; j < issued; ++j)  // loads issued but not consumed (abort path)
      bounded_wait(&ss->epi_full[j & 1], (static_cast<uint32_t>(j) >> 1) & 1u, p, ss, false);
  }
}

// A compute warp of the FORGE epilogue.  Warp w reads TMEM lanes 32*(w%4)..
// (its rows) and a quarter of each chunk's columns; its weights (bf16, or fp32
// with fp32 states) and old INT8 scales come straight from global memory one
// chunk ahead, its states from the staged chunk in shared memory.
template <int KIND, int WDT, int SDT, int MODE>
__device__ void epilogue_compute_role(const GemmParams& p, SharedState* ss, uint8_t* epi,
                                      int warp, int lane, uint32_t rank) {
  using G = StagedGeom<KIND, SDT>;
  constexpr bool STEP = MODE == kModeStep, SCALE = MODE == kModeFusedFp8;
  constexpr bool F32W = WDT == kWFp32;
  constexpr int kCC = G::kCC, kChunks = G::kChunks, kWPerThread = G::kWPerThread;
  constexpr int kWV = kWPerThread * (F32W ? 4 : 2) / 16;  // 16-byte words of weights per thread and chunk
  const int quarter = warp & 3, sub = (warp - 2) >> 2;  // TMEM lane quarter, column quarter
  const int r = quarter * 32 + lane;
  const int64_t K = p.Ncols;
  TileWalk<kChunks> walk;
  walk.init(p, rank);
  const int total = walk.total;
  const uint32_t empty0 = ptx::mapa(ptx::smem_addr(&ss->tmem_empty[0]), 0);
  // INT8 block width (columns) and its base-2 logarithm
  const int qb = G::QB ? G::QB : p.qblock;
  const int qs = G::QB ? 6 : p.qshift;
  // every thread loads its own old scale (32-column blocks, compact layout),
  // or one quarter of a row loads them and hands them to the other three
  const bool own = G::CMP || qb == 32;

  // This thread's weights of chunk j (and, for INT8 states, the old absmax of
  // its code block): loaded one chunk ahead.  They are 2 of the 10 or 4.25
  // bytes per element, so they bypass the staging; plain (L1-allocating)
  // loads let the four warps that own the 64 bytes of a row's chunk share one
  // L1 fill instead of four L2 requests.
  auto prefetch = [&](int j, uint4 (&v)[kWV], float& o1, float& o2) {
    int row0, col0;
    walk.where(j, kCC, row0, col0);
    const int64_t row = static_cast<int64_t>(row0) + r;
    const int col = col0 + sub * kWPerThread;
    const bool ok = row < p.M && col < K;
    if (!G::WST) {
      const uint8_t* q = static_cast<const uint8_t*>(p.W) + (row * K + col) * (F32W ? 4 : 2);
#pragma unroll
      for (int h = 0; h < kWV; ++h)
        v[h] = ok ? *reinterpret_cast<const uint4*>(q + 16 * h) : make_uint4(0, 0, 0, 0);
    }
    // the old scale of this thread's code block; blocks of 64 or more
    // columns are whole in a quarter's row of the chunk, so after the first
    // chunk one quarter loads a row's old scales and hands them to the other
    // three, unless every thread loads its own (`own`)
    if (G::I8 && (j == 0 || sub == 0 || own)) {
      const bool okb = row < p.M && col < K;
      const int64_t sidx = row * (K >> qs) + (col >> qs);
      if (G::U1) o1 = okb ? p.s1_scale[sidx] : 0.f;
      if (G::U2) o2 = okb ? p.s2_scale[sidx] : 0.f;
    }
  };
  uint4 wnext[kWV];
  float o1next = 0.f, o2next = 0.f;  // old INT8 scales of the next chunk
  int local = -1;
  if (STEP) {  // the pair's dX tiles: 64 columns per warp into the staging boxes
    const int ndx = my_dx_tiles(p);
    for (int i = 0; i < ndx; ++i) {
      ++local;
      if (ptx::bar_red_or(kEpiBarrier, G::kNB, false)) return;  // the I/O warp's verdict
      ptx::tc_fence_after();
      const int acc = local & 1;
      const uint32_t taddr = ss->tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * kTileN + sub * 64);
      epi_dx_stage(taddr, epi + sub * 16384, r);
      ptx::fence_proxy_async_smem();  // the staged values, visible to the TMA store
      ptx::tc_fence_before();
      ptx::bar_sync(kEpiBarrier, G::kNB);
      if (lane == 0) ptx::mbar_arrive_cluster(empty0 + static_cast<uint32_t>(acc) * 8u);
    }
  }
  const int first = local + 1;  // accumulator index of the first dW tile
  auto begin = [&](int j) {  // chunk j is about to start: the walk follows its tile
    if (j % kChunks == 0) {
      ++local;
      if (local > first) walk.advance(local - first, p, rank);
    }
  };
  bool stop = total == 0;
  if (!stop) {
    prefetch(0, wnext, o1next, o2next);
    if (MODE == kModeFusedOpt) ptx::grid_dep_wait();  // before the first write
    begin(0);
    stop = ptx::bar_red_or(kEpiBarrier, G::kNB, false);  // the I/O warp's verdict
  }
  for (int j = 0; j < total && !stop; ++j) {
    const int c = j % kChunks;
    int row0, col0;
    walk.where(j, kCC, row0, col0);
    const int64_t row = static_cast<int64_t>(row0) + r;
    uint4 wcur[kWV];
    uint8_t* buf = epi + (j & 1) * G::kBuf;
    float o1 = o1next, o2 = o2next;
    if (G::WST) {  // staged weights; old scales from the quarter that loaded them
#pragma unroll
      for (int h = 0; h < kWPerThread / 8; ++h)
        wcur[h] = *reinterpret_cast<const uint4*>(buf + G::kOffW + sw128(r, 2 * sub + h));
      if (j > 0 && !own) {
        const float* old = reinterpret_cast<const float*>(buf + G::kOffOld);
        o1 = old[r];
        o2 = old[128 + r];
      }
      if (j + 1 < total && (sub == 0 || own)) prefetch(j + 1, wnext, o1next, o2next);
    } else {
#pragma unroll
      for (int h = 0; h < kWV; ++h) wcur[h] = wnext[h];
      if (G::I8 && j > 0 && !own) {  // old scales from the quarter that loaded them
        const float* old = reinterpret_cast<const float*>(buf + G::kOffOld);
        o1 = old[r];
        o2 = old[128 + r];
      }
      if (j + 1 < total) prefetch(j + 1, wnext, o1next, o2next);
    }
    ptx::tc_fence_after();
    const int acc = local & 1;
    const int col = col0 + sub * kWPerThread;
    const uint32_t taddr = ss->tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(acc * kTileN + c * kCC + sub * kWPerThread);
    const int64_t e0 = row * K + col;
    float n1 = 0.f, n2 = 0.f;  // INT8: the new absmax of this thread's block
    if (G::I8) {
      float wd1 = 0.f, wd2 = 0.f;  // blocks of 128 or 256 columns: their absmax, found ahead
      if (!G::QB && qb > 64) {
        if (c == 0) {  // a new unit
          const uint32_t tunit = ss->tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(acc * kTileN);
          int8_wide_absmax<KIND, SCALE>(tunit, row, col0, min(kChunks, total - j), r, sub, qs,
                                        reinterpret_cast<float*>(buf + G::kOffAmax),
                                        reinterpret_cast<float*>(epi + ((j + 1) & 1) * G::kBuf + G::kOffAmax),
                                        G::kNC, p);
        }
        const float* fin = reinterpret_cast<const float*>(buf + G::kOffAmax);
        const int wb = (c * kCC) >> qs;
        wd1 = fin[(0 * 2 + wb) * 128 + r];
        wd2 = fin[(1 * 2 + wb) * 128 + r];
      }
      epi_chunk_int8<KIND, SCALE, G::CMP>(taddr, buf, r, sub, e0, *reinterpret_cast<uint4(*)[2]>(wcur), o1,
                                          o2, &n1, &n2, G::kNC, qb, wd1, wd2, p);
    } else if (G::BF) {
      epi_chunk_bf16s<KIND, SCALE>(taddr, buf, r, sub, e0, wcur[0], p);
    } else {
      if constexpr (F32W)
        epi_chunk_fp32w<KIND>(taddr, buf, r, sub, *reinterpret_cast<uint4(*)[2]>(wcur), p);
      else
        epi_chunk_fp32<KIND, SCALE>(taddr, buf, r, sub, e0, wcur[0], p);
    }
    if (G::WST) {  // back to the staged chunk (TMA-stored); the next chunk's old scales
#pragma unroll
      for (int h = 0; h < kWPerThread / 8; ++h)
        *reinterpret_cast<uint4*>(buf + G::kOffW + sw128(r, 2 * sub + h)) = wcur[h];
      if (G::I8 && j + 1 < total && sub == 0 && !own) {
        float* nold = reinterpret_cast<float*>(epi + ((j + 1) & 1) * G::kBuf + G::kOffOld);
        nold[r] = o1next;
        nold[128 + r] = o2next;
      }
    } else {
      if (G::I8 && j + 1 < total && sub == 0 && !own) {  // the next chunk's old scales, for all quarters
        float* nold = reinterpret_cast<float*>(epi + ((j + 1) & 1) * G::kBuf + G::kOffOld);
        nold[r] = o1next;
        nold[128 + r] = o2next;
      }
    }
    const bool more = j + 1 < total;
    const bool unit_end = !more || c == kChunks - 1;  // the unit's accumulator is read out
    if (unit_end) ptx::tc_fence_before();
    // The staged states, visible to the TMA stores.  The global stores below
    // come after this fence, so that it has no global write in flight to
    // wait for: they are ordered by nothing in this CTA.
    ptx::fence_proxy_async_smem();
    if (!G::WST && row < p.M && col < K) {
      uint8_t* q = static_cast<uint8_t*>(p.W) + e0 * (F32W ? 4 : 2);
#pragma unroll
      for (int h = 0; h < kWV; ++h) *reinterpret_cast<uint4*>(q + 16 * h) = wcur[h];
    }
    // INT8: the thread with the block's last 16 columns stores the block's
    // new absmax; a block wider than a chunk keeps its old one until its last
    // chunk has read it (the next chunks' old scales are loaded a chunk ahead)
    if (G::I8 && (col & (qb - 1)) == qb - 16 && row < p.M && col < K) {
      const int64_t sidx = row * (K >> qs) + (col >> qs);
      if (G::U1) p.s1_scale[sidx] = n1;
      if (G::U2) p.s2_scale[sidx] = n2;
    }
    if (!unit_end) {  // end of chunk j = start of chunk j + 1 (same unit)
      begin(j + 1);
      stop = ptx::bar_red_or(kEpiBarrier, G::kNB, false);
    } else {
      ptx::bar_sync(kEpiBarrier, G::kNB);
      if (lane == 0) ptx::mbar_arrive_cluster(empty0 + static_cast<uint32_t>(acc) * 8u);
      if (more) {
        begin(j + 1);
        stop = ptx::bar_red_or(kEpiBarrier, G::kNB, false);
      }
    }
  }
}

template <int KIND, int WDT, int SDT, int MODE>
__device__ __forceinline__ void epilogue_staged(const CUtensorMap* mS1, const CUtensorMap* mS2,
                                                const CUtensorMap* mDX, const CUtensorMap* mW,
                                                const GemmParams& p,
                                                SharedState* ss, uint8_t* epi, int warp, int lane,
                                                uint32_t rank) {
  if (warp == 2 + kNumEpiWarpsStaged)
    epilogue_io_role<KIND, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, lane, rank);
  else
    epilogue_compute_role<KIND, WDT, SDT, MODE>(p, ss, epi, warp, lane, rank);
}

template <int WDT, int SDT, int MODE>
__device__ __forceinline__ void epilogue_tma_dispatch(const CUtensorMap* mS1, const CUtensorMap* mS2,
                                                      const CUtensorMap* mDX, const CUtensorMap* mW,
                                                      const GemmParams& p,
                                                      SharedState* ss, uint8_t* epi, int warp,
                                                      int lane, uint32_t rank) {
  switch (p.sc.kind) {
    case kAdamW: epilogue_staged<kAdamW, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    case kNAdam: epilogue_staged<kNAdam, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    case kRAdam: epilogue_staged<kRAdam, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    case kLion: epilogue_staged<kLion, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    case kRMSprop: epilogue_staged<kRMSprop, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    case kAdaGrad: epilogue_staged<kAdaGrad, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    case kSGD: epilogue_staged<kSGD, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
    default: epilogue_staged<kSGDMomentum, WDT, SDT, MODE>(mS1, mS2, mDX, mW, p, ss, epi, warp, lane, rank); break;
  }
}

// ------------------------------------------------------------------ kernel

template <int MODE, int WDT, int SDT>
__global__ void __launch_bounds__(KCfg<MODE, WDT, SDT>::kThreads, 1)
    tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
              const __grid_constant__ CUtensorMap mapDA, const __grid_constant__ CUtensorMap mapDB,
              const __grid_constant__ CUtensorMap mapS1,
              const __grid_constant__ CUtensorMap mapS2, const __grid_constant__ CUtensorMap mapDX,
              const __grid_constant__ CUtensorMap mapW, const GemmParams p) {
  using Cfg = KCfg<MODE, WDT, SDT>;
  constexpr int STG = Cfg::kStg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STG * Cfg::kA;
  uint8_t* epi = smB + STG * Cfg::kB;
  SharedState* ss = reinterpret_cast<SharedState*>(epi + Cfg::kEpiBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();  // 0 = leader of the pair

  if (threadIdx.x == 0) {
    for (int s = 0; s < STG; ++s) {
      ptx::mbar_init(&ss->full[s], 1);   // the leader's: armed once, both CTAs' bytes
      ptx::mbar_init(&ss->empty[s], 1);  // each CTA's: the leader's multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&ss->tmem_full[a], 1);
      ptx::mbar_init(&ss->tmem_empty[a], 2 * Cfg::kEpiWarps);  // the leader's: both CTAs' warps
      ptx::mbar_init(&ss->epi_full[a], 1);
    }
    ptx::mbar_init(&ss->mma_done, 1);
    ss->abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&mapA);
    ptx::prefetch_tensormap(&mapB);
    if (MODE == kModeStep) {
      ptx::prefetch_tensormap(&mapDA);
      ptx::prefetch_tensormap(&mapDB);
    }
  }
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_alloc_pair(&ss->tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  // Each warp reconverges before the CTA barrier (lanes of warps 0 and 1 took
  // different paths above), so the barrier counts every thread.
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other's
  ptx::tc_fence_after();
  if (MODE == kModeStep && threadIdx.x == 0) atomicAdd(p.dx_done + p.tiles_n, 1u);  // residency_gate

  if (warp == 0) {
    if (lane == 0) producer_role<MODE, STG, Cfg::kBK>(&mapA, &mapB, &mapDA, &mapDB, p, smA, smB, ss, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_role<MODE, STG, Cfg::kBK>(p, smA, smB, ss);
  } else {
    if constexpr (Cfg::kTmaEpi)
      epilogue_tma_dispatch<WDT, SDT, MODE>(&mapS1, &mapS2, &mapDX, &mapW, p, ss, epi, warp, lane, rank);
    else
      epilogue_role<MODE, WDT, SDT>(p, ss, warp, lane, rank);
  }

  // A dependent launch (after the fp32-weight dX kernel) ends only after that
  // grid, on every path (the epilogue's waits are skipped when a CTA aborts).
  if (MODE == kModeFusedOpt) ptx::grid_dep_wait();
  __syncwarp();  // the producer's and MMA thread's lanes rejoin their warps first
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's shared and tensor memory stay valid until the pair is done
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(ss->tmem_base, kTmemCols);
  }
}

// Launch on clusters of two CTAs (the tcgen05 pair); grid is a multiple of 2.
// `early`: the launch may begin before the previous kernel on the stream ends
// (programmatic stream serialisation; that kernel lets it in, and the
// epilogue's grid_dep_wait orders the writes after it).
template <typename Kernel>
inline cudaError_t launch_pair(Kernel k, int grid, int threads, int smem, cudaStream_t s,
                               const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& da,
                               const CUtensorMap& db, const CUtensorMap& s1,
                               const CUtensorMap& s2, const CUtensorMap& dx, const CUtensorMap& w,
                               const GemmParams& p, bool early = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, a, b, da, db, s1, s2, dx, w, p);
}

}  // namespace forge
