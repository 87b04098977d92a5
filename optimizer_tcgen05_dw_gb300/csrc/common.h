// Definitions shared by the host API and the kernels of libforge.
#pragma once

#include <cstdint>

namespace forge {

// Rule identifiers (values match forge_opt_kind_t).
enum OptKind : int32_t {
  kAdamW = 0, kNAdam = 1, kRAdam = 2, kLion = 3,
  kRMSprop = 4, kAdaGrad = 5, kSGD = 6, kSGDMomentum = 7
};
enum WDtype : int32_t { kWFp32 = 0, kWBf16 = 1 };
enum SDtype : int32_t { kSFp32 = 0, kSInt8 = 1, kSBf16 = 2,
                        // INT8 states with the bf16 weights staged through shared
                        // memory by TMA (kernel-side only; the host picks it for
                        // short reductions, T <= kStageWeightsMaxT)
                        kSInt8W = 3,
                        // kSInt8 / kSInt8W with the absmax block width read from
                        // the parameters (32, 128 or 256 columns); the two above
                        // are compiled for the method's block of 64
                        kSInt8X = 4, kSInt8WX = 5 };
constexpr int kNumKernelSdt = 6;
// Longest reduction for which the INT8 epilogue stages the weights: it frees
// the compute warps from row-strided weight accesses (+40 % at T = 4096); over
// longer reductions the direct form is as fast or faster (block 64 keeps all
// operand stages either way; the other block widths give one up to staging).
constexpr int64_t kStageWeightsMaxT = 8192;

// Device-side status codes (values match forge_status_t).
enum DeviceStatus : uint32_t { kStatusOk = 0, kStatusTimeout = 4 };

// Per-step scalars of a rule, formed on the host in double from the float
// hyper-parameters and the step number and rounded once to float.  Field use
// per rule (everything else is zero):
//   AdamW   decay b1 omb1 b2 omb2 step_size inv_sqrt_c2 eps
//   NAdam   l2 b1 omb1 b2 omb2 inv_c2 eps coef_g coef_m
//   RAdam   l2 b1 omb1 b2 omb2 eps; rectified ? (step_size, sqrt_c2) : step_size
//   Lion    decay lr b1 omb1 b2 omb2
//   RMSprop l2 alpha oma lr eps
//   AdaGrad l2 lr eps
//   SGD     l2 lr
//   SGD-m   l2 lr mom
struct OptScalars {
  int32_t kind;
  int32_t rectified;
  float l2, decay, lr, b1, omb1, b2, omb2, eps;
  float step_size, sqrt_c2, inv_sqrt_c2, inv_c2, coef_g, coef_m, alpha, oma, mom;
};

// Which state buffers a rule keeps.
inline constexpr bool uses_s1(int k) {
  return k == kAdamW || k == kNAdam || k == kRAdam || k == kLion || k == kSGDMomentum;
}
inline constexpr bool uses_s2(int k) {
  return k == kAdamW || k == kNAdam || k == kRAdam || k == kRMSprop || k == kAdaGrad;
}

// Tensor-core GEMM geometry: a CTA pair computes a 256 x 256 output tile
// (each CTA 128 x 256: two 128 x 128 optimizer tiles side by side) in
// 64-token stages; a stage holds this CTA's 128 rows of A and 128 of B's
// 256 columns (32 KiB).  Plain modes keep a 6-stage ring (192 KiB); the FORGE
// step with bf16 weights keeps five stages (160 KiB) next to the 64 KiB of
// staged optimizer-state buffers.
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kBlockK = 64;
constexpr int kStages = 6;
#ifndef FORGE_FUSED_BK
#define FORGE_FUSED_BK 64
#endif
#ifndef FORGE_FUSED_STAGES
#define FORGE_FUSED_STAGES 5
#endif
#ifndef FORGE_WGRAD_BK
#define FORGE_WGRAD_BK 64
#endif
#ifndef FORGE_WGRAD_STAGES
#define FORGE_WGRAD_STAGES 6
#endif
constexpr int kFusedBlockK = FORGE_FUSED_BK;
constexpr int kWgradBlockK = FORGE_WGRAD_BK;      // unfused weight-gradient pass
constexpr int kFp8BlockK = 128;                   // tokens per stage with E4M3 operands (128-byte rows)
constexpr int kWgradStages = FORGE_WGRAD_STAGES;
constexpr int kFusedStages = FORGE_FUSED_STAGES;
constexpr int kNumEpiWarps = 8;                          // epilogue warps, plain epilogues
constexpr int kNumEpiWarpsStaged = 16;                   // epilogue warps, staged FORGE epilogue
constexpr int kTmemCols = 2 * kTileN;                    // double-buffered fp32 accumulator

enum GemmMode : int32_t {
  kModeFusedOpt = 0,   // dW tile -> optimizer epilogue (the FORGE step)
  kModeWgradStore = 1, // dW tile -> fp32 store (unfused pass 1)
  kModeDgrad = 2,      // dX tile -> bf16 store
  kModeStep = 3,       // one launch: the dX tiles, then the dW tiles -> optimizer epilogue
  kModeFusedFp8 = 4    // the FORGE step from E4M3 operands (token-contiguous, scaled)
};

// Column blocks (of kTileN) whose dX-completion counters the one-launch step
// keeps in device memory: K up to 1M.
constexpr int kMaxDxBlocks = 4096;

// Parameters of one tensor-core launch.  Output tile space is M x Ncols
// (wgrad: M = N_out rows of W, Ncols = K; dgrad: M = T, Ncols = K).
struct GemmParams {
  int32_t M, Ncols;
  int32_t num_kb;            // reduction blocks of 64
  int32_t tiles_m, tiles_n, num_tiles;
  // Work units of the weight tiles: tiles 0 .. split_from-1 whole, then each
  // remaining tile as two 128-column halves (units split_from ..
  // num_units-1), so that a last partial wave of pair tiles becomes half as
  // long, or (split_from == 0) a small layer's tiles spread over twice the
  // pairs.  A pair holds at most one half unit, its last.  split_from ==
  // num_tiles == num_units when nothing is split.
  int32_t num_units, split_from;
  void* out;                 // wgrad store: fp32 [M x Ncols]; dgrad: bf16 [M x Ncols]
  void* W;                   // fused: [M x Ncols] fp32 or bf16
  void* s1;
  void* s2;
  float* s1_scale;
  float* s2_scale;
  OptScalars sc;
  uint64_t seed;
  uint64_t step;
  // Added to each 8-element group's index (element index / 8) in the
  // stochastic-rounding counter: row_offset * K / 8 for a row shard of a
  // larger matrix, so a shard draws the bits of its rows in the whole matrix.
  uint64_t sr_base;
  // Philox4x32-10 round keys of `seed` (key words 0 and 1 of rounds 0..9),
  // formed once on the host for the stochastic rounding of the weights.
  uint32_t round_keys[20];
  uint64_t wait_limit_ns;
  uint32_t* status;          // device status word (first error wins)
  int32_t op3d;              // MN-major operands described as 3-D maps: one load per stage
  int32_t skip_loads;
  // kModeStep: the dX tiles (a T x Ncols output, reduction over M) that run
  // ahead of the dW tiles in the same launch.  A dW tile writes its weights
  // only after every dX tile of its column block has finished its MMAs (so
  // has read the pre-update weights): dx_done[column block] counts them, one
  // per CTA of the pair, up to dx_target.
  int32_t dx_rows;           // T
  int32_t dx_tiles_m;        // 256-row pair tiles over T
  int32_t dx_tiles;          // dx_tiles_m * tiles_n
  int32_t dx_num_kb;         // reduction blocks of 64 over M
  uint32_t* dx_done;         // [tiles_n + 2], zero at launch (+ the residency gate's words)
  uint32_t dx_target;        // 2 * dx_tiles_m
  // How the dX tiles are dealt (balancing the pairs' total work): every pair
  // takes one per round for dx_rounds rounds; the rest go round-robin to the
  // pairs from dx_heavy on, those without an extra dW tile.
  int32_t dx_rounds;
  int32_t dx_heavy;
  // kModeFusedFp8: the accumulated sum of code products times gscale
  // (= x_scale * dy_scale) is the gradient.
  float gscale;
  // INT8 states: elements per absmax block along a row (32, 64, 128 or 256;
  // the scale arrays are [M x Ncols / qblock]) and its base-2 logarithm.
  int32_t qblock, qshift;
};

}  // namespace forge
