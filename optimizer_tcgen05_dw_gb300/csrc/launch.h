// Host-side launchers of the kernels, one per translation unit, called by the
// C ABI in api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.h"

namespace forge {

// Parameters of the elementwise (non-tensor-core) kernels.
struct ElemParams {
  const float* dW;   // optimizer step: fp32 gradient (nullptr = zero); quantise: input
  void* W;
  void* s1;
  void* s2;
  float* s1_scale;
  float* s2_scale;
  int64_t N, K;      // rows, columns
  OptScalars sc;
  uint64_t seed, step;
  uint64_t sr_base;  // added to each 8-element group's index in the rounding counter
  int32_t is_signed; // quantise / dequantise
  int32_t qblock;    // INT8 states: elements per absmax block (32, 64, 128 or 256)
};

// tc_fused.cu: the FORGE step (mode kModeFusedOpt) for one (W dtype, state dtype).
// s1, s2: tensor maps of the state tiles the bf16-weight epilogue stages
// through shared memory (unused, any valid map, for fp32 weights or for
// states the rule does not keep); w: bf16 W in 64-column x 128-row boxes
// (128-byte swizzle), staged when sdt is kSInt8W (else any valid map); bh:
// the B operand in 64-column boxes for half units (GemmParams::split_from;
// any valid map when nothing is split).
// With `after_dx` the launch may start while the fp32-weight dX kernel before
// it on the stream still runs (programmatic dependent launch); its epilogue
// waits for that grid before writing weights or states.
cudaError_t launch_tc_fused(int wdt, int sdt, const CUtensorMap& a, const CUtensorMap& b,
                            const CUtensorMap& bh, const CUtensorMap& s1, const CUtensorMap& s2,
                            const CUtensorMap& w, const GemmParams& p, int grid, cudaStream_t s,
                            bool after_dx = false);
// tc_step.cu: dX and the FORGE step in one launch (mode kModeStep, bf16
// weights): a, b the dW operands, da, db the dX operands (dY K-major, W),
// dx the dX output (bf16, 64-column x 128-row boxes, 128-byte swizzle).
cudaError_t launch_tc_step(int sdt, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& da, const CUtensorMap& db, const CUtensorMap& s1,
                           const CUtensorMap& s2, const CUtensorMap& dx, const CUtensorMap& w,
                           const GemmParams& p, int grid, cudaStream_t s);
// CTA pairs of the one-launch step that can be resident at once (its dW tiles
// wait for dX tiles of other pairs, so its grid must not exceed this); 0 if
// the query fails.
int step_max_pairs(int sdt);
// tc_fp8.cu: the FORGE step from E4M3 operands (mode kModeFusedFp8, bf16
// weights): a = dY^T codes [N x T], b = X^T codes [K x T], 128 x 128-byte
// boxes with the 128-byte swizzle; p.gscale the product of the scales.
cudaError_t launch_tc_fp8(int sdt, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bh,
                          const CUtensorMap& s1, const CUtensorMap& s2, const CUtensorMap& w,
                          const GemmParams& p, int grid, cudaStream_t s);
// tc_plain.cu: unfused pass 1 (kModeWgradStore) or dX (kModeDgrad).
cudaError_t launch_tc_plain(int mode, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int grid, cudaStream_t s);
// elementwise.cu
cudaError_t launch_opt_step(int wdt, int sdt, const ElemParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_quantize(const ElemParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_dequantize(const ElemParams& p, int num_sms, cudaStream_t s);
// dX = dY * bf16(W) for fp32 master weights (CUDA cores); its blocks let the
// next launch on the stream start early (programmatic dependent launch).
cudaError_t launch_dgrad_fp32w(const void* dY, const float* W, void* dX, int64_t T, int64_t N,
                               int64_t K, int num_sms, cudaStream_t s);

}  // namespace forge
