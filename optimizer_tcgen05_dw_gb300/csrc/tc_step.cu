// Instantiations of the tensor-core kernel for the one-launch step: the dX
// tiles (dX = dY W from the weights before the update), then the FORGE
// weight-gradient + optimizer tiles, with bf16 weights.
#include "launch.h"
#include "tc_kernel.cuh"

namespace forge {

template <int SDT>
static cudaError_t run_step(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& da,
                            const CUtensorMap& db, const CUtensorMap& s1, const CUtensorMap& s2,
                            const CUtensorMap& dx, const CUtensorMap& w, const GemmParams& p, int grid,
                            cudaStream_t s) {
  auto* k = tc_kernel<kModeStep, kWBf16, SDT>;
  using Cfg = KCfg<kModeStep, kWBf16, SDT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pair(k, grid, Cfg::kThreads, Cfg::kSmem, s, a, b, da, db, s1, s2, dx, w, p);
}

template <int SDT>
static int step_pairs() {
  auto* k = tc_kernel<kModeStep, kWBf16, SDT>;
  constexpr int smem = KCfg<kModeStep, kWBf16, SDT>::kSmem;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(KCfg<kModeStep, kWBf16, SDT>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) return 0;
  return n;
}

int step_max_pairs(int sdt) {
  return sdt == kSInt8     ? step_pairs<kSInt8>()
         : sdt == kSInt8W  ? step_pairs<kSInt8W>()
         : sdt == kSInt8X  ? step_pairs<kSInt8X>()
         : sdt == kSInt8WX ? step_pairs<kSInt8WX>()
         : sdt == kSBf16   ? step_pairs<kSBf16>()
                           : step_pairs<kSFp32>();
}

cudaError_t launch_tc_step(int sdt, const CUtensorMap& a, const CUtensorMap& b,
                           const CUtensorMap& da, const CUtensorMap& db, const CUtensorMap& s1,
                           const CUtensorMap& s2, const CUtensorMap& dx, const CUtensorMap& w,
                           const GemmParams& p, int grid, cudaStream_t s) {
  return sdt == kSInt8     ? run_step<kSInt8>(a, b, da, db, s1, s2, dx, w, p, grid, s)
         : sdt == kSInt8W  ? run_step<kSInt8W>(a, b, da, db, s1, s2, dx, w, p, grid, s)
         : sdt == kSInt8X  ? run_step<kSInt8X>(a, b, da, db, s1, s2, dx, w, p, grid, s)
         : sdt == kSInt8WX ? run_step<kSInt8WX>(a, b, da, db, s1, s2, dx, w, p, grid, s)
         : sdt == kSBf16   ? run_step<kSBf16>(a, b, da, db, s1, s2, dx, w, p, grid, s)
                           : run_step<kSFp32>(a, b, da, db, s1, s2, dx, w, p, grid, s);
}

}  // namespace forge
