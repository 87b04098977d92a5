// Instantiations of the tensor-core kernel for the fused FORGE step.
#include "launch.h"
#include "tc_kernel.cuh"

namespace forge {

template <int WDT, int SDT>
static cudaError_t run_fused(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& s1,
                             const CUtensorMap& s2, const GemmParams& p, int grid, cudaStream_t s) {
  auto* k = tc_kernel<kModeFusedOpt, WDT, SDT>;
  constexpr int smem = KCfg<kModeFusedOpt, WDT>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pair(k, grid, KCfg<kModeFusedOpt, WDT>::kThreads, smem, s, a, b, a, b, s1, s2, a, p);
}

cudaError_t launch_tc_fused(int wdt, int sdt, const CUtensorMap& a, const CUtensorMap& b,
                            const CUtensorMap& s1, const CUtensorMap& s2, const GemmParams& p,
                            int grid, cudaStream_t s) {
  if (wdt == kWBf16) {
    return sdt == kSInt8   ? run_fused<kWBf16, kSInt8>(a, b, s1, s2, p, grid, s)
           : sdt == kSBf16 ? run_fused<kWBf16, kSBf16>(a, b, s1, s2, p, grid, s)
                           : run_fused<kWBf16, kSFp32>(a, b, s1, s2, p, grid, s);
  }
  return sdt == kSInt8 ? run_fused<kWFp32, kSInt8>(a, b, s1, s2, p, grid, s)
                       : run_fused<kWFp32, kSFp32>(a, b, s1, s2, p, grid, s);
}

}  // namespace forge
