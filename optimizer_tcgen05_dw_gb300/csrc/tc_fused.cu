// Instantiations of the tensor-core kernel for the fused FORGE step.
#include "launch.h"
#include "tc_kernel.cuh"

namespace forge {

template <int WDT, int SDT>
static cudaError_t run_fused(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bh,
                             const CUtensorMap& s1, const CUtensorMap& s2, const CUtensorMap& w,
                             const GemmParams& p, int grid, cudaStream_t s, bool after_dx) {
  auto* k = tc_kernel<kModeFusedOpt, WDT, SDT>;
  using Cfg = KCfg<kModeFusedOpt, WDT, SDT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pair(k, grid, Cfg::kThreads, Cfg::kSmem, s, a, b, a, bh, s1, s2, a, w, p, after_dx);
}

cudaError_t launch_tc_fused(int wdt, int sdt, const CUtensorMap& a, const CUtensorMap& b,
                            const CUtensorMap& bh, const CUtensorMap& s1, const CUtensorMap& s2,
                            const CUtensorMap& w, const GemmParams& p, int grid, cudaStream_t s,
                            bool after_dx) {
  const bool d = after_dx;
  if (wdt == kWBf16) {
    return sdt == kSInt8     ? run_fused<kWBf16, kSInt8>(a, b, bh, s1, s2, w, p, grid, s, d)
           : sdt == kSInt8W  ? run_fused<kWBf16, kSInt8W>(a, b, bh, s1, s2, w, p, grid, s, d)
           : sdt == kSInt8X  ? run_fused<kWBf16, kSInt8X>(a, b, bh, s1, s2, w, p, grid, s, d)
           : sdt == kSInt8WX ? run_fused<kWBf16, kSInt8WX>(a, b, bh, s1, s2, w, p, grid, s, d)
           : sdt == kSBf16   ? run_fused<kWBf16, kSBf16>(a, b, bh, s1, s2, w, p, grid, s, d)
                             : run_fused<kWBf16, kSFp32>(a, b, bh, s1, s2, w, p, grid, s, d);
  }
  return sdt == kSInt8 ? run_fused<kWFp32, kSInt8>(a, b, bh, s1, s2, w, p, grid, s, d)
                       : run_fused<kWFp32, kSFp32>(a, b, bh, s1, s2, w, p, grid, s, d);
}

}  // namespace forge
