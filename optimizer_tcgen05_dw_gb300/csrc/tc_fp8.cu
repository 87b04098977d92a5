// Instantiations of the tensor-core kernel for the FORGE step from E4M3
// operands (bf16 weights; fp32, INT8 or bf16 states).
#include "launch.h"
#include "tc_kernel.cuh"

namespace forge {

template <int SDT>
static cudaError_t run_fp8(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bh,
                           const CUtensorMap& s1, const CUtensorMap& s2, const CUtensorMap& w,
                           const GemmParams& p, int grid, cudaStream_t s) {
  auto* k = tc_kernel<kModeFusedFp8, kWBf16, SDT>;
  using Cfg = KCfg<kModeFusedFp8, kWBf16, SDT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pair(k, grid, Cfg::kThreads, Cfg::kSmem, s, a, b, a, bh, s1, s2, a, w, p);
}

cudaError_t launch_tc_fp8(int sdt, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bh,
                          const CUtensorMap& s1, const CUtensorMap& s2, const CUtensorMap& w,
                          const GemmParams& p, int grid, cudaStream_t s) {
  return sdt == kSInt8     ? run_fp8<kSInt8>(a, b, bh, s1, s2, w, p, grid, s)
         : sdt == kSInt8W  ? run_fp8<kSInt8W>(a, b, bh, s1, s2, w, p, grid, s)
         : sdt == kSInt8X  ? run_fp8<kSInt8X>(a, b, bh, s1, s2, w, p, grid, s)
         : sdt == kSInt8WX ? run_fp8<kSInt8WX>(a, b, bh, s1, s2, w, p, grid, s)
         : sdt == kSBf16   ? run_fp8<kSBf16>(a, b, bh, s1, s2, w, p, grid, s)
                           : run_fp8<kSFp32>(a, b, bh, s1, s2, w, p, grid, s);
}

}  // namespace forge
