// Instantiations of the tensor-core kernel with plain store epilogues: the
// unfused weight-gradient pass (fp32 dW to global memory) and dX = dY W.
#include "launch.h"
#include "tc_kernel.cuh"

namespace forge {

template <int MODE>
static cudaError_t run_plain(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                             int grid, cudaStream_t s) {
  auto* k = tc_kernel<MODE, kWBf16, kSFp32>;
  constexpr int smem = KCfg<MODE, kWBf16>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pair(k, grid, KCfg<MODE, kWBf16>::kThreads, smem, s, a, b, a, b, a, a, a, a, p);  // only a, b used
}

cudaError_t launch_tc_plain(int mode, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmParams& p, int grid, cudaStream_t s) {
  return mode == kModeDgrad ? run_plain<kModeDgrad>(a, b, p, grid, s)
                            : run_plain<kModeWgradStore>(a, b, p, grid, s);
}

}  // namespace forge
