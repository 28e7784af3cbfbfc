// Grouped GEMM instances for one weight format (see gemm.cuh).
#include "gemm_launch.cuh"

namespace moe {
cudaError_t launch_gemm_nvfp4(bool gated, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  return launch_gemm_fmt<MOE_W_NVFP4>(gated, bn, g, grid, st);
}
}  // namespace moe
