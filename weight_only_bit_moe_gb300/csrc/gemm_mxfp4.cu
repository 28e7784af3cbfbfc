// Grouped GEMM instances for one weight format (see gemm.cuh and gemm_small.cuh).
#include "gemm_launch.cuh"

namespace moe {
cudaError_t launch_gemm_mxfp4(bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  return small ? launch_gemm_small_fmt<MOE_W_MXFP4>(stage, bn, g, grid, st) : launch_gemm_fmt<MOE_W_MXFP4>(stage, bn, g, grid, st);
}
}  // namespace moe
