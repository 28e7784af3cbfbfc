// Grouped GEMM instances for INT4 banks with zero points or groups of 32 / 64
// (the INT4X packed format; see gemm.cuh and gemm_small.cuh).
#include "gemm_launch.cuh"

namespace moe {
cudaError_t launch_gemm_int4x(bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  return small ? launch_gemm_small_fmt<kFmtInt4X>(stage, bn, g, grid, st) : launch_gemm_fmt<kFmtInt4X>(stage, bn, g, grid, st);
}
}  // namespace moe
