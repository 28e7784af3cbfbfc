// Launch helpers for the grouped GEMM instantiations (one translation unit per
// weight format, so the three compile in parallel).
#pragma once

#include "gemm.cuh"
#include "gemm_small.cuh"

namespace moe {

// Launch one (FMT, GATED, BN) instance on `grid` CTAs; sets the kernel's
// dynamic shared-memory limit once per device.
template <int FMT, bool GATED, int BN>
cudaError_t launch_gemm_instance(const GemmArgs& g, int grid, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(moe_gemm_kernel<FMT, GATED, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               GemmSmem<BN>::kAlloc);
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  return launch_dependent(moe_gemm_kernel<FMT, GATED, BN>, dim3(grid), dim3(kGemmThreads), GemmSmem<BN>::kAlloc, st, g);
}

template <int FMT>
cudaError_t launch_gemm_fmt(bool gated, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (bn) {
    case 64: return gated ? launch_gemm_instance<FMT, true, 64>(g, grid, st) : launch_gemm_instance<FMT, false, 64>(g, grid, st);
    case 128: return gated ? launch_gemm_instance<FMT, true, 128>(g, grid, st) : launch_gemm_instance<FMT, false, 128>(g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// Register-fed kernel for token blocks of 8, 16 or 32 (gemm_small.cuh).
template <int FMT, bool GATED, int BN>
cudaError_t launch_gemm_small_instance(const GemmArgs& g, int grid, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(moe_gemm_small_kernel<FMT, GATED, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SmallSmem<BN>::kAlloc);
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  return launch_dependent(moe_gemm_small_kernel<FMT, GATED, BN>, dim3(grid), dim3(kSmallThreads),
                          SmallSmem<BN>::kAlloc, st, g);
}

template <int FMT>
cudaError_t launch_gemm_small_fmt(bool gated, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (bn) {
    case 8: return gated ? launch_gemm_small_instance<FMT, true, 8>(g, grid, st) : launch_gemm_small_instance<FMT, false, 8>(g, grid, st);
    case 16: return gated ? launch_gemm_small_instance<FMT, true, 16>(g, grid, st) : launch_gemm_small_instance<FMT, false, 16>(g, grid, st);
    case 32: return gated ? launch_gemm_small_instance<FMT, true, 32>(g, grid, st) : launch_gemm_small_instance<FMT, false, 32>(g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// small = true selects the register-fed kernel (bn = block_m in {8, 16, 32}).
cudaError_t launch_gemm_int4(bool small, bool gated, int bn, const GemmArgs& g, int grid, cudaStream_t st);
cudaError_t launch_gemm_mxfp4(bool small, bool gated, int bn, const GemmArgs& g, int grid, cudaStream_t st);
cudaError_t launch_gemm_nvfp4(bool small, bool gated, int bn, const GemmArgs& g, int grid, cudaStream_t st);

}  // namespace moe
