// Launch helpers for the grouped GEMM instantiations (one translation unit per
// weight format, so the three compile in parallel).
#pragma once

#include "gemm.cuh"
#include "gemm_small.cuh"

namespace moe {

// Launch one (FMT, STAGE, BN) instance on `grid` CTAs; sets the kernel's
// dynamic shared-memory limit once per device.
template <int FMT, int STAGE, int BN>
cudaError_t launch_gemm_instance(const GemmArgs& g, int grid, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(moe_gemm_kernel<FMT, STAGE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               GemmSmem<BN, FMT>::kAlloc);
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  return launch_dependent(moe_gemm_kernel<FMT, STAGE, BN>, dim3(grid), dim3(GemmCfg<FMT, BN, STAGE>::kThreads), GemmSmem<BN, FMT>::kAlloc, st, g);
}

template <int FMT, int BN>
cudaError_t launch_gemm_stage(int stage, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (stage) {
    case kGemm2: return launch_gemm_instance<FMT, kGemm2, BN>(g, grid, st);
    case kGemm1Gated: return launch_gemm_instance<FMT, kGemm1Gated, BN>(g, grid, st);
    case kGemm1Relu2: return launch_gemm_instance<FMT, kGemm1Relu2, BN>(g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int FMT>
cudaError_t launch_gemm_fmt(int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (bn) {
    case 64: return launch_gemm_stage<FMT, 64>(stage, g, grid, st);
    case 128: return launch_gemm_stage<FMT, 128>(stage, g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// Register-fed kernel for token blocks of 8, 16 or 32 (gemm_small.cuh).
template <int FMT, int STAGE, int BN>
cudaError_t launch_gemm_small_instance(const GemmArgs& g, int grid, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(moe_gemm_small_kernel<FMT, STAGE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SmallSmem<BN, FMT>::kAlloc);
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  return launch_dependent(moe_gemm_small_kernel<FMT, STAGE, BN>, dim3(grid), dim3(SmallCfg<BN, STAGE>::kThreads),
                          SmallSmem<BN, FMT>::kAlloc, st, g);
}

template <int FMT, int BN>
cudaError_t launch_gemm_small_stage(int stage, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (stage) {
    case kGemm2: return launch_gemm_small_instance<FMT, kGemm2, BN>(g, grid, st);
    case kGemm1Gated: return launch_gemm_small_instance<FMT, kGemm1Gated, BN>(g, grid, st);
    case kGemm1Relu2: return launch_gemm_small_instance<FMT, kGemm1Relu2, BN>(g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int FMT>
cudaError_t launch_gemm_small_fmt(int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (bn) {
    case 8: return launch_gemm_small_stage<FMT, 8>(stage, g, grid, st);
    case 16: return launch_gemm_small_stage<FMT, 16>(stage, g, grid, st);
    case 32: return launch_gemm_small_stage<FMT, 32>(stage, g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// small = true selects the register-fed kernel (bn = block_m in {8, 16, 32});
// stage is a GemmStage.
cudaError_t launch_gemm_int4(bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st);
cudaError_t launch_gemm_mxfp4(bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st);
cudaError_t launch_gemm_nvfp4(bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st);
cudaError_t launch_gemm_int4x(bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st);

}  // namespace moe
