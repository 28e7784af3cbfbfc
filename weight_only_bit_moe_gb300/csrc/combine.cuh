// Arguments of the combine kernel (combine.cu).
#pragma once

#include "common.cuh"

namespace moe {

struct CombineArgs {
  int M, top_k, K, expert_base, E;
  const int32_t* topk_ids;      // [M, top_k]
  const float* topk_weights;    // [M, top_k]
  const float* y;               // GEMM2 output, fp32 [pairs, K] (rows of local pairs)
  const uint16_t* post_norm_w;  // [K] or NULL
  float norm_eps, rsf;
  uint16_t* out;                // [M, K]
};

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t st);

}  // namespace moe
