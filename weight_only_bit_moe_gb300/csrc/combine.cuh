// Arguments of the combine kernel (combine.cu).
#pragma once

#include "common.cuh"

namespace moe {

struct CombineArgs {
  int M, top_k, K, Kpad2, expert_base, E;
  const int32_t* topk_ids;      // [M, top_k]
  const float* topk_weights;    // [M, top_k]
  const float* y;               // GEMM2 fp32 output [pairs, K] (split == 1)
  const float* partial;         // GEMM2 fp32 partial slices (split > 1)
  int split_rows;
  const int32_t* split_used;    // split chosen by GEMM2 (device)
  const int32_t* inv_pos;       // pair -> sorted position
  const float* gs2;             // [E] epilogue scale of GEMM2
  const uint16_t* b2;           // [E, Kpad2] or NULL
  const uint16_t* post_norm_w;  // [K] or NULL
  float norm_eps, rsf;
  uint16_t* out;                // [M, K]
};

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t st);

}  // namespace moe
