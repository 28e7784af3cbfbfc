// Forward prologue kernel (prep.cu).
#pragma once

#include "common.cuh"

namespace moe {

struct PrepArgs {
  uint32_t* zero;            // words to clear
  int64_t zero_words;
  const uint16_t* x;         // bf16 [M, K]
  uint16_t* xs;              // 16-bit [cap, K], row pos = routed row of sorted slot pos
  const int32_t* sorted_ids;
  const int32_t* n_padded;
  int64_t cap;
  int pairs, top_k, K;
  int to_f16;                // convert bf16 -> fp16
};

cudaError_t launch_prep(const PrepArgs& a, int sms, cudaStream_t st);

}  // namespace moe
