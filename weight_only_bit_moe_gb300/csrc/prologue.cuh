// The forward's first kernel (align.cu): routing alignment, the bf16 -> fp16
// conversion of the activations and the clearing of the workspace header, in
// one launch.  moe_align runs the same kernel with the alignment part only.
#pragma once

#include "common.cuh"

namespace moe {

struct PrologueArgs {
  // alignment (topk_ids == NULL: none in this launch)
  const int32_t* topk_ids;   // [M, top_k]
  int pairs, expert_base, E, block_m;
  int64_t cap;               // sorted slots (moe_align_capacity)
  int32_t* sorted_ids;       // [cap]
  int32_t* expert_ids;       // [cap / block_m]
  int32_t* n_padded;         // [1]
  // activations: x (bf16) to fp16, as x's own rows or in sorted order (x == NULL: neither)
  const uint16_t* x;         // bf16 [M, K]
  int M, K, top_k;
  uint16_t* xh;              // fp16 [M, K]: row t = x[t] (register-fed GEMMs gather from it), or NULL
  uint16_t* xs;              // fp16 [cap, K]: row pos = x[sorted_ids[pos] / top_k] for routed slots
                             // (tcgen05 GEMMs), or NULL; written as this launch aligns, or else from
                             // the caller's alignment below (padding rows are not written)
  const int32_t* given_sorted;   // the caller's alignment (moe_align), read when this launch does not align
  const int32_t* given_expert_ids;
  const int32_t* given_n_padded;
  const int32_t* perm13;     // act-order banks: int32 [E][K], x column of packed column k of expert e
                             // (xs rows then hold x's columns in their expert's order), or NULL
  int32_t* pair_pos;         // [pairs] scratch: sorted position of each local pair (xs while aligning)
  int align_ctas;            // CTAs that align (and copy their pairs' rows); 0: the minimum
  // workspace header words to clear (zero_words == 0: none)
  uint32_t* zero;
  int64_t zero_words;
};

// Launches the kernel on `st` as a programmatic dependent of its predecessor.
cudaError_t launch_prologue(const PrologueArgs& a, int sms, cudaStream_t st);

// align_ctas for a launch that also copies the pairs' rows of K columns.
int align_copy_ctas(int pairs, int K, int sms);

}  // namespace moe
