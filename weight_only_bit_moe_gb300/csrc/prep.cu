// Forward prologue kernel.  It zeroes the workspace header (status word and the
// split-K arrival counters) and gathers the routed activation rows into sorted
// order -- row pos of xs is x[sorted_ids[pos] / top_k] -- so both grouped GEMMs
// read their token operand as plain 2-D tiles.  The copy is converted to fp16
// (exact inside the fp16 range) for the fp16 x fp16 tensor-core operands.
// Padding slots are left untouched: the GEMMs discard their columns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "prep.cuh"

namespace moe {

__global__ void __launch_bounds__(256) prep_kernel(PrepArgs a) {
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = tid; i < a.zero_words; i += nthreads) a.zero[i] = 0u;
  const int lane = threadIdx.x & 31;
  const int64_t warp = tid >> 5, nwarps = nthreads >> 5;
  const int n_padded = *a.n_padded;
  const int chunks = a.K / 8;  // 16-byte chunks per row
  for (int64_t pos = warp; pos < n_padded; pos += nwarps) {
    const int sid = a.sorted_ids[pos];
    if (sid >= a.pairs) continue;
    const uint4* src = reinterpret_cast<const uint4*>(a.x) + (int64_t)(sid / a.top_k) * chunks;
    uint4* dst = reinterpret_cast<uint4*>(a.xs) + pos * chunks;
    for (int c = lane; c < chunks; c += 32) {
      const uint4 v = src[c];
      dst[c] = a.to_f16 ? make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                                     bf16x2_to_f16x2(v.w))
                        : v;
    }
  }
}

cudaError_t launch_prep(const PrepArgs& a, int sms, cudaStream_t st) {
  const int64_t work = a.zero_words > a.cap * 32 ? a.zero_words : a.cap * 32;
  int64_t blocks = (work + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  prep_kernel<<<(int)blocks, 256, 0, st>>>(a);
  return cudaPeekAtLastError();
}

}  // namespace moe
