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
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = tid; i < a.zero_words; i += nthreads) a.zero[i] = 0u;
  // one 16-byte chunk of one routed row per thread and iteration, so short
  // batches still issue all their loads at once
  const int64_t n_padded = *a.n_padded;
  const int chunks = a.K / 8;  // 16-byte chunks per row
  const int64_t total = n_padded * chunks;
  for (int64_t idx = tid; idx < total; idx += nthreads) {
    const int64_t pos = idx / chunks;
    const int c = (int)(idx - pos * chunks);
    const int sid = a.sorted_ids[pos];
    if (sid >= a.pairs) continue;
    const uint4 v = reinterpret_cast<const uint4*>(a.x)[(int64_t)(sid / a.top_k) * chunks + c];
    reinterpret_cast<uint4*>(a.xs)[pos * chunks + c] =
        a.to_f16 ? make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w))
                 : v;
  }
}

cudaError_t launch_prep(const PrepArgs& a, int sms, cudaStream_t st) {
  // the routed row count is only known on the device: size for the capacity
  const int64_t work = a.zero_words > a.cap * (a.K / 8) ? a.zero_words : a.cap * (a.K / 8);
  int64_t blocks = (work + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  return launch_dependent(prep_kernel, dim3((unsigned)blocks), dim3(256), 0, st, a);
}

}  // namespace moe
