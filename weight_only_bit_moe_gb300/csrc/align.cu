// Routing alignment: sort the local (token, slot) pairs by expert and pad each
// expert's run to block_m ("013-moe-middle-tiles.py", kernel_fn:
// moe_align_block_size(local_ids, block_size_m, n_experts); the -1 invalid
// block of the expert-parallel filter in "Marlin MoE kernel occupancy ..."
// (sglang PR #31552), marlin_template.h).
//
// One CTA of 1024 threads does the whole job, which at the layer's sizes
// (<= 32768 pairs) costs a few microseconds:
//   1. histogram of local expert ids in shared memory;
//   2. padded counts -> exclusive scan -> run starts, n_padded, block experts;
//   3. stable scatter, 1024 pairs per round: each warp's __match_any_sync mask
//      is the 32-bit membership word of its expert; one warp per expert scans
//      the 32 words of a round, which gives every pair its rank among earlier
//      pairs of the same expert without atomics, so ties keep pair order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignMaxExperts = 1024;

__global__ void __launch_bounds__(kAlignThreads, 1)
    align_kernel(const int32_t* __restrict__ topk_ids, int pairs, int expert_base, int num_experts, int block_m,
                 int64_t cap, int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                 int32_t* __restrict__ n_padded) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int E = num_experts;
  uint32_t* words = reinterpret_cast<uint32_t*>(smem);           // [E][32] membership words
  uint16_t* prefix = reinterpret_cast<uint16_t*>(words + E * 32);  // [E][32] exclusive ranks
  int* count = reinterpret_cast<int*>(prefix + E * 32);           // [E]
  int* start = count + E;                                         // [E]
  int* run = start + E;                                           // [E] pairs placed so far
  int* tot = run + E;                                             // [E] pairs in this round
  __shared__ int warp_sums[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < E * 32; i += kAlignThreads) words[i] = 0u;
  for (int e = tid; e < E; e += kAlignThreads) { count[e] = 0; run[e] = 0; }
  __syncthreads();

  // 1. histogram
  for (int p = tid; p < pairs; p += kAlignThreads) {
    const int e = topk_ids[p] - expert_base;
    if (e >= 0 && e < E) atomicAdd(&count[e], 1);
  }
  __syncthreads();

  // 2. exclusive scan of padded counts (E <= 1024: one value per thread)
  const int padded = tid < E ? (count[tid] + block_m - 1) / block_m * block_m : 0;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += v;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int total = warp_sums[31];
  if (tid < E) start[tid] = incl - padded + (warp ? warp_sums[warp - 1] : 0);
  if (tid == 0) *n_padded = total;
  __syncthreads();

  // block experts, padding sentinels, tail
  const int32_t sentinel = pairs;
  for (int e = tid; e < E; e += kAlignThreads) {
    const int s0 = start[e], c = count[e];
    const int pe = (c + block_m - 1) / block_m * block_m;
    for (int b = s0 / block_m; b < (s0 + pe) / block_m; ++b) expert_ids[b] = e;
    for (int i = c; i < pe; ++i) sorted_ids[s0 + i] = sentinel;
  }
  for (int64_t i = total + tid; i < cap; i += kAlignThreads) sorted_ids[i] = sentinel;
  for (int64_t b = total / block_m + tid; b < cap / block_m; b += kAlignThreads) expert_ids[b] = -1;

  // 3. stable scatter, one round of 1024 pairs at a time
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < pairs; base += kAlignThreads) {
    const int p = base + tid;
    int e = -1;
    if (p < pairs) {
      e = topk_ids[p] - expert_base;
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (m & lt_mask) == 0) words[e * 32 + warp] = m;  // group leader
    __syncthreads();
    // one warp per expert: exclusive prefix of popcounts over the 32 warps
    for (int ex = warp; ex < E; ex += 32) {
      const uint32_t w = words[ex * 32 + lane];
      const int c = __popc(w);
      int s = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
      }
      prefix[ex * 32 + lane] = (uint16_t)(s - c);
      words[ex * 32 + lane] = 0u;
      if (lane == 31) tot[ex] = s;
    }
    __syncthreads();
    if (e >= 0) sorted_ids[start[e] + run[e] + prefix[e * 32 + warp] + __popc(m & lt_mask)] = p;
    __syncthreads();
    for (int ex = tid; ex < E; ex += kAlignThreads) run[ex] += tot[ex];
    __syncthreads();
  }
}

}  // namespace moe

using namespace moe;

extern "C" int64_t moe_align_capacity(int M, int top_k, int num_experts, int block_m) {
  if (M < 0 || top_k <= 0 || num_experts <= 0 || block_m <= 0) return -1;
  const int64_t pairs = (int64_t)M * top_k;
  const int64_t busy = pairs < num_experts ? pairs : num_experts;
  const int64_t n = pairs + busy * (block_m - 1);
  return (n + block_m - 1) / block_m * block_m;
}

extern "C" int moe_align(const int32_t* topk_ids, int M, int top_k, int expert_base, int num_experts,
                         int block_m, int32_t* sorted_ids, int32_t* expert_ids, int32_t* n_padded,
                         void* stream) {
  if (M < 0 || top_k <= 0 || num_experts <= 0 || num_experts > kAlignMaxExperts) return MOE_ERR_INVALID;
  if (block_m != 8 && block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) return MOE_ERR_INVALID;
  if ((int64_t)M * top_k >= (int64_t)1 << 31) return MOE_ERR_INVALID;
  if (!sorted_ids || !expert_ids || !n_padded || (M > 0 && !topk_ids)) return MOE_ERR_INVALID;
  const int64_t cap = moe_align_capacity(M, top_k, num_experts, block_m);
  const size_t smem = (size_t)num_experts * 32 * (4 + 2) + (size_t)num_experts * 4 * 4;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)((size_t)kAlignMaxExperts * 32 * 6 + kAlignMaxExperts * 16)) != cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set = true;
  }
  align_kernel<<<1, kAlignThreads, smem, (cudaStream_t)stream>>>(topk_ids, M * top_k, expert_base, num_experts,
                                                                 block_m, cap, sorted_ids, expert_ids, n_padded);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
