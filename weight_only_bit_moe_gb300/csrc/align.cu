// Routing alignment: sort the local (token, slot) pairs by expert and pad each
// expert's run to block_m ("013-moe-middle-tiles.py", kernel_fn:
// moe_align_block_size(local_ids, block_size_m, n_experts); the -1 invalid
// block of the expert-parallel filter in "Marlin MoE kernel occupancy ..."
// (sglang PR #31552), marlin_template.h).
//
// One CTA of 1024 threads does the whole job, which at the layer's sizes
// (<= 32768 pairs) costs a few microseconds.  It is a stable counting sort:
//   1. each of the 32 warps owns a contiguous segment of pairs and counts its
//      segment's local expert ids into its own row of a [32][E] table;
//   2. per expert, one warp scans the 32 segment counts into the expert's total
//      and the segments' offsets; the padded totals are scanned into run
//      starts and n_padded; every slot is pre-filled as padding;
//   3. the offsets become absolute and the block -> expert table is written;
//   4. each warp walks its segment in order, 32 pairs at a time: the lanes that
//      share an expert (found with one ballot per key bit) take consecutive slots after that
//      expert's running offset, so equal experts keep ascending pair order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignMaxExperts = 1024;
constexpr int kAlignBatch = 16;  // rounds of 32 ids a warp loads at once

// Lanes of the warp whose key equals this lane's: one ballot per key bit (keys
// are local expert + 1, so non-local pairs share key 0).
__device__ __forceinline__ uint32_t peer_mask(int key, int nbits) {
  uint32_t m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const int bit = (key >> b) & 1;
    const uint32_t bal = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

__device__ __forceinline__ int local_expert(const int32_t* ids, int p, int base, int E) {
  const int e = ids[p] - base;
  return (e >= 0 && e < E) ? e : -1;
}

__global__ void __launch_bounds__(kAlignThreads, 1)
    align_kernel(const int32_t* __restrict__ topk_ids, int pairs, int expert_base, int num_experts, int block_m,
                 int64_t cap, int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                 int32_t* __restrict__ n_padded) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int E = num_experts;
  const int Ep = E + 1;                     // row stride: column walks hit distinct banks
  int* tab = reinterpret_cast<int*>(smem);  // [32][Ep] segment counts, then segment offsets
  int* count = tab + kAlignWarps * Ep;      // [E]
  int* start = count + E;                   // [E]
  __shared__ int warp_sums[32];

  grid_dependency_wait();
  grid_dependents_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (pairs + kAlignWarps - 1) / kAlignWarps;
  const int p0 = warp * seg, p1 = min(pairs, p0 + seg);
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int key_bits = 32 - __clz(E);  // keys 0..E
  int* row = tab + warp * Ep;

  // 1. segment counts; a warp loads up to kAlignBatch rounds of 32 ids at once
  //    (one round trip), then counts them.  A segment that fits one batch keeps
  //    its ids in registers for the scatter.
  for (int e = lane; e < E; e += 32) row[e] = 0;
  __syncwarp();
  const bool one_batch = p1 - p0 <= 32 * kAlignBatch;
  int keep[kAlignBatch];
  for (int pass = p0; pass < p1; pass += 32 * kAlignBatch) {
    int ev[kAlignBatch];
#pragma unroll
    for (int i = 0; i < kAlignBatch; ++i) {
      const int p = pass + 32 * i + lane;
      ev[i] = p < p1 ? local_expert(topk_ids, p, expert_base, E) : -1;
      keep[i] = ev[i];
    }
#pragma unroll
    for (int i = 0; i < kAlignBatch; ++i) {
      if (pass + 32 * i >= p1) break;
      const uint32_t m = peer_mask(ev[i] + 1, key_bits);
      if (ev[i] >= 0 && (m & lt_mask) == 0) row[ev[i]] += __popc(m);
      __syncwarp();
    }
  }
  __syncthreads();

  // 2. per expert, one warp scans the 32 segment counts (lane = segment): the
  //    expert's total and each segment's offset inside the expert's run
  for (int e = warp; e < E; e += kAlignWarps) {
    const int v = tab[lane * Ep + e];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    tab[lane * Ep + e] = incl - v;
    if (lane == 31) count[e] = incl;
  }
  __syncthreads();

  //    padded scan over experts (E <= 1024: one expert per thread)
  const int c = tid < E ? count[tid] : 0;
  const int padded = (c + block_m - 1) / block_m * block_m;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int sum = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, sum, o);
      if (lane >= o) sum += v;
    }
    warp_sums[lane] = sum;  // inclusive over warps
  }
  __syncthreads();
  const int total = warp_sums[31];
  if (tid < E) start[tid] = incl - padded + (warp ? warp_sums[warp - 1] : 0);
  if (tid == 0) *n_padded = total;
  // every slot starts as padding and every block as -1; real entries and block
  // experts overwrite them after the barrier
  const int32_t sentinel = pairs;
  for (int64_t i = tid; i < cap; i += kAlignThreads) sorted_ids[i] = sentinel;
  for (int64_t b = tid; b < cap / block_m; b += kAlignThreads) expert_ids[b] = -1;
  __syncthreads();

  // 3. absolute offsets of each segment; block -> expert
  for (int idx = tid; idx < kAlignWarps * E; idx += kAlignThreads) {
    const int w = idx / E, e = idx - w * E;
    tab[w * Ep + e] += start[e];
  }
  for (int e = tid; e < E; e += kAlignThreads) {
    const int s0 = start[e];
    const int pe = (count[e] + block_m - 1) / block_m * block_m;
    for (int b = s0 / block_m; b < (s0 + pe) / block_m; ++b) expert_ids[b] = e;
  }
  __syncthreads();

  // 4. stable scatter of each segment, rounds in pair order
  for (int pass = p0; pass < p1; pass += 32 * kAlignBatch) {
    int ev[kAlignBatch];
#pragma unroll
    for (int i = 0; i < kAlignBatch; ++i) {
      const int p = pass + 32 * i + lane;
      ev[i] = one_batch ? keep[i] : (p < p1 ? local_expert(topk_ids, p, expert_base, E) : -1);
    }
#pragma unroll
    for (int i = 0; i < kAlignBatch; ++i) {
      if (pass + 32 * i >= p1) break;
      const int e = ev[i];
      const uint32_t m = peer_mask(e + 1, key_bits);
      if (e >= 0) sorted_ids[row[e] + __popc(m & lt_mask)] = pass + 32 * i + lane;
      __syncwarp();
      if (e >= 0 && (m & lt_mask) == 0) row[e] += __popc(m);
      __syncwarp();
    }
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
  const size_t smem = ((size_t)kAlignWarps * (num_experts + 1) + 2 * (size_t)num_experts) * 4;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(((size_t)kAlignWarps * (kAlignMaxExperts + 1) + 2 * (size_t)kAlignMaxExperts) * 4)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev] = true;
  }
  const cudaError_t err = launch_dependent(align_kernel, dim3(1), dim3(kAlignThreads), smem, (cudaStream_t)stream,
                                           topk_ids, M * top_k, expert_base, num_experts, block_m, cap, sorted_ids,
                                           expert_ids, n_padded);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
