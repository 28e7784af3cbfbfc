// Routing alignment: sort the local (token, slot) pairs by expert and pad each
// expert's run to block_m ("013-moe-middle-tiles.py", kernel_fn:
// moe_align_block_size(local_ids, block_size_m, n_experts); the -1 invalid
// block of the expert-parallel filter in "Marlin MoE kernel occupancy ..."
// (sglang PR #31552), marlin_template.h).
//
// A stable counting sort spread over G CTAs with no communication between
// them.  The pairs are cut into G contiguous chunks; CTA c
//   1. counts every local pair per expert (shared-memory atomics) -- the
//      expert totals -- and, apart, the pairs of the chunks before its own, and
//      counts its own chunk per warp segment into a [32][E] table;
//   2. scans the padded totals into run starts (every CTA gets the same
//      starts) and, per expert, the segment counts into segment offsets;
//   3. writes the padding slots, block experts and -1 blocks of the experts
//      and ranges it owns (round-robin over CTAs), and n_padded (CTA 0);
//   4. scatters its chunk: each warp walks its segment 32 pairs at a time; the
//      lanes that share an expert (one ballot per key bit) take consecutive
//      slots after that expert's running offset, so equal experts keep
//      ascending pair order across segments and chunks.
// Each CTA reads all ids once (L2-resident after the first), so the cost is
// one pass over the ids per CTA plus a chunk of ~1024 pairs: a few
// microseconds at 32768 pairs, against one CTA's ~50 walking them all.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignMaxExperts = 1024;
constexpr int kAlignChunk = 1024;   // pairs scattered per CTA (the grid covers the pairs)
constexpr int kAlignMaxCtas = 128;  // beyond this the chunks grow instead

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
  const int e = __ldg(ids + p) - base;
  return (e >= 0 && e < E) ? e : -1;
}

__global__ void __launch_bounds__(kAlignThreads, 1)
    align_kernel(const int32_t* __restrict__ topk_ids, int pairs, int expert_base, int num_experts, int block_m,
                 int64_t cap, int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                 int32_t* __restrict__ n_padded) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int E = num_experts;
  const int Ep = E + 1;                     // row stride: column walks hit distinct banks
  int* tab = reinterpret_cast<int*>(smem);  // [32][Ep] segment counts, then absolute offsets
  int* total = tab + kAlignWarps * Ep;      // [E] local pairs per expert
  int* before = total + E;                  // [E] ... in the chunks before this CTA's
  int* start = before + E;                  // [E] padded run start
  __shared__ int warp_sums[32];

  grid_dependency_wait();
  grid_dependents_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int chunk = (pairs + G - 1) / G;
  const int q0 = min(pairs, c * chunk), q1 = min(pairs, q0 + chunk);
  const int seg = (q1 - q0 + kAlignWarps - 1) / kAlignWarps;
  const int p0 = min(q1, q0 + warp * seg), p1 = min(q1, p0 + seg);
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int key_bits = 32 - __clz(E);  // keys 0..E
  int* row = tab + warp * Ep;

  for (int i = tid; i < kAlignWarps * Ep + 2 * E; i += kAlignThreads) tab[i] = 0;
  __syncthreads();

  // 1. expert totals and the counts of the earlier chunks (every id, one pass;
  //    eight loads in flight per thread before their atomics)
  constexpr int kBatch = 8;
  for (int pass = 0; pass < pairs; pass += kBatch * kAlignThreads) {
    int ev[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int p = pass + i * kAlignThreads + tid;
      ev[i] = p < pairs ? local_expert(topk_ids, p, expert_base, E) : -1;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (ev[i] >= 0) {
        atomicAdd(&total[ev[i]], 1);
        if (pass + i * kAlignThreads + tid < q0) atomicAdd(&before[ev[i]], 1);
      }
    }
  }
  //    this warp's segment, per expert
  for (int p = p0 + lane; p < p1; p += 32) {
    const int e = local_expert(topk_ids, p, expert_base, E);
    if (e >= 0) atomicAdd(&row[e], 1);
  }
  __syncthreads();

  // 2. padded scan over experts (E <= 1024: one expert per thread) ...
  const int cnt = tid < E ? total[tid] : 0;
  const int padded = (cnt + block_m - 1) / block_m * block_m;
  int incl = padded;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  //    ... and, per expert, one warp scans the 32 segment counts (lane = segment)
  for (int e = warp; e < E; e += kAlignWarps) {
    const int v = tab[lane * Ep + e];
    int s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    tab[lane * Ep + e] = s - v + before[e];  // offset of the segment inside the expert's run
  }
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
  const int n_total = warp_sums[31];
  if (tid < E) start[tid] = incl - padded + (warp ? warp_sums[warp - 1] : 0);
  if (c == 0 && tid == 0) *n_padded = n_total;
  __syncthreads();

  // 3. padding slots and block experts of the experts this CTA owns; the tail
  //    past n_padded (sentinel slots, -1 blocks) split over all CTAs
  //    (one warp per expert: a thread's global stores issue one after another,
  //    so the experts' stores go out from different warps side by side)
  const int32_t sentinel = pairs;
  for (int e = c + warp * G; e < E; e += kAlignWarps * G) {
    const int s0 = start[e], n = total[e];
    const int pe = (n + block_m - 1) / block_m * block_m;
    for (int i = s0 + n + lane; i < s0 + pe; i += 32) sorted_ids[i] = sentinel;
    for (int b = s0 / block_m + lane; b < (s0 + pe) / block_m; b += 32) expert_ids[b] = e;
  }
  for (int64_t i = n_total + (int64_t)c * kAlignThreads + tid; i < cap; i += (int64_t)G * kAlignThreads)
    sorted_ids[i] = sentinel;
  for (int64_t b = n_total / block_m + (int64_t)c * kAlignThreads + tid; b < cap / block_m;
       b += (int64_t)G * kAlignThreads)
    expert_ids[b] = -1;
  for (int idx = tid; idx < kAlignWarps * E; idx += kAlignThreads) {
    const int w = idx / E, e = idx - w * E;
    tab[w * Ep + e] += start[e];
  }
  __syncthreads();

  // 4. stable scatter of this warp's segment, rounds in pair order
  for (int pass = p0; pass < p1; pass += 32) {
    const int p = pass + lane;
    const int e = p < p1 ? local_expert(topk_ids, p, expert_base, E) : -1;
    const uint32_t m = peer_mask(e + 1, key_bits);
    if (e >= 0) sorted_ids[row[e] + __popc(m & lt_mask)] = p;
    __syncwarp();
    if (e >= 0 && (m & lt_mask) == 0) row[e] += __popc(m);
    __syncwarp();
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
  const int pairs = M * top_k;
  const size_t smem = ((size_t)kAlignWarps * (num_experts + 1) + 3 * (size_t)num_experts) * 4;
  static bool configured[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(((size_t)kAlignWarps * (kAlignMaxExperts + 1) + 3 * (size_t)kAlignMaxExperts) * 4)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev] = true;
  }
  int ctas = (pairs + kAlignChunk - 1) / kAlignChunk;
  ctas = ctas < 1 ? 1 : (ctas > kAlignMaxCtas ? kAlignMaxCtas : ctas);
  const cudaError_t err = launch_dependent(align_kernel, dim3(ctas), dim3(kAlignThreads), smem, (cudaStream_t)stream,
                                           topk_ids, pairs, expert_base, num_experts, block_m, cap, sorted_ids,
                                           expert_ids, n_padded);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
