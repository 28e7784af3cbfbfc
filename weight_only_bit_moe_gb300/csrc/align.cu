// Routing alignment: sort the local (token, slot) pairs by expert and pad each
// expert's run to block_m ("013-moe-middle-tiles.py", kernel_fn:
// moe_align_block_size(local_ids, block_size_m, n_experts), and the
// moe_align_single_token path it takes for one token; the -1 invalid block of
// the expert-parallel filter in "Marlin MoE kernel occupancy ..." (sglang PR
// #31552), marlin_template.h).  It runs as the first part of the forward's
// prologue kernel, which also converts the activations to fp16 and clears the
// workspace header, or alone for moe_align.
//
// Up to 32 pairs (decode: a few tokens) one warp aligns them in registers:
// lane p holds pair p, finds the lanes routed to its expert with one shuffle
// per lane, and the run starts are sums over the first lane of each expert --
// no tables, no shared memory.
//
// Beyond that, a stable counting sort spread over G CTAs with no
// communication between them.  The pairs are cut into G contiguous chunks; CTA c
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

#include <algorithm>

#include "prologue.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignMaxExperts = 1024;
constexpr int kAlignChunk = 1024;   // pairs scattered per CTA (the grid covers the pairs)
constexpr int kAlignMaxCtas = 128;  // beyond this the chunks grow instead
constexpr int kAlignFew = 32;       // up to this many pairs one warp aligns them

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

// Columns [8c, 8c+8) of token row `token` of x as fp16 (exact inside the fp16
// range, beyond it infinity), in expert e's column order for act-order banks.
__device__ __forceinline__ uint4 x_chunk_f16(const PrologueArgs& a, int token, int e, int c) {
  const uint16_t* row = a.x + (int64_t)token * a.K;
  uint4 v;
  if (!a.perm13) {
    v = __ldg(reinterpret_cast<const uint4*>(row) + c);
  } else {
    const int4* pp = reinterpret_cast<const int4*>(a.perm13 + (int64_t)e * a.K + 8 * c);
    const int4 p0 = __ldg(pp), p1 = __ldg(pp + 1);
    const int idx[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = (uint32_t)__ldg(row + idx[2 * i]) | ((uint32_t)__ldg(row + idx[2 * i + 1]) << 16);
    v = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
}

// One routed row into sorted order: xs[pos] = fp16(x[token]) (columns in expert
// e's order for act-order banks), by the calling warp (16-byte chunks).
__device__ __forceinline__ void copy_row_f16(const PrologueArgs& a, int token, int e, int64_t pos, int lane) {
  uint4* dst = reinterpret_cast<uint4*>(a.xs + pos * a.K);
  const int chunks = a.K / 8;
  for (int c = lane; c < chunks; c += 32) dst[c] = x_chunk_f16(a, token, e, c);
}

// The one-warp alignment of align_few: writes the pairs, the run experts and
// n_padded, and each pair's sorted position (-1: not local) to pos_out.
__device__ void align_few_warp(const PrologueArgs& a, int lane, int* pos_out) {
  const int e = lane < a.pairs ? local_expert(a.topk_ids, lane, a.expert_base, a.E) : -1;
  uint32_t same = 0;  // lanes routed to this lane's expert
  for (int q = 0; q < 32; ++q) {
    const int eq = __shfl_sync(0xffffffffu, e, q);
    if (e >= 0 && eq == e) same |= 1u << q;
  }
  const int rank = __popc(same & ((1u << lane) - 1u));  // pair order within the expert
  const int padded = (e >= 0 && rank == 0) ? (__popc(same) + a.block_m - 1) / a.block_m * a.block_m : 0;
  int start = 0, total = 0;  // this expert's run start (experts in ascending id), all runs
  for (int q = 0; q < 32; ++q) {
    const int eq = __shfl_sync(0xffffffffu, e, q), pq = __shfl_sync(0xffffffffu, padded, q);
    total += pq;
    if (pq && eq < e) start += pq;
  }
  if (e >= 0) a.sorted_ids[start + rank] = lane;
  pos_out[lane] = e >= 0 ? start + rank : -1;
  if (padded)
    for (int b = start / a.block_m; b < (start + padded) / a.block_m; ++b) a.expert_ids[b] = e;
  if (lane == 0) *a.n_padded = total;
}

// Alignment of at most 32 pairs (one CTA).  Every thread of the CTA first
// fills the whole capacity with the sentinel and every block with -1; then warp
// 0, lane p holding pair p, writes the pairs, the run experts and n_padded.
__device__ void align_few(const PrologueArgs& a) {
  __shared__ int few_pos[32];  // sorted position of each pair, -1 when not local
  const int tid = threadIdx.x, lane = tid & 31;
  for (int64_t i = tid; i < a.cap; i += blockDim.x) a.sorted_ids[i] = a.pairs;
  for (int64_t b = tid; b < a.cap / a.block_m; b += blockDim.x) a.expert_ids[b] = -1;
  __syncthreads();
  if (tid < 32) align_few_warp(a, lane, few_pos);
  __syncthreads();
  // routed rows into sorted order: warp w copies pair w's
  const int w = tid >> 5;
  if (a.xs && w < a.pairs && few_pos[w] >= 0)
    copy_row_f16(a, w / a.top_k, local_expert(a.topk_ids, w, a.expert_base, a.E), few_pos[w], lane);
}

// The counting sort of the first G CTAs (c = this CTA), described above.
__device__ void align_many(const PrologueArgs& a, int G, int c, unsigned char* smem) {
  const int E = a.E, pairs = a.pairs, block_m = a.block_m, expert_base = a.expert_base;
  const int32_t* topk_ids = a.topk_ids;
  int32_t* sorted_ids = a.sorted_ids;
  int32_t* expert_ids = a.expert_ids;
  const int Ep = E + 1;                     // row stride: column walks hit distinct banks
  int* tab = reinterpret_cast<int*>(smem);  // [32][Ep] segment counts, then absolute offsets
  int* total = tab + kAlignWarps * Ep;      // [E] local pairs per expert
  int* before = total + E;                  // [E] ... in the chunks before this CTA's
  int* start = before + E;                  // [E] padded run start
  __shared__ int warp_sums[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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
  if (c == 0 && tid == 0) *a.n_padded = n_total;
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
  for (int64_t i = n_total + (int64_t)c * kAlignThreads + tid; i < a.cap; i += (int64_t)G * kAlignThreads)
    sorted_ids[i] = sentinel;
  for (int64_t b = n_total / block_m + (int64_t)c * kAlignThreads + tid; b < a.cap / block_m;
       b += (int64_t)G * kAlignThreads)
    expert_ids[b] = -1;
  for (int idx = tid; idx < kAlignWarps * E; idx += kAlignThreads) {
    const int w = idx / E, e = idx - w * E;
    tab[w * Ep + e] += start[e];
  }
  __syncthreads();

  // 4. stable scatter of this warp's segment, rounds in pair order; with xs the
  //    warp also copies each placed pair's row of x into its sorted position
  for (int pass = p0; pass < p1; pass += 32) {
    const int p = pass + lane;
    const int e = p < p1 ? local_expert(topk_ids, p, expert_base, E) : -1;
    const uint32_t m = peer_mask(e + 1, key_bits);
    const int pos = e >= 0 ? row[e] + __popc(m & lt_mask) : -1;
    if (e >= 0) sorted_ids[pos] = p;
    if (a.xs && p < p1) a.pair_pos[p] = pos;
    __syncwarp();
    if (e >= 0 && (m & lt_mask) == 0) row[e] += __popc(m);
    __syncwarp();
  }
  if (!a.xs) return;
  // 5. the CTA's routed rows of x into their sorted positions, every thread on
  //    16-byte chunks of the chunk's rows (the positions are this CTA's own writes)
  __syncthreads();
  const int chunks = a.K / 8;
  uint4* dst = reinterpret_cast<uint4*>(a.xs);
  for (int64_t i = tid; i < (int64_t)(q1 - q0) * chunks; i += kAlignThreads) {
    const int p = q0 + (int)(i / chunks), cc = (int)(i % chunks);
    const int pos = a.pair_pos[p];
    if (pos < 0) continue;
    const int e = a.perm13 ? local_expert(topk_ids, p, expert_base, E) : 0;
    dst[(int64_t)pos * chunks + cc] = x_chunk_f16(a, p / a.top_k, e, cc);
  }
}

// Number of CTAs that take part in the alignment.
__host__ __device__ inline int align_ctas(int pairs) {
  if (pairs <= kAlignFew) return 1;
  const int c = (pairs + kAlignChunk - 1) / kAlignChunk;
  return c > kAlignMaxCtas ? kAlignMaxCtas : c;
}

// CTAs that align when they also copy the routed rows: enough that each moves
// about 64 KB of rows, up to one per SM, and never fewer than the alignment
// alone takes (more chunks, each CTA still counting every id).
int align_copy_ctas(int pairs, int K, int sms) {
  if (pairs <= kAlignFew) return 1;
  const int64_t want = ((int64_t)pairs * K * 2 + (64 << 10) - 1) / (64 << 10);
  const int base = align_ctas(pairs);
  const int64_t c = want < sms ? want : sms;
  return c > base ? (int)c : base;
}

__global__ void __launch_bounds__(kAlignThreads, 1) prologue_kernel(const __grid_constant__ PrologueArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  grid_dependency_wait();
  grid_dependents_launch();
  if (a.topk_ids) {
    const int G = a.align_ctas > 0 ? a.align_ctas : align_ctas(a.pairs);
    if ((int)blockIdx.x < G) {
      if (a.pairs <= kAlignFew) align_few(a);
      else align_many(a, G, blockIdx.x, smem);
    }
  }
  // header words and activations, spread over every CTA
  // (8 bf16 -> 8 fp16 per 16-byte chunk: exact inside the fp16 range, beyond it infinity)
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = tid; i < a.zero_words; i += nthreads) a.zero[i] = 0u;
  if (!a.x) return;
  const int chunks = a.K / 8;
  const uint4* src = reinterpret_cast<const uint4*>(a.x);
  if (a.xh) {  // x's own rows
    uint4* dst = reinterpret_cast<uint4*>(a.xh);
    for (int64_t i = tid; i < (int64_t)a.M * chunks; i += nthreads) {
      const uint4 v = src[i];
      dst[i] = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
    }
  }
  if (a.xs && !a.topk_ids) {  // sorted order from the caller's alignment (two launches back, complete)
    uint4* dst = reinterpret_cast<uint4*>(a.xs);
    const int64_t n_padded = min((int64_t)max(*a.given_n_padded, 0), a.cap);  // (the GEMMs report a bad one)
    for (int64_t i = tid; i < n_padded * chunks; i += nthreads) {
      const int64_t pos = i / chunks;
      const int c = (int)(i - pos * chunks);
      const int sid = a.given_sorted[pos];
      if ((unsigned)sid >= (unsigned)a.pairs) continue;  // padding (or an id no pair has)
      int e = 0;
      if (a.perm13) {
        e = a.given_expert_ids[pos / a.block_m];
        if ((unsigned)e >= (unsigned)a.E) continue;  // (the GEMMs skip and report the block)
      }
      dst[i] = x_chunk_f16(a, sid / a.top_k, e, c);
    }
  }
}

cudaError_t launch_prologue(const PrologueArgs& a, int sms, cudaStream_t st) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)(((size_t)kAlignWarps * (kAlignMaxExperts + 1) + 3 * (size_t)kAlignMaxExperts) * 4));
    if (err != cudaSuccess) return err;
    configured[dev] = true;
  }
  int grid = 1;
  size_t smem = 0;
  if (a.topk_ids) {
    grid = a.align_ctas > 0 ? a.align_ctas : align_ctas(a.pairs);
    if (a.pairs > kAlignFew) smem = ((size_t)kAlignWarps * (a.E + 1) + 3 * (size_t)a.E) * 4;
  }
  int64_t work = a.zero_words;
  if (a.x && a.xh) work = std::max<int64_t>(work, (int64_t)a.M * (a.K / 8));
  if (a.x && a.xs && !a.topk_ids) work = std::max<int64_t>(work, a.cap * (a.K / 8));
  int64_t conv = (work + kAlignThreads - 1) / kAlignThreads;
  if (conv > 2 * (int64_t)sms) conv = 2 * (int64_t)sms;
  if (conv > grid) grid = (int)conv;
  return launch_dependent(prologue_kernel, dim3(grid), dim3(kAlignThreads), smem, st, a);
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
  PrologueArgs a{};
  // (an empty batch still writes n_padded = 0 and the sentinel tail; the ids are never read)
  a.topk_ids = topk_ids ? topk_ids : reinterpret_cast<const int32_t*>(n_padded);
  a.pairs = M * top_k;
  a.expert_base = expert_base;
  a.E = num_experts;
  a.block_m = block_m;
  a.cap = moe_align_capacity(M, top_k, num_experts, block_m);
  a.sorted_ids = sorted_ids;
  a.expert_ids = expert_ids;
  a.n_padded = n_padded;
  return launch_prologue(a, 0, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
