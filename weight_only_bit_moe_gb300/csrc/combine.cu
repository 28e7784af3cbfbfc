// Top-k weighted combine, optionally through the post-expert RMSNorm.
//
//   plain:     out[t] = bf16(rsf * sum_j w[t,j] * y[t,j])   over local slots
//              (per-expert reference loop of test_fused_marlin_moe_large_non_ep_schedule,
//              "Marlin MoE kernel occupancy ..." (sglang PR #31552): the routed
//              output times topk_weights, index-added in fp32);
//   post-norm: z = y * nw, nw = bf16(fp32(1 + w_norm)), inv = 1/sqrt(mean(z^2) + eps),
//              out[t] = bf16(rsf * sum_j w[t,j] * inv_j * z_j)
//              ("013-moe-middle-tiles.py": _expert_norm_factors and
//              _expert_norm_sum, weight_first, eps 1e-8; non-local slots get
//              factor 0).
//
// y is fp32 (the expert outputs keep their accumulation precision: the top-k
// sum can cancel terms of a few hundred down to a fraction of one), summed in
// fp32.  Each thread owns 8 consecutive columns (two 16-byte loads per slot,
// one 16-byte bf16 store) and issues every slot's loads before it sums, in
// slot order.  Plain rows spread a token over a 2-D grid of 128-thread
// column blocks; post-norm rows take one CTA per token, wide enough to cover
// the row in one pass (up to 1024 threads), so the row reduction stays in it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "combine.cuh"

namespace moe {

constexpr int kCols = 8;  // columns per thread
constexpr int kMaxTopK = 16;

__device__ __forceinline__ void bf16x8(const uint16_t* p, float (&v)[8]) {  // 8 bf16 -> fp32
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// y of one pair at columns [col, col+8) (two 16-byte loads).  The loads are
// streaming (evict-first): y is read once, and the normal policy measured about
// 54 us slower on the int4 M=4096 combine (122 us).  Storing y with streaming
// stores in GEMM2 as well measured no different.
__device__ __forceinline__ void pair_y8(const CombineArgs& c, int pair, int col, float (&v)[8]) {
  const float4* p = reinterpret_cast<const float4*>(c.y + (int64_t)pair * c.K + col);
  const float4 a = __ldcs(p), b = __ldcs(p + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void norm_w8(const uint16_t* w, int col, float (&v)[8]) {
  bf16x8(w + col, v);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = round_bf16(1.0f + v[i]);  // bf16(fp32(1 + w))
}

__device__ __forceinline__ void store8(uint16_t* out, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = (uint32_t)float_to_bf16_bits(v[2 * i]) | ((uint32_t)float_to_bf16_bits(v[2 * i + 1]) << 16);
  *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
}

// blockIdx.x = token; plain rows: blockIdx.y = column block.
__global__ void __launch_bounds__(1024) combine_kernel(const __grid_constant__ CombineArgs c) {
  grid_dependency_wait();
  const int t = blockIdx.x, tid = threadIdx.x, nthreads = blockDim.x;
  const int k = c.top_k;
  int e[kMaxTopK];
  float w[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    e[j] = -1;
    w[j] = 0.f;
    if (j < k) {
      const int ej = c.topk_ids[(int64_t)t * k + j] - c.expert_base;
      if (ej >= 0 && ej < c.E) {
        e[j] = ej;
        w[j] = c.topk_weights[(int64_t)t * k + j];
      }
    }
  }
  uint16_t* orow = c.out + (int64_t)t * c.K;

  if (!c.post_norm_w) {
    for (int col = (blockIdx.y * nthreads + tid) * kCols; col < c.K; col += gridDim.y * nthreads * kCols) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j >= k) break;
        if (e[j] < 0) continue;
        float y[8];
        pair_y8(c, t * k + j, col, y);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += w[j] * y[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= c.rsf;
      store8(orow + col, acc);
    }
    return;
  }

  // post-expert norm: per-slot sum of squares over the whole row first
  __shared__ float s_red[1024 / 32][kMaxTopK];
  __shared__ float s_inv[kMaxTopK];
  float ss[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) ss[j] = 0.f;
  for (int col = tid * kCols; col < c.K; col += nthreads * kCols) {
    float nw[8];
    norm_w8(c.post_norm_w, col, nw);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= k) break;
      if (e[j] < 0) continue;
      float y[8];
      pair_y8(c, t * k + j, col, y);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float z = y[i] * nw[i];
        ss[j] += z * z;
      }
    }
  }
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    float v = ss[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_red[warp][j] = v;
  }
  __syncthreads();
  if (tid < kMaxTopK) {
    float v = 0.f;
    for (int i = 0; i < nwarps; ++i) v += s_red[i][tid];
    s_inv[tid] = 1.0f / sqrtf(v / (float)c.K + c.norm_eps);
  }
  __syncthreads();
  for (int col = tid * kCols; col < c.K; col += nthreads * kCols) {
    float nw[8];
    norm_w8(c.post_norm_w, col, nw);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= k) break;
      if (e[j] < 0) continue;
      float y[8];
      pair_y8(c, t * k + j, col, y);
      const float f = w[j] * s_inv[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f * (y[i] * nw[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= c.rsf;
    store8(orow + col, acc);
  }
}

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t st) {
  if (c.M == 0) return cudaSuccess;
  if (c.top_k > kMaxTopK || c.K % kCols) return cudaErrorInvalidValue;
  const int chunks = c.K / kCols;
  if (!c.post_norm_w) {  // plain rows: a 2-D grid of column blocks of up to 128 threads, none idle at small K
    const int threads = chunks < 128 ? (chunks + 31) / 32 * 32 : 128;
    return launch_dependent(combine_kernel, dim3(c.M, (chunks + threads - 1) / threads), dim3(threads), 0, st, c);
  }
  int threads = (chunks + 31) / 32 * 32;
  if (threads > 1024) threads = 1024;
  return launch_dependent(combine_kernel, dim3(c.M), dim3(threads), 0, st, c);
}

}  // namespace moe
