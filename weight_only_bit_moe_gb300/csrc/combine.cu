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
// One CTA per token; y is fp32.  When GEMM2 ran split-K the combine also
// finishes GEMM2: it sums the fp32 partial slices in split order and applies the
// global scale and bias -- what GEMM2's own epilogue does otherwise.
#include <cuda_runtime.h>
#include <stdint.h>

#include "combine.cuh"

namespace moe {

constexpr int kCombineThreads = 256;
constexpr int kMaxTopK = 16;

__device__ __forceinline__ float pair_y(const CombineArgs& c, int split, int pair, int e, int col) {
  if (split == 1) return c.y[(int64_t)pair * c.K + col];
  const int pos = c.inv_pos[pair];
  float acc = 0.f;
  for (int s = 0; s < split; ++s) acc += __ldcg(c.partial + ((int64_t)s * c.split_rows + pos) * c.K + col);
  const float b = c.b2 ? bf16_bits_to_float(c.b2[(int64_t)e * c.Kpad2 + col]) : 0.f;
  return acc * c.gs2[e] + b;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ CombineArgs c) {
  __shared__ int s_e[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  __shared__ float s_red[kCombineThreads / 32][kMaxTopK];
  __shared__ float s_inv[kMaxTopK];
  const int t = blockIdx.x, tid = threadIdx.x;
  const int k = c.top_k;
  if (tid < k) {
    const int e = c.topk_ids[(int64_t)t * k + tid] - c.expert_base;
    s_e[tid] = (e >= 0 && e < c.E) ? e : -1;
    s_w[tid] = c.topk_weights[(int64_t)t * k + tid];
  }
  __syncthreads();
  const int split = *c.split_used;
  if (c.post_norm_w) {
    float ss[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) ss[j] = 0.f;
    for (int col = tid; col < c.K; col += kCombineThreads) {
      const float nw = round_bf16(1.0f + bf16_bits_to_float(c.post_norm_w[col]));
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k && s_e[j] >= 0) {
          const float z = pair_y(c, split, t * k + j, s_e[j], col) * nw;
          ss[j] += z * z;
        }
      }
    }
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      float v = ss[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_red[warp][j] = v;
    }
    __syncthreads();
    if (tid < k) {
      float v = 0.f;
      for (int w = 0; w < kCombineThreads / 32; ++w) v += s_red[w][tid];
      s_inv[tid] = 1.0f / sqrtf(v / (float)c.K + c.norm_eps);
    }
    __syncthreads();
  }
  for (int col = tid; col < c.K; col += kCombineThreads) {
    const float nw = c.post_norm_w ? round_bf16(1.0f + bf16_bits_to_float(c.post_norm_w[col])) : 1.0f;
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = s_e[j];
      if (e < 0) continue;
      const float y = pair_y(c, split, t * k + j, e, col);
      acc += c.post_norm_w ? s_w[j] * s_inv[j] * (y * nw) : s_w[j] * y;
    }
    c.out[(int64_t)t * c.K + col] = float_to_bf16_bits(c.rsf * acc);
  }
}

cudaError_t launch_combine(const CombineArgs& c, cudaStream_t st) {
  if (c.M == 0) return cudaSuccess;
  if (c.top_k > kMaxTopK) return cudaErrorInvalidValue;
  combine_kernel<<<c.M, kCombineThreads, 0, st>>>(c);
  return cudaPeekAtLastError();
}

}  // namespace moe
