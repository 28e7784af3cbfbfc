// Per-token -> per-tensor FP8 requantisation of an expert-major activation
// payload ("W4AFP8 requant ..." (sglang PR #35760):
// _fp8_per_token_quant_to_per_tensor_quant_kernel, _requant_row and
// requant_launch_geometry).  Expert e holds max_m row slots of K FP8 (E4M3)
// values, of which its first masked_m[e] are valid; each valid row carries one
// fp32 scale per 128-wide (group-wide) column group, addressed through
// strides so that the column-major layout of the low-latency dispatcher
// (entry (e, g, m) at e*se + g*sg + m) and a row-major one are both read in
// place.  Every valid element becomes
//     out = e4m3_rn_satfinite(fp32(fp32(x * s) * r)),   r = fp32(1 / S),
// two fp32 multiplies per element as the page describes; invalid rows are not
// touched.
//
// GB300 design.  The job is a pure stream (one byte in, one byte out, a
// scale per 128), so the kernel is shaped for HBM: each warp owns one valid
// row at a time and each lane moves 16-byte chunks (16 elements of one
// group), eight chunks' loads in flight before their math (4 KB per warp), one
// scalar scale load per chunk (the 8 lanes of a group read the same address);
// registers are capped so that three CTAs (24 row streams) share an SM.  The rows are
// scheduled flat: each CTA scans masked_m into row offsets in shared memory
// and maps a flat row index to (expert, row) by binary search, so a hot expert
// spreads over the whole grid and empty experts cost nothing -- the page's two
// phases (per-expert rows up to a cap, then overflow rows shared through a
// prefix sum) with the cap at zero.  The launch geometry only sizes the grid
// from the caller's row estimate; any geometry writes the same bytes.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "../../include/moe_requant.h"

namespace moe {

constexpr int kRqThreads = 256;             // 8 warps, one row each at a time
constexpr int kRqWarps = kRqThreads / 32;
constexpr int kRqMaxExperts = 1024;
constexpr int kRqMaxCtasPerSm = 8;          // 64 warps of row streams per SM at most
constexpr int kRqResident = 3;              // CTAs that fit on an SM at once (registers capped for it)
constexpr int kRqChunksPerLane = 8;         // 4 KB of a row in flight per warp per pass

struct RequantArgs {
  const uint8_t* x;
  const float* scale;
  int64_t se, sg, sm;
  const int32_t* masked_m;
  const float* tensor_scale;
  uint8_t* out;
  int E, max_m, K, group;
};

// 16 E4M3 values -> times s, then times r (fp32, rounded after each) -> E4M3.
__device__ __forceinline__ uint4 requant16(uint4 v, float s, float r) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t packed = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i] >> (16 * h)) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);  // exact
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      float2 t;
      t.x = __fmul_rn(__fmul_rn(f.x, s), r);
      t.y = __fmul_rn(__fmul_rn(f.y, s), r);
      const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(t, __NV_SATFINITE, __NV_E4M3);
      packed |= (uint32_t)q << (16 * h);
    }
    o[i] = packed;
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(kRqThreads, kRqResident) requant_kernel(const __grid_constant__ RequantArgs a) {
  __shared__ int row_start[kRqMaxExperts + 1];  // flat index of each expert's first valid row
  __shared__ int warp_tot[kRqWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // --- prefix over the experts' valid rows (clamped to [0, max_m])
  constexpr int kPer = (kRqMaxExperts + kRqThreads - 1) / kRqThreads;
  int cnt[kPer], run = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid * kPer + i;
    const int v = e < a.E ? min(max(a.masked_m[e], 0), a.max_m) : 0;
    cnt[i] = v;
    run += v;
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  int pos = before + incl - run;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid * kPer + i;
    if (e <= a.E) row_start[e] = pos;  // (e == E: the total)
    pos += cnt[i];
  }
  if (tid == kRqThreads - 1) row_start[kRqMaxExperts] = pos;  // the total when E is the maximum
  __syncthreads();
  const int total = row_start[a.E];
  const float r = __frcp_rn(*a.tensor_scale);  // fp32(1 / S), correctly rounded
  const int chunks = a.K / 16;
  const int gshift = 31 - __clz(a.group);      // group is a power of two

  for (int f = blockIdx.x * kRqWarps + warp; f < total; f += gridDim.x * kRqWarps) {
    // expert of flat row f: the last e with row_start[e] <= f
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (row_start[mid] <= f) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo, m = f - row_start[e];
    const int64_t row = (int64_t)e * a.max_m + m;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + row * a.K);
    uint4* dst = reinterpret_cast<uint4*>(a.out + row * a.K);
    const float* srow = a.scale + e * a.se + (int64_t)m * a.sm;
    for (int c0 = 0; c0 < chunks; c0 += 32 * kRqChunksPerLane) {
      uint4 v[kRqChunksPerLane];
      float s[kRqChunksPerLane];
#pragma unroll
      for (int i = 0; i < kRqChunksPerLane; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < chunks) {
          v[i] = __ldcs(src + c);                           // read once: stream past L2
          s[i] = __ldg(srow + (int64_t)((c * 16) >> gshift) * a.sg);
        }
      }
#pragma unroll
      for (int i = 0; i < kRqChunksPerLane; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < chunks) __stcs(dst + c, requant16(v[i], s[i], r));
      }
    }
  }
}

// Largest power of two <= v (v >= 1).
static int floor_pow2(int v) {
  int p = 1;
  while (p <= v / 2) p *= 2;
  return p;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_requant_launch_geometry(int num_experts, int K, int expected_rows, int sm_count, int* ctas,
                                           int* threads) {
  if (num_experts <= 0 || K <= 0 || sm_count <= 0 || !ctas || !threads) return MOE_ERR_INVALID;
  const int full = sm_count * kRqMaxCtasPerSm;
  int c = full;  // no estimate: the whole machine, rows spread by the flat schedule
  if (expected_rows > 0) {
    // one warp per row of the estimate, rounded down to a power of two so that an
    // estimate rounded up by its producer ((rows + E) / E) does not grow the grid
    const int64_t rows = (int64_t)num_experts * floor_pow2(expected_rows);
    const int64_t want = (rows + kRqWarps - 1) / kRqWarps;
    c = (int)(want < full ? want : full);
    if (c < 1) c = 1;
  }
  *ctas = c;
  *threads = kRqThreads;
  return MOE_OK;
}

extern "C" int moe_requant_fp8(const void* x, const float* scale, int64_t scale_stride_e,
                               int64_t scale_stride_g, int64_t scale_stride_m, const int32_t* masked_m,
                               int num_experts, int max_m, int K, int group, const float* tensor_scale, void* out,
                               int expected_rows, void* stream) {
  if (num_experts <= 0 || num_experts > kRqMaxExperts || max_m < 0 || K <= 0) return MOE_ERR_INVALID;
  if (group < 16 || (group & (group - 1)) || K % group) return MOE_ERR_INVALID;
  if (!scale || !masked_m || !tensor_scale || !out || (!x && max_m > 0)) return MOE_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15) return MOE_ERR_INVALID;
  if (max_m == 0) return MOE_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
  int ctas = 0, threads = 0;
  moe_requant_launch_geometry(num_experts, K, expected_rows, sms, &ctas, &threads);
  RequantArgs a;
  a.x = static_cast<const uint8_t*>(x);
  a.scale = scale;
  a.se = scale_stride_e;
  a.sg = scale_stride_g;
  a.sm = scale_stride_m;
  a.masked_m = masked_m;
  a.tensor_scale = tensor_scale;
  a.out = static_cast<uint8_t*>(out);
  a.E = num_experts;
  a.max_m = max_m;
  a.K = K;
  a.group = group;
  requant_kernel<<<ctas, threads, 0, (cudaStream_t)stream>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
