// Load-time repack of checkpoint expert weights into the tile-native layout
// described in common.cuh ("013-moe-middle-tiles.py", prepare():
// prepare_moe_nvfp4_layer_for_marlin; "SM120 MXFP4 MoE ... Marlin" (sglang
// PR #28231): deinterleave_moe_mxfp4_w13_for_marlin, _pad_w13 / _pad_w2; the
// INT4 zero points, g_idx / sort_indices and group sizes of fused_marlin_moe,
// "Marlin MoE kernel occupancy ..." (sglang PR #31552)).
//
// Every output byte is written by exactly one thread; reading the source is
// byte-gather work, so the kernels are simple and run once per layer.  Before
// the scales are written, one CTA per expert matrix finds the exponent range of
// its scales and the power-of-two shift that moves them into the fp16 operand
// window (common.cuh); the scales are stored shifted and the expert's epilogue
// factor carries the inverse power.
//
// Act-order banks: packed column k of an expert matrix holds the checkpoint's
// column sort_indices[k] (groups contiguous, group k / group_size), and w13's
// output features follow w2's sort order (feature f of the packed bank is the
// checkpoint's feature w2_sort_indices[f], gate, up and bias alike), so GEMM1
// writes the activations in the order GEMM2's packed columns read them.
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

struct RepackArgs {
  Layout L;
  int interleaved, has_b13, has_b2;
  const uint8_t* w13;
  const uint8_t* w13_s;
  const float* w13_gs;
  const uint16_t* b13;
  const uint8_t* w13_z;       // INT4 zero points [E, R, groups] (u8 or bf16), or NULL
  const int32_t* w13_gidx;    // act-order [E, K]
  const int32_t* w13_perm;    // act-order [E, K]
  const uint8_t* w2;
  const uint8_t* w2_s;
  const float* w2_gs;
  const uint16_t* b2;
  const uint8_t* w2_z;
  const int32_t* w2_gidx;     // [E, N]
  const int32_t* w2_perm;     // [E, N]
  uint8_t* out;
};

__device__ __forceinline__ bool int4_family(int fmt) { return fmt == MOE_W_INT4_U4B8 || fmt == kFmtInt4X; }

// Checkpoint feature of packed GEMM1 feature f of expert e (w2's sort order under act-order).
__device__ __forceinline__ int source_feature(const RepackArgs& a, int e, int f) {
  return a.L.act_order ? a.w2_perm[(int64_t)e * a.L.N + f] : f;
}

// Source row of tile row r of expert e for matrix `which` (0 = w13, 1 = w2), or
// -1 for a padding row.  Gated w13: half 0 = gate, half 1 = up; interleaved
// storage keeps gate i in row 2i and up i in row 2i+1.  Non-gated w13 tiles are
// 256 consecutive rows, like w2's.
__device__ __forceinline__ int source_row(const RepackArgs& a, int which, int e, int tile, int r) {
  const Layout& L = a.L;
  if (which == 0 && !L.gated) {
    const int f = tile * kTileRows + r;
    return f < L.N ? source_feature(a, e, f) : -1;
  }
  if (which == 0) {
    const int f = tile * 128 + (r & 127), half = r >> 7;
    if (f >= L.N) return -1;
    const int sf = source_feature(a, e, f);
    return a.interleaved ? 2 * sf + half : half * L.N + sf;
  }
  const int c = tile * kTileRows + r;
  return c < L.K ? c : -1;
}

// Checkpoint column of packed column k (reduction index) of expert e's matrix.
__device__ __forceinline__ int source_col(const RepackArgs& a, int which, int e, int k) {
  if (!a.L.act_order) return k;
  const int red = which ? a.L.N : a.L.K;
  return (which ? a.w2_perm : a.w13_perm)[(int64_t)e * red + k];
}

// Group of packed column k (contiguous after the act-order sort), and groups per row.
__device__ __forceinline__ int group_of(const Layout& L, int k) { return L.group > 0 ? k / L.group : 0; }
__device__ __forceinline__ int groups_per_row(const Layout& L, int red) { return L.group > 0 ? red / L.group : 1; }

__device__ __forceinline__ uint32_t zero_code(int fmt) { return int4_family(fmt) ? 8u : 0u; }

// Act-order banks: every packed column's checkpoint group must be its position's
// group (groups of group_size indices each); otherwise the blob is marked.
__global__ void repack_check_groups_kernel(RepackArgs a) {
  const Layout& L = a.L;
  const int64_t n13 = (int64_t)L.E * L.K, n2 = (int64_t)L.E * L.N;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < n13 + n2;
       u += (int64_t)gridDim.x * blockDim.x) {
    const int which = u >= n13;
    const int64_t v = which ? u - n13 : u;
    const int red = which ? L.N : L.K;
    const int e = (int)(v / red), k = (int)(v % red);
    const int32_t* perm = (which ? a.w2_perm : a.w13_perm) + (int64_t)e * red;
    const int32_t* gidx = (which ? a.w2_gidx : a.w13_gidx) + (int64_t)e * red;
    const int src = perm[k];
    if (src < 0 || src >= red || gidx[src] != group_of(L, k)) atomicOr(reinterpret_cast<unsigned*>(a.out), kFlagGroups);
  }
}

// Scale-exponent shift of one expert matrix: blockIdx.x = which * E + e.  The
// exponent of a finite nonzero INT4 scale is floor(log2 |s|); an MXFP4 scale's is
// its E8M0 byte (255, NaN, is skipped); NVFP4 needs no shift.  The shift d puts
// [lo + d, hi + d] inside the window, as close to 0 as possible; when the span is
// wider than the window it keeps the largest scales exact and flags the blob.
// INT4 with zero points (|q - z| up to 15) has a window one binade lower.
__global__ void __launch_bounds__(256) repack_shift_kernel(RepackArgs a) {
  const Layout& L = a.L;
  const int which = blockIdx.x / L.E, e = blockIdx.x % L.E;
  int32_t* shift = reinterpret_cast<int32_t*>(a.out + L.shift_off) + which * L.E + e;
  if (L.fmt == MOE_W_NVFP4) {
    if (threadIdx.x == 0) *shift = 0;
    return;
  }
  const int red = which ? L.N : L.K;
  const int64_t rows = which ? L.K : (L.gated ? 2 : 1) * (int64_t)L.N;
  const int64_t n = rows * groups_per_row(L, red);  // scales of one expert
  const uint8_t* src = which ? a.w2_s : a.w13_s;
  int lo = INT_MAX, hi = INT_MIN;
  const bool int4 = int4_family(L.fmt);
  if (int4) {
    const uint16_t* sp = reinterpret_cast<const uint16_t*>(src) + (int64_t)e * n;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t bits = sp[i];
      if ((bits & 0x7F80u) == 0x7F80u || (bits & 0x7FFFu) == 0) continue;  // inf, NaN, zero
      int ex;
      frexpf(bf16_bits_to_float((uint16_t)bits), &ex);  // |s| in [2^(ex-1), 2^ex)
      lo = min(lo, ex - 1);
      hi = max(hi, ex - 1);
    }
  } else {
    const uint8_t* sp = src + (int64_t)e * n;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      const int b = sp[i];
      if (b == 255) continue;
      lo = min(lo, b);
      hi = max(hi, b);
    }
  }
  __shared__ int s_lo[8], s_hi[8];
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if ((threadIdx.x & 31) == 0) {
    s_lo[threadIdx.x >> 5] = lo;
    s_hi[threadIdx.x >> 5] = hi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      lo = min(lo, s_lo[w]);
      hi = max(hi, s_hi[w]);
    }
    const int wmin = int4 ? kInt4ExpMin : kE8m0Min;
    const int wmax = int4 ? (L.zero_kind ? kInt4ExpMax - 1 : kInt4ExpMax) : kE8m0Max;
    int d = 0;
    if (lo <= hi) {
      const int dlo = wmin - lo, dhi = wmax - hi;
      if (dlo <= dhi) {
        d = min(max(0, dlo), dhi);
      } else {
        d = dhi;
        // plain INT4 applies scales in fp16 only on the tcgen05 path; MXFP4 and the
        // INT4 entries of zero-point / small-group banks on both
        atomicOr(reinterpret_cast<unsigned*>(a.out), L.fmt == MOE_W_INT4_U4B8 ? kFlagInt4Window : kFlagFp16Window);
      }
    }
    *shift = d;
  }
}

// One thread per 16-byte unit of packed codes: unit (e, tile, stage, j, r).
__global__ void repack_codes_kernel(RepackArgs a, int which) {
  const Layout& L = a.L;
  const int T = which ? L.T2 : L.T1, S = which ? L.S2 : L.S1;
  const int red = which ? L.N : L.K;  // real reduction length
  const int64_t units = (int64_t)L.E * T * S * 512;
  const int64_t tile_bytes = which ? L.tile2_bytes : L.tile1_bytes;
  const uint8_t* src = which ? a.w2 : a.w13;
  const int64_t src_row_bytes = red / 2;
  const int64_t src_rows = which ? L.K : (L.gated ? 2 : 1) * (int64_t)L.N;
  const bool int4 = int4_family(L.fmt);
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(u % 256);
    const int j = (int)((u / 256) % 2);
    const int s = (int)((u / 512) % S);
    const int tile = (int)((u / (512LL * S)) % T);
    const int e = (int)(u / (512LL * S * T));
    const int row = source_row(a, which, e, tile, r);
    const uint8_t* srow = row >= 0 ? src + ((int64_t)e * src_rows + row) * src_row_bytes : nullptr;
    uint32_t words[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      // word v = 2t + h of the row's stage holds pairs starting at 32h + 2t + 8p
      const int v = 4 * j + w, t = v >> 1, h = v & 1;
      uint32_t word = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int k = s * kStageK + 32 * h + 2 * t + 8 * p + e2;
          uint32_t q = zero_code(L.fmt);
          if (srow && k < red) {
            const int c = source_col(a, which, e, k);
            const uint8_t b = srow[c >> 1];
            q = (c & 1) ? (b >> 4) : (b & 15u);
          }
          // INT4: first element of pair p at bits 4p, second at 16 + 4p (mask-and-magic
          // pairs); FP4: pair p in byte p, first element in the low nibble, as the
          // hardware E2M1x2 conversion reads them
          const int pos = int4 ? (e2 ? 16 + 4 * p : 4 * p) : 8 * p + 4 * e2;
          word |= q << pos;
        }
      words[w] = word;
    }
    uint8_t* dst = a.out + (which ? L.w2_off : L.w13_off) + ((int64_t)e * T + tile) * tile_bytes +
                   stage_offset(L, s) + (stage_has_scales(L, s) ? L.scale_bytes : 0) + ((int64_t)j * 256 + r) * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
  }
}

// bf16 scale times 2^d (exact while the result is a normal bf16, which the window guarantees).
__device__ __forceinline__ float shifted_scale(uint16_t bits, int d) {
  const float v = bf16_bits_to_float(bits);
  if ((bits & 0x7F80u) == 0x7F80u || (bits & 0x7FFFu) == 0) return v;
  return ldexpf(v, d);
}

// INT4X entry of one row and 32-element half stage: f16 m (the shifted scale)
// and f16 x (1024 + z, 1032 without zero points, or -z * m for float zeros).
__device__ __forceinline__ uint32_t int4x_entry(const RepackArgs& a, int which, int e, int row, int red, int k0,
                                                int d) {
  const Layout& L = a.L;
  // padding (codes 8): m = 1 and a zero term that makes the weight 0 -- x = 1032, or o = -8
  // for float zero points (w = q * m + o)
  if (row < 0 || k0 >= red) return 0x3C00u | ((L.zero_kind == 2 ? 0xC800u : 0x6408u) << 16);
  const int gpr = groups_per_row(L, red);
  const int64_t rows = which ? L.K : (L.gated ? 2 : 1) * (int64_t)L.N;
  const int64_t idx = ((int64_t)e * rows + row) * gpr + group_of(L, k0);
  const uint16_t* sp = reinterpret_cast<const uint16_t*>(which ? a.w2_s : a.w13_s);
  const float sv = shifted_scale(sp[idx], d);
  const uint16_t m = __half_as_ushort(__float2half_rn(sv));
  uint16_t x = 0x6408;  // 1032: uint4b8
  if (L.zero_kind == 1) {
    x = __half_as_ushort(__float2half_rn(1024.0f + (float)(which ? a.w2_z : a.w13_z)[idx]));
  } else if (L.zero_kind == 2) {
    const float z = bf16_bits_to_float(reinterpret_cast<const uint16_t*>(which ? a.w2_z : a.w13_z)[idx]);
    x = __half_as_ushort(__float2half_rn(-z * sv));  // z * s exact in fp32 (8 + 8 bits), one rounding
  }
  return (uint32_t)m | ((uint32_t)x << 16);
}

// One thread per (e, tile, scale chunk, row): its scales (or INT4X entries).
__global__ void repack_scales_kernel(RepackArgs a, int which) {
  const Layout& L = a.L;
  const int T = which ? L.T2 : L.T1, S = which ? L.S2 : L.S1;
  const int chunks = S / L.period;
  const int red = which ? L.N : L.K;
  const int groups = groups_per_row(L, red);  // real groups per source row
  const int64_t total = (int64_t)L.E * T * chunks * 256;
  const int64_t tile_bytes = which ? L.tile2_bytes : L.tile1_bytes;
  const uint8_t* src = which ? a.w2_s : a.w13_s;
  const int64_t src_rows = which ? L.K : (L.gated ? 2 : 1) * (int64_t)L.N;
  const int sb = int4_family(L.fmt) ? 2 : 1;  // source bytes per scale
  const int32_t* shift = reinterpret_cast<const int32_t*>(a.out + L.shift_off) + which * L.E;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(u % 256);
    const int q = (int)((u / 256) % chunks);
    const int tile = (int)((u / (256LL * chunks)) % T);
    const int e = (int)(u / (256LL * chunks * T));
    const int row = source_row(a, which, e, tile, r);
    const uint8_t* srow = row >= 0 ? src + ((int64_t)e * src_rows + row) * groups * sb : nullptr;
    uint8_t* dst = a.out + (which ? L.w2_off : L.w13_off) + ((int64_t)e * T + tile) * tile_bytes +
                   stage_offset(L, q * L.period);
    const int d = shift[e];
    if (L.fmt == kFmtInt4X) {  // stage q: entries of K halves [64q, 64q+32) and [64q+32, 64q+64)
      uint2 v;
      v.x = int4x_entry(a, which, e, row, red, 64 * q, d);
      v.y = int4x_entry(a, which, e, row, red, 64 * q + 32, d);
      reinterpret_cast<uint2*>(dst)[r] = v;
    } else if (L.fmt == MOE_W_INT4_U4B8) {  // stages 2q, 2q+1: K [128q, 128q+128) in one group
      uint16_t v = 0x3F80;                 // 1.0 for padding
      if (srow && 128 * q < red) v = float_to_bf16_bits(shifted_scale(reinterpret_cast<const uint16_t*>(srow)[group_of(L, 128 * q)], d));
      reinterpret_cast<uint16_t*>(dst)[r] = v;
    } else if (L.fmt == MOE_W_MXFP4) {  // groups 2q, 2q+1 (32 each)
      uint32_t v = 0;
      for (int g = 0; g < 2; ++g) {
        const int gi = 2 * q + g;
        uint32_t b = 127;  // 2^0 for padding
        if (srow && gi < groups) {
          b = srow[gi];
          if (b != 255u) b = (uint32_t)min(max((int)b + d, 0), 254);  // 2^d; NaN stays NaN
        }
        v |= b << (8 * g);
      }
      reinterpret_cast<uint16_t*>(dst)[r] = (uint16_t)v;
    } else {  // NVFP4: groups 4q .. 4q+3 (16 each)
      uint32_t v = 0;
      for (int g = 0; g < 4; ++g) {
        const int gi = 4 * q + g;
        uint32_t b = 0x38;  // 1.0 for padding
        if (srow && gi < groups) b = srow[gi];
        v |= b << (8 * g);
      }
      reinterpret_cast<uint32_t*>(dst)[r] = v;
    }
  }
}

// Bias rows (deinterleaved, in the packed feature order, zero padded), global
// scales and, for act-order banks, w13's column order for the forward.
__global__ void repack_misc_kernel(RepackArgs a) {
  const Layout& L = a.L;
  const int halves = L.gated ? 2 : 1;  // gate and up rows, or h rows only
  const int64_t n13 = a.has_b13 ? (int64_t)L.E * halves * L.Npad : 0;
  const int64_t n2 = a.has_b2 ? (int64_t)L.E * L.Kpad2 : 0;
  const int64_t ngs = L.E;
  const int64_t nperm = L.act_order ? (int64_t)L.E * L.K : 0;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < n13 + n2 + ngs + nperm;
       u += (int64_t)gridDim.x * blockDim.x) {
    if (u < n13) {
      const int f = (int)(u % L.Npad), half = (int)((u / L.Npad) % halves);
      const int e = (int)(u / ((int64_t)halves * L.Npad));
      uint16_t v = 0;
      if (f < L.N) {
        const int sf = source_feature(a, e, f);
        const int row = a.interleaved ? 2 * sf + half : half * L.N + sf;
        v = a.b13[(int64_t)e * halves * L.N + row];
      }
      reinterpret_cast<uint16_t*>(a.out + L.b13_off)[u] = v;
    } else if (u < n13 + n2) {
      const int64_t v2 = u - n13;
      const int c = (int)(v2 % L.Kpad2), e = (int)(v2 / L.Kpad2);
      reinterpret_cast<uint16_t*>(a.out + L.b2_off)[v2] = c < L.K ? a.b2[(int64_t)e * L.K + c] : (uint16_t)0;
    } else if (u < n13 + n2 + ngs) {
      const int e = (int)(u - n13 - n2);
      const int32_t* shift = reinterpret_cast<const int32_t*>(a.out + L.shift_off);
      float g13 = ldexpf(1.0f, -shift[e]), g2 = ldexpf(1.0f, -shift[L.E + e]);  // undo the scale shift
      if (L.fmt == MOE_W_NVFP4) {  // no shift for NVFP4 (every E4M3 scale is exact)
        g13 = a.w13_gs[e];
        g2 = a.w2_gs[e];
      }
      if (!int4_family(L.fmt)) {
        g13 *= kFp4Unscale;
        g2 *= kFp4Unscale;
      }
      reinterpret_cast<float*>(a.out + L.gs13_off)[e] = g13;
      reinterpret_cast<float*>(a.out + L.gs2_off)[e] = g2;
    } else {
      const int64_t v = u - n13 - n2 - ngs;
      reinterpret_cast<int32_t*>(a.out + L.perm13_off)[v] = a.w13_perm[v];
    }
  }
}

}  // namespace moe

using namespace moe;

extern "C" int64_t moe_repack_size(const moe_layer_desc* desc) {
  Layout L;
  if (!desc || !make_layout(*desc, &L)) return -1;
  return L.total;
}

extern "C" int moe_repack_weights_ex(const moe_layer_desc* desc, const moe_repack_tensors* t, void* packed,
                                     void* stream) {
  Layout L;
  if (!desc || !t || !make_layout(*desc, &L)) return MOE_ERR_INVALID;
  if (!t->w13 || !t->w13_s || !t->w2 || !t->w2_s || !packed) return MOE_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(packed) & 255) != 0) return MOE_ERR_INVALID;
  if (desc->fmt == MOE_W_NVFP4 && (!t->w13_gs || !t->w2_gs)) return MOE_ERR_INVALID;
  if ((desc->has_bias13 && !t->b13) || (desc->has_bias2 && !t->b2)) return MOE_ERR_INVALID;
  if (L.zero_kind && (!t->w13_zeros || !t->w2_zeros)) return MOE_ERR_INVALID;
  if (L.act_order && (!t->w13_g_idx || !t->w13_sort_indices || !t->w2_g_idx || !t->w2_sort_indices))
    return MOE_ERR_INVALID;
  // (Interleaved storage needs an even row count and scale / bias rows matching
  // the weight rows; here every count derives from desc -- 2N rows -- so only
  // the gating rule can be broken, and make_layout rejects interleaved
  // non-gated banks.)
  RepackArgs a;
  a.L = L;
  a.interleaved = desc->w13_interleaved != 0;
  a.has_b13 = desc->has_bias13 != 0;
  a.has_b2 = desc->has_bias2 != 0;
  a.w13 = static_cast<const uint8_t*>(t->w13);
  a.w13_s = static_cast<const uint8_t*>(t->w13_s);
  a.w13_gs = t->w13_gs;
  a.b13 = static_cast<const uint16_t*>(t->b13);
  a.w13_z = static_cast<const uint8_t*>(t->w13_zeros);
  a.w13_gidx = t->w13_g_idx;
  a.w13_perm = t->w13_sort_indices;
  a.w2 = static_cast<const uint8_t*>(t->w2);
  a.w2_s = static_cast<const uint8_t*>(t->w2_s);
  a.w2_gs = t->w2_gs;
  a.b2 = static_cast<const uint16_t*>(t->b2);
  a.w2_z = static_cast<const uint8_t*>(t->w2_zeros);
  a.w2_gidx = t->w2_g_idx;
  a.w2_perm = t->w2_sort_indices;
  a.out = static_cast<uint8_t*>(packed);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(packed, 0, 256, st) != cudaSuccess) return MOE_ERR_CUDA;  // header
  const int threads = 256, blocks = 152 * 16;
  if (L.act_order) repack_check_groups_kernel<<<blocks, threads, 0, st>>>(a);
  repack_shift_kernel<<<2 * L.E, threads, 0, st>>>(a);  // before the scales and the global factors
  for (int which = 0; which < 2; ++which) {
    repack_codes_kernel<<<blocks, threads, 0, st>>>(a, which);
    repack_scales_kernel<<<blocks, threads, 0, st>>>(a, which);
  }
  repack_misc_kernel<<<blocks, threads, 0, st>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_repack_weights(const moe_layer_desc* desc, const void* w13, const void* w13_s,
                                  const float* w13_gs, const void* b13, const void* w2, const void* w2_s,
                                  const float* w2_gs, const void* b2, void* packed, void* stream) {
  moe_repack_tensors t = {};
  t.w13 = w13;
  t.w13_s = w13_s;
  t.w13_gs = w13_gs;
  t.b13 = b13;
  t.w2 = w2;
  t.w2_s = w2_s;
  t.w2_gs = w2_gs;
  t.b2 = b2;
  return moe_repack_weights_ex(desc, &t, packed, stream);
}
