// Grouped W4A16 GEMM for small token blocks (block_m = 8, 16 or 32): the
// decode and small-batch shapes, where every routed expert's weights are
// streamed from HBM once per token block and the layer is bound by HBM
// bandwidth, not by tensor math.
//
// Same function as moe_gemm_kernel (gemm.cuh) -- GEMM1 with the fused gated
// or relu^2 activation, or GEMM2 -- on the same packed layout, built for a
// different bottleneck:
//
//   * weights reach registers, never tensor memory: the consumer warps (16
//     for 8-token blocks, 8 otherwise) each own 16 or 32 rows of the 256-row
//     tile, load their 4-bit codes from the staged chunk (one 8-byte load per
//     row and stage, in the register-fragment order the repack writes),
//     dequantise them in registers to fp16 and feed them as the A operand of
//     m16n8k16 tensor-core instructions; tokens are the 8-wide N side.  At
//     8..32 tokens a 64-K stage costs 128..512 tensor cycles per SM, under the
//     ~380 cycles HBM needs to deliver it, and no cross-warp handoff sits
//     between dequantisation and the MMA;
//   * gated GEMM1 pairs gate and up rows inside each 16-row fragment (rows
//     0..7 gate features, rows 8..15 the same up features), so the activation
//     is applied in the registers that hold both accumulators; non-gated GEMM1
//     and GEMM2 take 16 consecutive rows per fragment;
//   * one producer thread streams 4-stage chunks (~34 KB of packed codes and
//     scales in one bulk copy, plus the block's activation rows for those
//     stages in one 3-D TMA tile) into a 4..6-deep ring; large copies keep a
//     single issuing thread at HBM speed;
//   * the persistent grid walks the items (tile, token block) in the order of
//     moe_gemm_kernel (tile fastest), but the work is divided evenly: the
//     items' scale periods, laid end to end, are cut into one contiguous range
//     per CTA (stream-K).  An item cut between CTAs is finished by the last of
//     them to arrive, which sums the fp32 partials of its segments in CTA
//     order (bitwise reproducible, no spinning).  Decode shapes rarely fill a
//     whole number of waves, and this keeps every SM streaming to the end.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "gemm.cuh"

namespace moe {

constexpr int kSmallChunk = 4;  // 64-K stages per TMA chunk
// Consumer warps per CTA: sixteen of one 16-row fragment each for 8-token
// blocks and for GEMM2's 16-token blocks (the lightest per-byte work, where
// latency hiding needs the warps), eight of two fragments otherwise (16-token
// GEMM1 measured slower with sixteen: its gated fragments keep more state).
template <int BN, int STAGE>
struct SmallCfg {
  static constexpr int kConsumerWarps = (BN == 8 || (BN <= 32 && STAGE == kGemm2)) ? 16 : 8;
  static constexpr int kMI = kTileRows / 16 / kConsumerWarps;  // 16-row fragments per consumer warp
  static constexpr int kThreads = (1 + kConsumerWarps) * 32;
};

template <int BN, int FMT>
struct SmallSmem {
  static constexpr int kWBytes = PackedFmt<FMT>::kSlotBytes(kSmallChunk);  // codes + scale blocks of a chunk
  static constexpr int kBBytes = kSmallChunk * BN * 128;  // activation rows of a chunk, [stage][row][64]
  static constexpr int kSlotBytes = kWBytes + kBBytes;
  static constexpr int kFit = (kSmemBudget - 2048) / kSlotBytes;
  static constexpr int kSlots = kFit > 6 ? 6 : kFit;
  static constexpr int kBar = kSlots * kSlotBytes;
  static constexpr int kMisc = kBar + 2 * kSlots * 8;
  static constexpr int kRows = kMisc + 64;  // GEMM1 token rows: the current item's, then one set per slot
  static constexpr int kBytes = kRows + (1 + kSlots) * 32 * 4;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSlots >= 4, "ring too shallow");
  static_assert(kAlloc <= 232448, "shared memory over the per-CTA limit");
  static_assert(kBBytes % 1024 == 0 && kWBytes % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
};

// Work division.  W scale periods in all (items x periods per item, item w =
// block * T + tile); CTA c < G takes periods [c W / G, (c + 1) W / G), so
// every CTA below G has at least one period (G <= W).  Three cases, by the
// item count (base) against the grid:
//   * below one wave, G = base * S: each item's K is split S ways (one segment
//     per CTA; S weighs the shorter streams against writing and summing S
//     partials, in 1/8-stage units);
//   * whole items would leave over 20% of the grid's item slots idle and the
//     items are long (>= 32 stages): G = the grid, items cut where the ranges
//     fall (measured faster on GB300 for such shapes);
//   * otherwise, for 32-token blocks, and whenever the workspace holds no
//     partial area (max_split <= 1): whole items round-robin (a partly filled last wave of
//     whole items measured faster than cut items there -- the SMs of a partial
//     wave take a larger share of HBM).
struct SmallPlan {
  int nb, T, U;  // valid blocks, tiles, scale periods per item
  int G;         // CTAs with work (stream-K)
  int64_t W;
  bool streamk;
};

__device__ __forceinline__ SmallPlan make_plan_small(const GemmArgs& g, bool gemm1, int bn) {
  SmallPlan p;
  p.nb = valid_blocks(g);
  p.T = gemm1 ? g.L.T1 : g.L.T2;
  p.U = (gemm1 ? g.L.S1 : g.L.S2) / g.L.period;
  p.W = (int64_t)p.T * p.nb * p.U;
  p.streamk = false;
  p.G = 0;
  const int base = p.T * p.nb;
  const int grid = (int)gridDim.x;
  if (base <= 0 || g.max_split <= 1 || bn >= 32) return p;
  if (base < grid) {
    const int per = g.L.period * 8;
    int best = p.U * per + bn, S = 1;
    const int smax = min(grid / base, p.U);
    for (int s = 2; s <= smax; ++s) {
      const int cost = ((p.U + s - 1) / s) * per + bn + s * bn;
      if (cost < best) { best = cost; S = s; }
    }
    if (S > 1) {
      p.streamk = true;
      p.G = base * S;
      return p;
    }
  }
  const int waves = (base + grid - 1) / grid;
  if (5 * base < 4 * waves * grid && p.U * g.L.period >= 32) {
    p.streamk = true;
    p.G = (int)(p.W < (int64_t)grid ? p.W : (int64_t)grid);
  }
  return p;
}
__device__ __forceinline__ int64_t sk_lo(const SmallPlan& p, int c) { return (int64_t)c * p.W / p.G; }
// The CTA whose range holds period u: the largest c with sk_lo(c) <= u.
__device__ __forceinline__ int sk_owner(const SmallPlan& p, int64_t u) {
  return (int)(((u + 1) * p.G - 1) / p.W);
}

// This CTA's segments in order: item w, periods [u0, u1) of it; `first` marks
// the segment that opens the CTA's range (its partial slot 0; a later cut
// segment, the range's last, uses slot 1).
template <bool kSK>
struct SegIter {
  int64_t lo, u, hi;
  int U, items, w_rr;
  static constexpr bool streamk = kSK;
  __device__ __forceinline__ explicit SegIter(const SmallPlan& p) {
    U = p.U;
    items = p.T * p.nb;
    w_rr = blockIdx.x;
    lo = u = hi = 0;
    if (streamk && (int)blockIdx.x < p.G) {
      lo = u = sk_lo(p, blockIdx.x);
      hi = sk_lo(p, blockIdx.x + 1);
    }
  }
  __device__ __forceinline__ bool next(int& w, int& u0, int& u1, bool& first) {
    if (!streamk) {
      if (w_rr >= items) return false;
      w = w_rr;
      w_rr += gridDim.x;
      u0 = 0;
      u1 = U;
      first = true;
      return true;
    }
    if (u >= hi) return false;
    w = (int)(u / U);
    const int64_t base = (int64_t)w * U;
    u0 = (int)(u - base);
    u1 = (int)(hi - base < (int64_t)U ? hi - base : (int64_t)U);
    first = u == lo;
    u = base + u1;
    return true;
  }
};

// 8 INT4 (uint4b8) codes of one word -> its 4 pairs of (q - 8) as f16x2, exact:
// pairs 0 and 2 are (1024 + q) - 1032, pairs 1 and 3 (1024 + 16q) / 16 - 72.
__device__ __forceinline__ void int4x8_f16_unscaled(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t t[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x64006400u,
                         (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x64006400u};
  const __half2 c1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 r16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
  const __half2 cm72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));  // -72
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 x = *reinterpret_cast<const __half2*>(&t[i]);
    const __half2 r = (i & 1) ? __hfma2(x, r16, cm72) : __hsub2(x, c1032);
    o[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// f16x2 multipliers of one FP4 row from its scale bytes: MXFP4 one per 32 K
// (m[0], m[1]), NVFP4 one per 16 K (m[0..3]).
template <int FMT>
__device__ __forceinline__ void fp4_row_multipliers(uint32_t sv, uint32_t (&m)[4]) {
  if (FMT == MOE_W_MXFP4) {
    const uint32_t ac = e8m0x2_mult_f16(sv);
    m[0] = __byte_perm(ac, 0, 0x1010);
    m[1] = __byte_perm(ac, 0, 0x3232);
  } else {
    const uint32_t lo = e4m3x2_mult_f16(sv & 0xFFFF), hi = e4m3x2_mult_f16(sv >> 16);
    m[0] = __byte_perm(lo, 0, 0x1010);
    m[1] = __byte_perm(lo, 0, 0x3232);
    m[2] = __byte_perm(hi, 0, 0x1010);
    m[3] = __byte_perm(hi, 0, 0x3232);
  }
}

// Per-warp constants of the consumer loop (byte offsets inside a slot).
template <int NT, int MI>
struct SmallFrag {
  static constexpr int NQ = NT > 1 ? NT / 2 : 1;
  int rows[MI][2];           // tile rows: row gq + 8h of 16-row fragment i
  uint32_t code_off[MI][2];  // this lane's 8 bytes of each row inside a stage's code block
  uint32_t sc_off[MI][2];    // each row's scale inside a scale block
  uint32_t b_off[4][NQ];           // ldmatrix row address of K-step j (token group q) in a stage block
};

// Activation fragments of one stage block ([BN][64] fp16, 128-byte swizzle):
// bf[step][n-tile][0..1].
template <int NT, int MI>
__device__ __forceinline__ void load_b_frags(uint32_t sb, const SmallFrag<NT, MI>& F, uint32_t (&bf)[4][NT][2]) {
  if (NT == 1) {
#pragma unroll
    for (int j0 = 0; j0 < 4; j0 += 2)
      ldmatrix_x4(sb + F.b_off[j0][0], bf[j0][0][0], bf[j0][0][1], bf[j0 + 1][0][0], bf[j0 + 1][0][1]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < SmallFrag<NT, MI>::NQ; ++q)
        ldmatrix_x4(sb + F.b_off[j][q], bf[j][2 * q][0], bf[j][2 * q][1], bf[j][2 * q + 1][0], bf[j][2 * q + 1][1]);
  }
}

// NST stages of a chunk (starting on a scale period; wsl its shared address)
// into the accumulators.  INT4 keeps each 128-K group's sum of (q - 8) * x in
// its own accumulators and adds it times the group's fp32 scale; FP4 scales the
// codes in fp16 (exact).
template <int FMT, int NT, int BN, int NST, int MI>
__device__ __forceinline__ void consume_chunk(uint32_t wsl, uint32_t bsl, const SmallFrag<NT, MI>& F,
                                              float (&acc)[MI][NT][4], uint32_t (&m)[MI][2][4],
                                              int zp_float) {
  using PF = PackedFmt<FMT>;
  if constexpr (FMT == MOE_W_INT4_U4B8) {
#pragma unroll
    for (int gp = 0; gp < NST / 2; ++gp) {
      float sc[MI][2];
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) sc[i][h] = __uint_as_float(lds16(wsl + PF::stage_off(2 * gp) + F.sc_off[i][h]) << 16);
      float part[MI][NT][4];
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) part[i][n][c] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int ss = 2 * gp + s2;
        uint2 wv[MI][2];
#pragma unroll
        for (int i = 0; i < MI; ++i)
#pragma unroll
          for (int h = 0; h < 2; ++h) wv[i][h] = lds64(wsl + PF::codes_off(ss) + F.code_off[i][h]);
        uint32_t bf[4][NT][2];
        load_b_frags<NT, MI>(bsl + (uint32_t)(ss * BN * 128), F, bf);
#pragma unroll
        for (int i = 0; i < MI; ++i)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t p0[4], p1[4];  // fragment rows gq and gq + 8
            int4x8_f16_unscaled(h ? wv[i][0].y : wv[i][0].x, p0);
            int4x8_f16_unscaled(h ? wv[i][1].y : wv[i][1].x, p1);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              mma_16816(part[i][n], p0[0], p1[0], p0[1], p1[1], bf[2 * h][n][0], bf[2 * h][n][1]);
              mma_16816(part[i][n], p0[2], p1[2], p0[3], p1[3], bf[2 * h + 1][n][0], bf[2 * h + 1][n][1]);
            }
          }
      }
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[i][n][c] = fmaf(sc[i][c >> 1], part[i][n][c], acc[i][n][c]);
    }
  } else if constexpr (FMT == kFmtInt4X) {
    // one 32-bit entry (multiplier, zero term) per row and 32-element half stage;
    // codes dequantised to fp16 with it (as the tcgen05 kernel does)
#pragma unroll
    for (int ss = 0; ss < NST; ++ss) {
      uint2 ev[MI][2];
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) ev[i][hr] = lds64(wsl + PF::stage_off(ss) + F.sc_off[i][hr]);
      uint2 wv[MI][2];
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) wv[i][hr] = lds64(wsl + PF::codes_off(ss) + F.code_off[i][hr]);
      uint32_t bf[4][NT][2];
      load_b_frags<NT, MI>(bsl + (uint32_t)(ss * BN * 128), F, bf);
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t p0[4], p1[4];  // fragment rows gq and gq + 8, K half h
          int4x8_f16_zp(h ? wv[i][0].y : wv[i][0].x, int4zp_const(h ? ev[i][0].y : ev[i][0].x, zp_float), p0);
          int4x8_f16_zp(h ? wv[i][1].y : wv[i][1].x, int4zp_const(h ? ev[i][1].y : ev[i][1].x, zp_float), p1);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            mma_16816(acc[i][n], p0[0], p1[0], p0[1], p1[1], bf[2 * h][n][0], bf[2 * h][n][1]);
            mma_16816(acc[i][n], p0[2], p1[2], p0[3], p1[3], bf[2 * h + 1][n][0], bf[2 * h + 1][n][1]);
          }
        }
    }
  } else {
#pragma unroll
    for (int ss = 0; ss < NST; ++ss) {
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t a = wsl + PF::stage_off(ss) + F.sc_off[i][h];
          fp4_row_multipliers<FMT>(FMT == MOE_W_MXFP4 ? lds16(a) : lds32(a), m[i][h]);
        }
      uint2 wv[MI][2];
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) wv[i][h] = lds64(wsl + PF::codes_off(ss) + F.code_off[i][h]);
      uint32_t bf[4][NT][2];
      load_b_frags<NT, MI>(bsl + (uint32_t)(ss * BN * 128), F, bf);
#pragma unroll
      for (int i = 0; i < MI; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t p0[4], p1[4];
          if (FMT == MOE_W_MXFP4) {
            e2m1x8_f16(h ? wv[i][0].y : wv[i][0].x, m[i][0][h], m[i][0][h], p0);
            e2m1x8_f16(h ? wv[i][1].y : wv[i][1].x, m[i][1][h], m[i][1][h], p1);
          } else {
            e2m1x8_f16(h ? wv[i][0].y : wv[i][0].x, m[i][0][2 * h], m[i][0][2 * h + 1], p0);
            e2m1x8_f16(h ? wv[i][1].y : wv[i][1].x, m[i][1][2 * h], m[i][1][2 * h + 1], p1);
          }
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            mma_16816(acc[i][n], p0[0], p1[0], p0[1], p1[1], bf[2 * h][n][0], bf[2 * h][n][1]);
            mma_16816(acc[i][n], p0[2], p1[2], p0[3], p1[3], bf[2 * h + 1][n][0], bf[2 * h + 1][n][1]);
          }
        }
    }
  }
}

template <int FMT, int STAGE, int BN>
__global__ void __launch_bounds__(SmallCfg<BN, STAGE>::kThreads, 1) moe_gemm_small_kernel(const __grid_constant__ GemmArgs g) {
  constexpr bool kG1 = STAGE != kGemm2;          // reads w13 (x rows) rather than w2 (a rows)
  constexpr bool kGated = STAGE == kGemm1Gated;  // fragment rows pair gate and up features
  using SM = SmallSmem<BN, FMT>;
  constexpr int kSmallWBytes = SM::kWBytes;
  constexpr int kSlots = SM::kSlots;
  constexpr int NT = BN / 8;  // 8-token column tiles
  constexpr int kCW = SmallCfg<BN, STAGE>::kConsumerWarps, MI = SmallCfg<BN, STAGE>::kMI;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBar);
  uint64_t* empty = full + kSlots;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + SM::kMisc);  // [1] abort, [2] last-arrival flag
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&misc[1]);
  uint64_t* starve = reinterpret_cast<uint64_t*>(&misc[4]);  // test hook's barrier (never arrived on)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Layout& L = g.L;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    misc[1] = 0;
    mbar_init(starve, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&g.tmap_b)) : "memory");
  __syncthreads();
  // Ordering against the stream predecessors (programmatic launch): this kernel
  // starts only once its predecessor has passed its own wait.  When the
  // alignment came from moe_align (align_early), it was written two launches
  // back and is complete, with the packed weights, so the producer streams
  // weights at once; the activation rows, the split-K counters and the outputs
  // belong to the predecessor, and every thread that touches them waits first.
  // When the prologue wrote the alignment, everyone waits.
  grid_dependents_launch();
  if (!g.align_early) grid_dependency_wait();

  const SmallPlan plan = make_plan_small(g, kG1, BN);
  const int64_t tile_bytes = kG1 ? L.tile1_bytes : L.tile2_bytes;
  const uint8_t* wbase = g.packed + (kG1 ? L.w13_off : L.w2_off);

  // The roles, compiled twice: with the stream-K cuts (kSK) and without them,
  // so that whole-item launches keep the leaner code (a uniform branch picks
  // one).  32-token blocks run whole items only: their register budget has no
  // room for the cut path.
  auto roles = [&](auto sk_tag) {
    constexpr bool kSK = decltype(sk_tag)::value;
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      // The whole warp runs the loop; lane 0 issues the weight copies.  GEMM1's
      // activation rows are gathered from x (fp16, one row per token) four at a
      // time by the warp's lanes, token = sorted id / top_k; GEMM2's are the
      // block's rows of a (sorted order), one 3-D box per chunk.  When the
      // alignment is older than the predecessor (align_early), the first ring's
      // worth of weight copies go out before the wait on the predecessor and their
      // activation copies (the predecessor's output) follow it; each slot's
      // barrier expects both byte counts from the start.
      const uint64_t pol = policy_evict_first();
      int32_t* item_rows = reinterpret_cast<int32_t*>(smem + SM::kRows);
      int32_t* pend_rows = item_rows + 32;  // [kSlots][32]
      int pend_row[kSlots], pend_stage[kSlots], pend_nst[kSlots];
      uint32_t npend = 0;
      bool waited = !g.align_early;
      uint32_t ck = 0;
      // GEMM1 gathers token rows, unless the prologue placed them in sorted order
      // (act-order banks, whose x columns follow each expert's order)
      const bool gather = kG1 && !g.gemm1_rows_sorted;
      // activation copies of chunk `stage0` (nst stages) into slot `slot`, rows from `rows`
      auto issue_act = [&](int slot, int row0, int stage0, int nst, const int32_t* rows) {
        const uint32_t dst = smem_u32(smem + slot * SM::kSlotBytes + kSmallWBytes);
        if (gather) {
          const uint32_t rows_s = smem_u32(rows);
          for (int q = lane; q < nst * (BN / 4); q += 32) {
            const int j = q / (BN / 4), r4 = q % (BN / 4);
            const uint4 rv = lds128(rows_s + 16 * r4);
            tma_gather4(dst + j * (BN * 128) + r4 * 512, &g.tmap_b, (stage0 + j) * kStageK,
                        make_int4((int)rv.x, (int)rv.y, (int)rv.z, (int)rv.w), &full[slot]);
          }
        } else if (lane == 0) {
          tma_tile3d(dst, &g.tmap_b, 0, row0, stage0, &full[slot]);
        }
      };
      SegIter<kSK> seg(plan);
      int w, u0, u1;
      bool first;
      while (seg.next(w, u0, u1, first)) {
        const int tile = w % plan.T, b = w / plan.T;
        const int s0 = u0 * L.period, s1 = u1 * L.period;
        const int e = block_expert(g, b);
        if (e < 0) continue;  // (the consumers skip it too)
        if (gather) {
          __syncwarp();  // the previous item's rows are consumed
          load_block_rows(g, b, BN, lane, item_rows);
          __syncwarp();
        }
        const uint8_t* tb = wbase + ((int64_t)e * plan.T + tile) * tile_bytes;
        for (int c0 = s0; c0 < s1; c0 += kSmallChunk, ++ck) {
          const int c1 = min(c0 + kSmallChunk, s1);
          const int slot = ck % kSlots;
          if (!waited && ck == (uint32_t)kSlots) {
            grid_dependency_wait();
            waited = true;
            for (uint32_t i = 0; i < npend; ++i) issue_act(i, pend_row[i], pend_stage[i], pend_nst[i], pend_rows + 32 * i);
          }
          mbar_wait(&empty[slot], ((ck / kSlots) + 1) & 1, abort_flag, g.status);
          // c0 and c1 lie on scale-period boundaries
          const int64_t off0 = (int64_t)(c0 / PackedFmt<FMT>::kPeriod) * PackedFmt<FMT>::kPeriodBytes;
          const uint32_t wbytes = (uint32_t)((c1 - c0) / PackedFmt<FMT>::kPeriod * PackedFmt<FMT>::kPeriodBytes);
          const uint32_t bbytes = gather ? (uint32_t)((c1 - c0) * BN * 128) : (uint32_t)SM::kBBytes;
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[slot], wbytes + bbytes);
            bulk_g2s(smem + slot * SM::kSlotBytes, tb + off0, wbytes, &full[slot], pol);
          }
          __syncwarp();
          if (waited) {
            issue_act(slot, b * g.block_m, c0, c1 - c0, item_rows);
          } else {  // ck < kSlots: slot == ck
            if (gather && lane < BN) pend_rows[32 * npend + lane] = item_rows[lane];
            pend_row[npend] = b * g.block_m;
            pend_stage[npend] = c0;
            pend_nst[npend] = c1 - c0;
            ++npend;
            __syncwarp();
          }
        }
      }
      if (!waited) {
        grid_dependency_wait();
        for (uint32_t i = 0; i < npend; ++i) issue_act(i, pend_row[i], pend_stage[i], pend_nst[i], pend_rows + 32 * i);
      }
      // leave no copy in flight
      if (lane == 0) {
        for (uint32_t i = 0; i < (uint32_t)kSlots && i < ck; ++i) {
          const uint32_t k = ck - 1 - i;
          mbar_drain(&full[k % kSlots], (k / kSlots) & 1, g.status);
        }
      }
    } else {
      // ------------------------------------------------------------ consumer warps
      grid_dependency_wait();
      const int cw = warp - 1;
      const int gq = lane >> 2, tq = lane & 3;
      SmallFrag<NT, MI> F;
      int (&rows)[MI][2] = F.rows;
  #pragma unroll
      for (int i = 0; i < MI; ++i) {
        if (kGated) {  // gate feature f in fragment row gq, its up row in gq + 8
          rows[i][0] = 8 * (MI * cw + i) + gq;
          rows[i][1] = 128 + rows[i][0];
        } else {
          rows[i][0] = 16 * (MI * cw + i) + gq;
          rows[i][1] = rows[i][0] + 8;
        }
      }
  #pragma unroll
      for (int i = 0; i < MI; ++i)
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          F.code_off[i][h] = (uint32_t)(((tq >> 1) * 256 + rows[i][h]) * 16 + (tq & 1) * 8);
          F.sc_off[i][h] = (uint32_t)(rows[i][h] * (FMT == kFmtInt4X ? 8 : (FMT == MOE_W_NVFP4 ? 4 : 2)));
        }
      // ldmatrix row addresses: token row n, 16-byte chunk c of a stage block sits
      // at n * 128 + ((c ^ (n & 7)) << 4) (the TMA's 128-byte swizzle)
      if (NT == 1) {
        const uint32_t n = (uint32_t)(lane & 7), sel = (uint32_t)(lane >> 3);  // two K-steps per load
  #pragma unroll
        for (int j = 0; j < 4; ++j) F.b_off[j][0] = n * 128 + ((((uint32_t)(2 * (j & ~1)) + sel) ^ (n & 7)) << 4);
      } else {
        const uint32_t sel = (uint32_t)((lane >> 3) & 1);
  #pragma unroll
        for (int q = 0; q < SmallFrag<NT, MI>::NQ; ++q) {
          const uint32_t n = (uint32_t)(16 * q + (lane & 7) + 8 * (lane >> 4));
  #pragma unroll
          for (int j = 0; j < 4; ++j) F.b_off[j][q] = n * 128 + ((((uint32_t)(2 * j) + sel) ^ (n & 7)) << 4);
        }
      }
      const float* gs_tab = reinterpret_cast<const float*>(g.packed + (kG1 ? L.gs13_off : L.gs2_off));
      const uint16_t* bias_tab = reinterpret_cast<const uint16_t*>(g.packed + (kG1 ? L.b13_off : L.b2_off));
      const int Npad = L.Npad;
      uint32_t m[MI][2][4] = {};
      uint32_t ck = 0;
      float vmax = 0.0f;  // largest |value| stored as fp16 (NaN ignored)

      SegIter<kSK> seg(plan);
      int w, u0, u1;
      bool first;
      while (seg.next(w, u0, u1, first)) {
        const int tile = w % plan.T, b = w / plan.T;
        const int s0 = u0 * L.period, s1 = u1 * L.period;
        const int e = block_expert(g, b);
        if (e < 0) {  // a block inside n_padded without one of this layer's experts
          if (cw == 0 && lane == 0 && u0 == 0) atomicOr(g.status, kStatusRouting);
          continue;
        }
        // what the item's epilogue reads from global memory (scale, sorted ids,
        // bias) is fetched before its K loop, off the critical path, where that
        // measured faster: GEMM2 and FP4 GEMM1 up to 16-token blocks (INT4 GEMM1,
        // which keeps per-group sums in registers, measured 1-1.5 % slower)
        constexpr bool kEpiPf = NT <= 2 && (!kG1 || FMT == MOE_W_MXFP4 || FMT == MOE_W_NVFP4);
        const float gsc_pf = kEpiPf ? gs_tab[e] : 0.f;
        int sid_pf[NT][2];
        float bias_pf[MI][2];  // gated: gate and up bias of the row; otherwise of rows h = 0, 1
        if (kEpiPf) {
  #pragma unroll
          for (int n = 0; n < NT; ++n)
  #pragma unroll
            for (int c = 0; c < 2; ++c) sid_pf[n][c] = g.sorted_ids[b * g.block_m + n * 8 + 2 * tq + c];
  #pragma unroll
          for (int i = 0; i < MI; ++i) {
            bias_pf[i][0] = 0.f;
            bias_pf[i][1] = 0.f;
            if (g.has_bias) {
              if (kGated) {
                const int f = tile * 128 + rows[i][0];
                bias_pf[i][0] = bf16_bits_to_float(bias_tab[(int64_t)e * 2 * Npad + f]);
                bias_pf[i][1] = bf16_bits_to_float(bias_tab[(int64_t)e * 2 * Npad + Npad + f]);
              } else {
  #pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int o = tile * 256 + rows[i][h];
                  if (kG1) bias_pf[i][h] = bf16_bits_to_float(bias_tab[(int64_t)e * Npad + o]);
                  else if (o < L.K) bias_pf[i][h] = bf16_bits_to_float(bias_tab[(int64_t)e * L.Kpad2 + o]);
                }
              }
            }
          }
        }
        float acc[MI][NT][4];
  #pragma unroll
        for (int i = 0; i < MI; ++i)
  #pragma unroll
          for (int n = 0; n < NT; ++n)
  #pragma unroll
            for (int c = 0; c < 4; ++c) acc[i][n][c] = 0.f;

        for (int c0 = s0; c0 < s1; c0 += kSmallChunk, ++ck) {
          const int slot = ck % kSlots;
          mbar_wait(&full[slot], (ck / kSlots) & 1, abort_flag, g.status);
          const uint32_t wsl = smem_u32(smem + slot * SM::kSlotBytes);
          const uint32_t bsl = wsl + kSmallWBytes;
          const int nst = min(kSmallChunk, s1 - c0);
          if (nst == 4) consume_chunk<FMT, NT, BN, 4, MI>(wsl, bsl, F, acc, m, g.zp_float);
          else if (nst == 2) consume_chunk<FMT, NT, BN, 2, MI>(wsl, bsl, F, acc, m, g.zp_float);
          else if (FMT != MOE_W_INT4_U4B8) {  // INT4 chunks always hold whole 2-stage periods
            if (nst == 3) consume_chunk<FMT, NT, BN, 3, MI>(wsl, bsl, F, acc, m, g.zp_float);
            else consume_chunk<FMT, NT, BN, 1, MI>(wsl, bsl, F, acc, m, g.zp_float);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ---------------------------------------------------------- epilogue
        if (kSK && (u0 > 0 || u1 < plan.U)) {
          // a cut item: store this segment's fp32 partial ([256 tile rows][BN
          // tokens] in the slot of this CTA's first or last segment); the last
          // of the item's CTAs to arrive sums all of them in CTA order
          const int slot = 2 * blockIdx.x + (first ? 0 : 1);
          float* dst = g.partial + (int64_t)slot * kTileRows * BN;
  #pragma unroll
          for (int i = 0; i < MI; ++i)
  #pragma unroll
            for (int h = 0; h < 2; ++h)
  #pragma unroll
              for (int n = 0; n < NT; ++n)
                __stcg(reinterpret_cast<float2*>(dst + rows[i][h] * BN + n * 8 + 2 * tq),
                       make_float2(acc[i][n][2 * h], acc[i][n][2 * h + 1]));
          // the CTA barrier orders every consumer's partial stores before one thread's
          // fence and arrival (release); the last CTA's arriving thread fences again
          // before the barrier that lets its warps read the others' partials (acquire)
          named_bar_sync(1, kCW * 32);
          const int64_t wu = (int64_t)w * plan.U;
          const int c_first = sk_owner(plan, wu), c_last = sk_owner(plan, wu + plan.U - 1);
          if (cw == 0 && lane == 0) {
            __threadfence();
            const unsigned old = atomicInc(reinterpret_cast<unsigned*>(&g.counters[w]), (unsigned)(c_last - c_first));
            misc[2] = old == (unsigned)(c_last - c_first) ? 1u : 0u;
            __threadfence();
          }
          named_bar_sync(1, kCW * 32);
          const bool last = misc[2] != 0;
          named_bar_sync(1, kCW * 32);  // misc[2] is read before the next segment rewrites it
          if (!last) continue;
  #pragma unroll
          for (int i = 0; i < MI; ++i)
  #pragma unroll
            for (int n = 0; n < NT; ++n)
  #pragma unroll
              for (int c = 0; c < 4; ++c) acc[i][n][c] = 0.f;
          // the partials of kPU CTAs are loaded before they are added (in CTA
          // order); INT4 GEMM1, at its register limit, measured slower with it
          constexpr bool kIntG1 = kG1 && (FMT == MOE_W_INT4_U4B8 || FMT == kFmtInt4X);
          constexpr int kPU = kIntG1 ? 1 : (MI * NT == 1 ? 4 : (MI * NT == 2 ? 2 : 1));
          for (int cc0 = c_first; cc0 <= c_last; cc0 += kPU) {
            float2 pv[kPU][MI][2][NT];
  #pragma unroll
            for (int uu = 0; uu < kPU; ++uu) {
              const int cc = cc0 + uu;
              if (cc > c_last) break;
              // CTA cc holds this item in its first segment iff its range starts inside the item
              const float* src = g.partial + (int64_t)(2 * cc + (sk_lo(plan, cc) >= wu ? 0 : 1)) * kTileRows * BN;
  #pragma unroll
              for (int i = 0; i < MI; ++i)
  #pragma unroll
                for (int h = 0; h < 2; ++h)
  #pragma unroll
                  for (int n = 0; n < NT; ++n)
                    pv[uu][i][h][n] = __ldcg(reinterpret_cast<const float2*>(src + rows[i][h] * BN + n * 8 + 2 * tq));
            }
  #pragma unroll
            for (int uu = 0; uu < kPU; ++uu) {
              if (cc0 + uu > c_last) break;
  #pragma unroll
              for (int i = 0; i < MI; ++i)
  #pragma unroll
                for (int h = 0; h < 2; ++h)
  #pragma unroll
                  for (int n = 0; n < NT; ++n) {
                    acc[i][n][2 * h] += pv[uu][i][h][n].x;
                    acc[i][n][2 * h + 1] += pv[uu][i][h][n].y;
                  }
            }
          }
        }
        const float gsc = kEpiPf ? gsc_pf : gs_tab[e];
  #pragma unroll
        for (int i = 0; i < MI; ++i) {
          if (kGated) {
            const int f = tile * 128 + rows[i][0];
            float bg = 0.f, bu = 0.f;
            if (kEpiPf) {
              bg = bias_pf[i][0];
              bu = bias_pf[i][1];
            } else if (g.has_bias) {
              bg = bf16_bits_to_float(bias_tab[(int64_t)e * 2 * Npad + f]);
              bu = bf16_bits_to_float(bias_tab[(int64_t)e * 2 * Npad + Npad + f]);
            }
  #pragma unroll
            for (int n = 0; n < NT; ++n)
  #pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int pos = b * g.block_m + n * 8 + 2 * tq + c;
                const int sid = kEpiPf ? sid_pf[n][c] : g.sorted_ids[pos];
                if ((unsigned)sid > (unsigned)g.pairs) atomicOr(g.status, kStatusRouting);  // neither a pair nor padding
                const float hg = acc[i][n][c] * gsc + bg;
                const float hu = acc[i][n][2 + c] * gsc + bu;
                const float a = live_sid(sid, g.pairs) ? act_fn(g.act_kind, hg, hu, g.alpha, g.limit) : 0.0f;
                vmax = fmax_nan(vmax, fabsf(a));
                g.a_out[(int64_t)pos * Npad + f] = __half_as_ushort(__float2half_rn(a));
              }
          } else if (kG1) {  // non-gated: relu(h)^2 of each row, fp16 rows by sorted position
  #pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int f = tile * 256 + rows[i][h];
              const float bf = kEpiPf ? bias_pf[i][h] : (g.has_bias ? bf16_bits_to_float(bias_tab[(int64_t)e * Npad + f]) : 0.f);
  #pragma unroll
              for (int n = 0; n < NT; ++n)
  #pragma unroll
                for (int c = 0; c < 2; ++c) {
                  const int pos = b * g.block_m + n * 8 + 2 * tq + c;
                  const int sid = kEpiPf ? sid_pf[n][c] : g.sorted_ids[pos];
                  if ((unsigned)sid > (unsigned)g.pairs) atomicOr(g.status, kStatusRouting);
                  const float hv = acc[i][n][2 * h + c] * gsc + bf;
                  const bool live = live_sid(sid, g.pairs);
                  const float a = live ? relu2(hv) : 0.0f;
                  vmax = fmax_nan(vmax, fmax_nan(a, live ? hv * 0.0f : 0.0f));  // hv * 0: NaN unless finite
                  g.a_out[(int64_t)pos * Npad + f] = __half_as_ushort(__float2half_rn(a));
                }
            }
          } else {
  #pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int o = tile * 256 + rows[i][h];
              if (o >= L.K) continue;
              const float bo = kEpiPf ? bias_pf[i][h] : (g.has_bias ? bf16_bits_to_float(bias_tab[(int64_t)e * L.Kpad2 + o]) : 0.f);
  #pragma unroll
              for (int n = 0; n < NT; ++n)
  #pragma unroll
                for (int c = 0; c < 2; ++c) {
                  const int pos = b * g.block_m + n * 8 + 2 * tq + c;
                  const int sid = kEpiPf ? sid_pf[n][c] : g.sorted_ids[pos];
                  if ((unsigned)sid > (unsigned)g.pairs) atomicOr(g.status, kStatusRouting);
                  if (live_sid(sid, g.pairs)) {
                    const float y = acc[i][n][2 * h + c] * gsc + bo;
                    vmax = fmax_nan(vmax, y * 0.0f);  // fp32 y: only a non-finite value is an error
                    g.y_out[(int64_t)sid * L.K + o] = y;
                  }
                }
            }
          }
        }
      }
      // Test hook of the failure path: after all its work, CTA 0's consumers wait
      // on a barrier nothing arrives on.  The bounded wait gives up after the wait
      // limit, records the timeout in the status word and the kernel ends
      // normally, so the host reads MOE_ERR_TIMEOUT and the context stays usable.
      if (g.test_starve_wait && blockIdx.x == 0) mbar_wait(starve, 0, abort_flag, g.status);
      report_epilogue_status(g, vmax, cw == 0 && lane == 0, kStatusBlobFlagsSmall);
    }
  };
  if (BN < 32 && plan.streamk) roles(std::integral_constant<bool, (BN < 32)>{});
  else roles(std::false_type{});
  __syncthreads();
}

}  // namespace moe
