// Grouped W4A16 GEMM on tcgen05 tensor cores (sm_103a), shared by GEMM1 (w13,
// fused gated or relu^2 activation) and GEMM2 (w2).
//
// The function is Marlin's moe_wna16_marlin_gemm as called twice by
// "013-moe-middle-tiles.py" kernel_fn (GEMM1 with top_k = 8 over x, GEMM2 with
// top_k = 1 over the activation rows), with the per-expert bias epilogue of
// "Marlin MoE kernel occupancy ..." (sglang PR #31552, kHasBias) and the -1
// block skip of its kIsEP path.  The design is GB300-native:
//
//   * swap-AB: weights are the MMA's M side (two 128-row halves per tile),
//     routed tokens of one aligned block are the N side (16..128), so decode
//     sizes still fill the 128-lane tensor-core tile;
//   * the dequantised weights never touch shared memory: eight dequant warps
//     (each thread one row of a 64-element stage) turn 4-bit codes into fp16 in
//     registers -- E2M1 through the hardware E2M1x2 conversion, INT4
//     through mask-and-magic-number pairs -- and store them into tensor memory
//     (tcgen05.st, one row per lane); the MMA reads its A operand from there, so
//     shared memory only holds the packed codes and the activation rows and
//     deep rings fit;
//   * operands are fp16 x fp16: every dequantised weight is exact in fp16, and
//     the activation operand keeps 11 significant bits.  Accumulation, bias,
//     scales and the activation are fp32;
//   * two producer threads, one per operand stream, keep both in flight with
//     TMA: a 1-D bulk copy of each stage's packed codes + scales (one
//     contiguous chunk thanks to the repack) and a 2-D tile of the block's
//     activation rows (GEMM1: the rows the prologue gathered in sorted order;
//     GEMM2: GEMM1's output), landing in the 128-byte swizzled K-major layout;
//   * a persistent grid (one CTA per SM) walks work items (tile, K-split, block)
//     with the tile index fastest, so the tiles of one block run together and
//     its activation rows are read from L2; K is split on the device when there
//     are too few items to fill the GPU (decode), and the last CTA to arrive on
//     an item's counter sums the fp32 partials in split order (bitwise
//     reproducible, no spinning);
//   * one elected lane of the MMA warp issues tcgen05.mma into TMEM accumulators (double-buffered up
//     to 64 tokens); eight epilogue warps (two per TMEM lane quarter, splitting
//     the token columns; sixteen in some 128-token instances, GemmCfg) add
//     bias and scales, apply the activation (GEMM1:
//     act(gate, up) of a lane's two halves, or relu(h)^2 of each half for
//     non-gated experts) or write rows to their pairs (GEMM2).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

constexpr int kSup = 2;                // 64-K stages per pipeline unit (one barrier round per unit)
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpBProducer = 2, kWarpDequant0 = 3;
// Warp roles per instance.  Dequant warps: eight, one per TMEM lane quarter
// and 128-row half, each thread one row of a whole 64-element stage.  The
// kernel also supports sixteen, the two 32-element halves of a stage on two
// warps (kSplitDq); within the 864 threads a CTA can run at 72 registers that
// leaves eight epilogue warps, and INT4 GEMM1 at 128-token tiles measured
// slower that way (headline GEMM1 725 -> 773 us), so every instance runs
// eight.  Epilogue warps: sixteen (four per TMEM lane quarter) at 128-token
// tiles and for the FP4 formats, whose epilogues then drain the accumulator in
// half the time (headline GEMM2 453 -> 422 us, mxfp4 M=1024 275 -> 248 us,
// nvfp4 M=512 -2.5 %); eight for INT4 at 64-token tiles, which measured 1-3 %
// slower with sixteen in the 72 registers a thread that an 864-thread CTA
// leaves.
template <int FMT, int BN, int STAGE>
struct GemmCfg {
  static constexpr bool kSplitDq = false;
  static constexpr int kDqWarps = kSplitDq ? 16 : 8;
  static constexpr int kEpiWarps = kSplitDq ? 8 : ((BN == 128 || FMT == MOE_W_MXFP4 || FMT == MOE_W_NVFP4) ? 16 : 8);
  static constexpr int kWarpEpi0 = kWarpDequant0 + kDqWarps;
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kEpiColStep = 8 * (kEpiWarps / 4);  // a warp's 8-column batches lie this far apart
  static constexpr int kThreads = (kWarpEpi0 + kEpiWarps) * 32;  // 608 or 864
};
constexpr int kSmemBudget = 227 * 1024;
constexpr uint32_t kTmemCols = 512;                         // whole TMEM (one CTA per SM)
constexpr uint32_t kAColsPerStage = 64;                     // 2 halves x 64 K / 2 per column
constexpr uint32_t kAColsPerUnit = kSup * kAColsPerStage;

struct GemmArgs {
  CUtensorMap tmap_b;         // activation rows: tcgen05 kernel, sorted order [cap, Kred] fp16 as 3-D
                              // boxes of 64 x BN x stages (GEMM1: the prologue's xs, GEMM2: a);
                              // register-fed GEMM1: x's rows [M, K] fp16 for 4-row gathers of 64
                              // columns; register-fed GEMM2: a as 3-D boxes
  Layout L;
  const uint8_t* packed;      // repacked blob
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* n_padded;
  int64_t cap;                // sorted slots the workspace holds (n_padded beyond it is an error)
  int pairs;                  // M * top_k (sentinel value)
  int top_k;                  // token of a pair = pair / top_k (GEMM1's row gather)
  int align_early;            // 1: the alignment was written two launches back (moe_align), so it may
                              // be read before the dependency wait; 0: the prologue just wrote it
  int block_m;
  int has_bias;
  int act_kind;               // moe_act
  float alpha, limit;
  int max_split;
  int split_rows;             // rows of each split-K partial slice
  uint16_t* a_out;            // GEMM1 output, fp16 [cap, Npad]
  float* y_out;               // GEMM2 output, fp32 [pairs, K]
  float* partial;             // split-K partials [max_split][split_rows][width]
  int32_t* counters;          // split-K arrival counters [T * blocks]
  unsigned* status;
  int test_starve_wait;       // test hook (register-fed kernel): CTA 0 ends with a wait nothing completes
  int zp_float;               // INT4X: entries carry -z * m (float zero points) instead of 1024 + z
  int gemm1_rows_sorted;      // register-fed GEMM1: read x's routed rows in sorted order (act-order banks)
};

template <int BN, int FMT>
struct GemmSmem {
  static constexpr int kPackedSlotBytes = PackedFmt<FMT>::kSlotBytes(kSup);  // a unit's codes + scale blocks
  static constexpr int kSA = 2;                    // dequantised-A ring in TMEM, in units
  static constexpr int kNacc = BN >= 128 ? 1 : 2;  // TMEM accumulators
  static constexpr int kBUnitBytes = kSup * BN * 128;  // activation rows of a unit, [stage][row][64]
  static constexpr int kSB = BN <= 64 ? 6 : 4;           // activation ring, in units
  static constexpr int kB = 0;
  static constexpr int kP = kB + kSB * kBUnitBytes;
  static constexpr int kSPfit = (kSmemBudget - kP - 3072) / kPackedSlotBytes;
  static constexpr int kSP = kSPfit > 8 ? 8 : kSPfit;  // packed-weight ring, in units
  static constexpr int kBar = kP + kSP * kPackedSlotBytes;
  // barriers: p_full, p_empty, a_full, a_empty, b_full, b_empty, acc_full, acc_empty, drain
  static constexpr int kNumBars = 2 * kSP + 2 * kSA + 2 * kSB + 2 * kNacc + 1;
  static constexpr int kEpiSid = (kBar + kNumBars * 8 + 15) / 16 * 16;  // epilogue copy of the block's sorted ids
  static constexpr int kMisc = kEpiSid + BN * 4;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSP >= 4, "packed ring too shallow");
  static_assert(kAlloc <= 232448, "shared memory over the per-CTA limit");
  static_assert(kSA * kAColsPerUnit + kNacc * 2 * BN <= kTmemCols, "TMEM over budget");
};

// Gated activations in fp32.  The logistic function is 1/2 + tanh(x/2)/2 on
// the hardware tanh approximation (one special-function op, relative error
// ~2^-11, the size of the fp16 rounding the activation gets anyway); it
// saturates cleanly, so a very negative gate gives 0.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float act_fn(int kind, float g, float u, float alpha, float limit) {
  if (kind == MOE_ACT_SILU_MUL) {
    const float hg = 0.5f * g;
    return fmaf(hg, tanh_approx(hg), hg) * u;  // g * sigmoid(g) * u
  }
  const float gc = fmin_nan(g, limit);  // clamp(max=limit), NaN stays NaN
  const float uc = fmin_nan(fmax_nan(u, -limit), limit);
  const float hg = 0.5f * gc;
  return fmaf(hg, tanh_approx(alpha * hg), hg) * (uc + 1.0f);  // gc * sigmoid(alpha * gc) * (uc + 1)
}
// Activation of non-gated experts: relu(h)^2.
__device__ __forceinline__ float relu2(float h) { return h > 0.0f ? h * h : 0.0f; }

// Warp transpose of 16-bit values in groups of 8 lanes, for coalesced epilogue
// stores.  On entry lane L holds feature L's values for tokens 0..7, packed
// w[j] = token 2j | token 2j+1 << 16; on exit it holds features (L & ~7) + 0..7
// of token L & 7, in feature order (one 16-byte store).  Three butterfly steps
// (lane bit i <-> token bit i), two shuffles each.
__device__ __forceinline__ uint4 transpose8x8_u16(const uint32_t (&w)[4], int lane) {
  const bool b0 = lane & 1, b1 = (lane >> 1) & 1, b2 = (lane >> 2) & 1;
  // step 1: keep the tokens whose bit 0 equals lane bit 0, trade the others
  const uint32_t keep_sel = b0 ? 0x5410u : 0x7632u;
  const uint32_t r0 = __shfl_xor_sync(0xffffffffu, __byte_perm(w[0], w[1], keep_sel), 1);
  const uint32_t r1 = __shfl_xor_sync(0xffffffffu, __byte_perm(w[2], w[3], keep_sel), 1);
  const uint32_t se = b0 ? 0x3254u : 0x5410u, so = b0 ? 0x3276u : 0x7610u;
  const uint32_t n0 = __byte_perm(w[0], r0, se), n1 = __byte_perm(w[1], r0, so);
  const uint32_t n2 = __byte_perm(w[2], r1, se), n3 = __byte_perm(w[3], r1, so);
  // step 2: words are tokens (t1, t2) = (j & 1, j >> 1); trade on t1
  const uint32_t ra = __shfl_xor_sync(0xffffffffu, b1 ? n0 : n1, 2);
  const uint32_t rb = __shfl_xor_sync(0xffffffffu, b1 ? n2 : n3, 2);
  const uint32_t x00 = b1 ? ra : n0, x01 = b1 ? n1 : ra, x10 = b1 ? rb : n2, x11 = b1 ? n3 : rb;
  // step 3: trade on t2
  const uint32_t rc = __shfl_xor_sync(0xffffffffu, b2 ? x00 : x10, 4);
  const uint32_t rd = __shfl_xor_sync(0xffffffffu, b2 ? x01 : x11, 4);
  return b2 ? make_uint4(rc, rd, x10, x11) : make_uint4(x00, x01, rc, rd);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

__device__ __forceinline__ void stg128(void* p, const uint4& v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

struct WorkPlan {
  int nb;      // valid blocks
  int T;       // tiles
  int S;       // K splits
  int units;   // scale periods per tile
  int items;
};

// Token blocks to run: n_padded / block_m, limited to the capacity the
// workspace was planned for.  An n_padded outside [0, cap] or off the block
// grid means the alignment came from other arguments: the clamp keeps every
// access inside the workspace and routing_check() reports it.
__device__ __forceinline__ int valid_blocks(const GemmArgs& g) {
  const int np = *g.n_padded;
  return (int)(min((int64_t)max(np, 0), g.cap) / g.block_m);
}
__device__ __forceinline__ bool routing_bad(const GemmArgs& g) {
  const int np = *g.n_padded;
  return np < 0 || (int64_t)np > g.cap || np % g.block_m != 0;
}
// The local expert of token block b, or -1 when the alignment names none of this
// layer's experts (the block is then skipped by every role alike).
__device__ __forceinline__ int block_expert(const GemmArgs& g, int b) {
  const int e = g.expert_ids[b];
  return (unsigned)e < (unsigned)g.L.E ? e : -1;
}

// A sorted slot holds a routed pair when its id is in [0, pairs) (the sentinel
// pairs marks padding; anything else is treated as padding too).
__device__ __forceinline__ bool live_sid(int sid, int pairs) { return (unsigned)sid < (unsigned)pairs; }

// Header flags of the packed blob that make a kernel's fp16 operands inexact:
// the tcgen05 path dequantises INT4 with fp16 scales, the register-fed path
// applies INT4 scales in fp32; both turn MXFP4 scales into fp16 multipliers.
constexpr uint32_t kStatusBlobFlagsTc = kFlagInt4Window | kFlagFp16Window | kFlagGroups;
constexpr uint32_t kStatusBlobFlagsSmall = kFlagFp16Window | kFlagGroups;

// End-of-kernel status of one epilogue thread (after its dependency wait): an
// fp16 value that overflowed (|v| >= 65520 rounds to infinity) or is not a
// number -- an activation that left the fp16 range makes GEMM1's sums
// infinite or NaN, so this also reports inputs outside it -- and (one thread
// of CTA 0) the blob's window flags and an inconsistent alignment.
__device__ __forceinline__ void report_epilogue_status(const GemmArgs& g, float vmax, bool reporter,
                                                       uint32_t blob_flags) {
  if (!(vmax < 65520.0f)) atomicOr(g.status, kStatusRange);
  if (reporter && blockIdx.x == 0) {
    if (*reinterpret_cast<const uint32_t*>(g.packed) & blob_flags) atomicOr(g.status, kStatusRange);
    if (routing_bad(g)) atomicOr(g.status, kStatusRouting);
  }
}

__device__ __forceinline__ WorkPlan make_plan(const GemmArgs& g, bool gemm1) {
  WorkPlan p;
  p.nb = valid_blocks(g);
  p.T = gemm1 ? g.L.T1 : g.L.T2;
  const int stages = gemm1 ? g.L.S1 : g.L.S2;
  p.units = stages / g.L.period;
  const int base = p.T * p.nb;
  const int grid = (int)gridDim.x;
  int S = 1;
  if (base > 0 && base < grid && p.nb * g.block_m <= g.split_rows) {
    // Cost in ninths of a weight stage (~9 KB streamed): every wave streams
    // ceil(units/S) scale periods of weights; a split item also writes its fp32
    // partial (2 x 128 rows x BN x 4 B ~ BN/9 stages) and the last CTA of each
    // item reads S of them back.  Ties keep the smaller S.
    const int bn = g.block_m < 16 ? 16 : g.block_m;
    const int per = g.L.period;
    int best = p.units * per * 9;  // S = 1: one wave of full-K items
    const int smax = min(g.max_split, p.units);
    for (int s = 2; s <= smax; ++s) {
      const int waves = (base * s + grid - 1) / grid;
      const int cost = waves * (((p.units + s - 1) / s) * per * 9 + bn) + s * bn;
      if (cost < best) { best = cost; S = s; }
    }
  }
  p.S = S;
  p.items = base * S;
  return p;
}

// item -> (block, tile, split), tile fastest
__device__ __forceinline__ void decode_item(const WorkPlan& p, int w, int& b, int& tile, int& split) {
  tile = w % p.T;
  const int r = w / p.T;
  split = r % p.S;
  b = r / p.S;
}

__device__ __forceinline__ void stage_range(const WorkPlan& p, const Layout& L, int split, int& s0, int& s1) {
  s0 = split * p.units / p.S * L.period;
  s1 = (split + 1) * p.units / p.S * L.period;
}

// TMA: a 3-D tile (box from the tensor map) at (c0, c1, c2).
__device__ __forceinline__ void tma_tile3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                           uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// TMA gather: four rows (r[0..3]) of a 2-D row-major tensor, 64 fp16 columns
// from c0 (the map's one-row box), land as four consecutive 128-byte rows at
// dst with the map's 128-byte swizzle (applied by shared address, so a 512-byte
// aligned dst continues the 1024-byte swizzle atom it sits in).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int c0, const int4& r,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w), "r"(smem_u32(bar))
      : "memory");
}

// Token rows of block b's slots (padding slots read token 0; their columns are
// discarded) into rows[0, n), by the n first lanes of the calling warp.
__device__ __forceinline__ void load_block_rows(const GemmArgs& g, int b, int n, int lane, int32_t* rows) {
  for (int i = lane; i < n; i += 32) {
    const int sid = g.sorted_ids[b * g.block_m + i];
    rows[i] = (unsigned)sid < (unsigned)g.pairs ? sid / g.top_k : 0;
  }
}

template <int FMT, int STAGE, int BN>
__global__ void __launch_bounds__(GemmCfg<FMT, BN, STAGE>::kThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmArgs g) {
  constexpr bool kG1 = STAGE != kGemm2;          // reads w13 (x rows) rather than w2 (a rows)
  constexpr bool kGated = STAGE == kGemm1Gated;  // tile halves are gate and up rows
  using SM = GemmSmem<BN, FMT>;
  constexpr int kPackedSlotBytes = SM::kPackedSlotBytes;
  using PF = PackedFmt<FMT>;
  constexpr int kSB = SM::kSB, kSP = SM::kSP, kNacc = SM::kNacc, kSA = SM::kSA;
  using Cfg = GemmCfg<FMT, BN, STAGE>;
  constexpr int kNumEpiWarps = Cfg::kEpiWarps, kEpiThreads = Cfg::kEpiThreads, kEpiColStep = Cfg::kEpiColStep;
  constexpr int kNumDequantWarps = Cfg::kDqWarps, kWarpEpi0 = Cfg::kWarpEpi0;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBar);
  uint64_t* p_full = bars;
  uint64_t* p_empty = p_full + kSP;
  uint64_t* a_full = p_empty + kSP;
  uint64_t* a_empty = a_full + kSA;
  uint64_t* b_full = a_empty + kSA;
  uint64_t* b_empty = b_full + kSB;
  uint64_t* acc_full = b_empty + kSB;
  uint64_t* acc_empty = acc_full + kNacc;
  uint64_t* drain_bar = acc_empty + kNacc;
  int32_t* epi_sid = reinterpret_cast<int32_t*>(smem + SM::kEpiSid);
  const uint32_t epi_sid_s = smem_u32(epi_sid);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + SM::kMisc);  // [0] tmem base, [1] abort, [2] last flag
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&misc[1]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Layout& L = g.L;
  constexpr uint32_t kBBytes = BN * 128;                      // activation bytes per stage
  constexpr uint32_t kAccCol0 = kSA * kAColsPerUnit;         // accumulators after the A ring

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSP; ++i) { mbar_init(&p_full[i], 1); mbar_init(&p_empty[i], kNumDequantWarps); }
    for (int i = 0; i < kSA; ++i) { mbar_init(&a_full[i], kNumDequantWarps); mbar_init(&a_empty[i], 1); }
    for (int i = 0; i < kSB; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], 1); }
    for (int i = 0; i < kNacc; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], kNumEpiWarps); }
    mbar_init(drain_bar, 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&misc[0], kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpBProducer && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&g.tmap_b)) : "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  // Ordering against the stream predecessors (programmatic launch): this kernel
  // starts only once its predecessor has passed its own wait.  When the
  // alignment came from moe_align (align_early), it was written two launches
  // back and is complete, with the packed weights, so the weight producer, the
  // dequant warps and the MMA warp need no wait; the activation producer and the
  // epilogue, which read the predecessor's rows or write counters and outputs,
  // wait first.  When the prologue wrote the alignment, everyone waits.
  grid_dependents_launch();
  if (!g.align_early) grid_dependency_wait();

  const WorkPlan plan = make_plan(g, kG1);
  const int64_t tile_bytes = kG1 ? L.tile1_bytes : L.tile2_bytes;
  const uint8_t* wbase = g.packed + (kG1 ? L.w13_off : L.w2_off);

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ TMA producer (packed weights)
    if (lane == 0) {
      // every token block of an expert streams the same tiles: keep them for the
      // blocks that follow (the tile-fastest order runs them close together)
      const uint64_t pol = policy_evict_normal();
      uint32_t pk = 0;
      for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
        int b, tile, split, s0, s1;
        decode_item(plan, w, b, tile, split);
        stage_range(plan, L, split, s0, s1);
        const int e = block_expert(g, b);
        if (e < 0) continue;
        const uint8_t* tb = wbase + ((int64_t)e * plan.T + tile) * tile_bytes;
        for (int s = s0; s < s1; s += kSup, ++pk) {
          const int slot = pk % kSP;
          mbar_wait(&p_empty[slot], ((pk / kSP) + 1) & 1, abort_flag, g.status);
          // a unit starts on a scale period and holds whole periods (INT4 ranges are even)
          const int nst = min(kSup, s1 - s);
          const int bytes = nst / PF::kPeriod * PF::kPeriodBytes;
          const int64_t off = (int64_t)(s / PF::kPeriod) * PF::kPeriodBytes;
          mbar_arrive_expect_tx(&p_full[slot], bytes);
          bulk_g2s(smem + SM::kP + slot * kPackedSlotBytes, tb + off, bytes, &p_full[slot], pol);
        }
      }
      // leave no copy in flight: wait for the last phase of every used slot
      for (uint32_t i = 0; i < (uint32_t)kSP && i < pk; ++i) {
        const uint32_t k = pk - 1 - i;
        mbar_drain(&p_full[k % kSP], (k / kSP) & 1, g.status);
      }
    }
  } else if (warp == kWarpBProducer) {
    // ------------------------------------------------------------ TMA producer (activation rows)
    // the block's rows in sorted order -- GEMM1: x's routed rows, which the
    // prologue placed in sorted order; GEMM2: GEMM1's output -- one 3-D box per
    // unit brings both of its stages (past K it reads zeros)
    if (lane == 0) {
      grid_dependency_wait();
      uint32_t bk = 0;
      for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
        int b, tile, split, s0, s1;
        decode_item(plan, w, b, tile, split);
        stage_range(plan, L, split, s0, s1);
        if (block_expert(g, b) < 0) continue;
        for (int s = s0; s < s1; s += kSup, ++bk) {
          const int bs = bk % kSB;
          mbar_wait(&b_empty[bs], ((bk / kSB) + 1) & 1, abort_flag, g.status);
          mbar_arrive_expect_tx(&b_full[bs], SM::kBUnitBytes);
          tma_tile3d(smem_u32(smem + SM::kB + bs * SM::kBUnitBytes), &g.tmap_b, 0, b * g.block_m, s, &b_full[bs]);
        }
      }
      for (uint32_t i = 0; i < (uint32_t)kSB && i < bk; ++i) {
        const uint32_t k = bk - 1 - i;
        mbar_drain(&b_full[k % kSB], (k / kSB) & 1, g.status);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop so descriptors and TMEM addresses are
    // warp-uniform; one elected lane issues.  __syncwarp reconverges the warp
    // after each wait before the elected issue.
    constexpr uint32_t idesc = idesc_f16_f32(128, BN, 0u);
    uint32_t ak = 0, bk = 0, ic = 0;
    const uint32_t b0 = smem_u32(smem + SM::kB);
    for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
      int b, tile, split, s0, s1;
      decode_item(plan, w, b, tile, split);
      stage_range(plan, L, split, s0, s1);
      if (block_expert(g, b) < 0) continue;  // (every role skips it; no counter moves)
      const int accb = ic % kNacc;
      mbar_wait(&acc_empty[accb], ((ic / kNacc) + 1) & 1, abort_flag, g.status);
      __syncwarp();
      tc_fence_after();
      const uint32_t d0 = tmem_base + kAccCol0 + accb * 2 * BN;
      for (int s = s0; s < s1; s += kSup, ++ak, ++bk) {
        const int as = ak % kSA, bs = bk % kSB;
        const int nst = min(kSup, s1 - s);
        mbar_wait(&a_full[as], (ak / kSA) & 1, abort_flag, g.status);
        mbar_wait(&b_full[bs], (bk / kSB) & 1, abort_flag, g.status);
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kSup; ++j) {
          if (j < nst) {
            const uint32_t a_t = tmem_base + as * kAColsPerUnit + j * kAColsPerStage;
            const uint64_t bd0 = smem_desc_sw128(b0 + bs * SM::kBUnitBytes + j * kBBytes);
            // 4 K-steps x 2 halves; the B start address advances 32 bytes per K-step
            umma_stage_2x4_elect(d0, BN, a_t, bd0, idesc, (s > s0 || j > 0) ? 1u : 0u);
          }
        }
        umma_commit_elect(&a_empty[as]);
        umma_commit_elect(&b_empty[bs]);
      }
      umma_commit_elect(&acc_full[accb]);
      ++ic;
    }
    // all issued MMAs complete before TMEM is released
    umma_commit_elect(drain_bar);
    mbar_drain(drain_bar, 0, g.status);
    __syncwarp();
  } else if (warp < kWarpEpi0) {
    // ------------------------------------------------------------ dequant warps
    // warp -> (TMEM lane quarter q = warp % 4, half): a warp may only touch TMEM
    // lanes 32q..32q+31; each thread dequantises one tile row per stage
    // (with sixteen warps, kh = which 32-element half of every stage the warp takes)
    const int q = warp & 3, half = ((warp - kWarpDequant0) >> 2) & 1, kh = (warp - kWarpDequant0) >> 3;
    constexpr int kHalves = Cfg::kSplitDq ? 1 : 2;  // 32-element halves of a stage per thread
    const int hr = q * 32 + lane;   // row within the half = TMEM lane
    const int r = half * 128 + hr;  // tile row
    const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16) + half * 32;
    uint32_t pk = 0, ak = 0;
    for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
      int b, tile, split, s0, s1;
      decode_item(plan, w, b, tile, split);
      stage_range(plan, L, split, s0, s1);
      if (block_expert(g, b) < 0) continue;
      for (int s = s0; s < s1; s += kSup, ++pk, ++ak) {
        const int ps = pk % kSP, as = ak % kSA;
        const int nst = min(kSup, s1 - s);
        mbar_wait(&p_full[ps], (pk / kSP) & 1, abort_flag, g.status);
        const uint32_t slot = smem_u32(smem + SM::kP) + (uint32_t)ps * kPackedSlotBytes;
        // codes (and scales) of both stages into registers, then release the slot
        uint4 u[kSup][2];
        uint32_t m[kSup][4];  // f16x2 multipliers (INT4: s, s/16; MXFP4: per 32; NVFP4: per 16)
#pragma unroll
        for (int j = 0; j < kSup; ++j) {
          if (j < nst) {
            const uint32_t st = slot + PF::stage_off(j);
            if (FMT == MOE_W_INT4_U4B8) {
              if (j == 0) {  // one scale per 128 K covers both stages
                const uint32_t h = bf16_scale_f16(lds16(st + 2 * r));
                const uint32_t h16 = __half_as_ushort(__hmul(__ushort_as_half((uint16_t)h), __ushort_as_half(0x2C00)));
                m[0][0] = h | (h << 16);      // s
                m[0][1] = h16 | (h16 << 16);  // s / 16
              } else {
                m[j][0] = m[0][0];
                m[j][1] = m[0][1];
              }
            } else if (FMT == MOE_W_MXFP4) {
              const uint32_t sv = lds16(st + 2 * r);
              const uint32_t ac = e8m0x2_mult_f16(sv);
              m[j][0] = __byte_perm(ac, 0, 0x1010);
              m[j][1] = __byte_perm(ac, 0, 0x3232);
            } else if (FMT == kFmtInt4X) {  // the row's entries of both 32-element halves
              const uint2 ev = lds64(st + 8 * r);
              m[j][0] = ev.x;
              m[j][1] = ev.y;
            } else {
              const uint32_t sv = lds32(st + 4 * r);
              const uint32_t lo = e4m3x2_mult_f16(sv & 0xFFFF), hi = e4m3x2_mult_f16(sv >> 16);
              m[j][0] = __byte_perm(lo, 0, 0x1010);
              m[j][1] = __byte_perm(lo, 0, 0x3232);
              m[j][2] = __byte_perm(hi, 0, 0x1010);
              m[j][3] = __byte_perm(hi, 0, 0x3232);
            }
            const uint32_t units = slot + PF::codes_off(j) + 16 * r;
            u[j][0] = lds128(units);
            u[j][1] = lds128(units + 256 * 16);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_empty[ps]);
        // the first half of the first stage is dequantised before the wait for its
        // TMEM slot, so mostly the stores trail the MMAs that free it
#pragma unroll
        for (int j = 0; j < kSup; ++j) {
          if (j < nst) {
            const uint32_t wd[8] = {u[j][0].x, u[j][0].y, u[j][0].z, u[j][0].w,
                                    u[j][1].x, u[j][1].y, u[j][1].z, u[j][1].w};
            // each 32-element half of the stage (TMEM columns 16h .. 16h+15, column c =
            // K pair (2c, 2c+1)) is dequantised into 16 registers and stored on its own
#pragma unroll
            for (int hh = 0; hh < kHalves; ++hh) {
              const int h = kHalves == 2 ? hh : kh;
              uint32_t o[16];
              if (FMT == kFmtInt4X) {  // the words of a half share its entry
                const Int4ZpConst kc = int4zp_const(h ? m[j][1] : m[j][0], g.zp_float);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  uint32_t t4[4];
                  int4x8_f16_zp(h ? wd[2 * t + 1] : wd[2 * t], kc, t4);
#pragma unroll
                  for (int p = 0; p < 4; ++p) o[t + 4 * p] = t4[p];
                }
              } else {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  // word v = (t, h): pair p starts at k = 32h + 2t + 8p -> column 16h + t + 4p;
                  // its group scale is k / 32 (MXFP4) or k / 16 (NVFP4)
                  const uint32_t wv = h ? wd[2 * t + 1] : wd[2 * t];
                  uint32_t t4[4];
                  if (FMT == MOE_W_INT4_U4B8) int4x8_f16(wv, m[j][0], m[j][1], t4);
                  else if (FMT == MOE_W_MXFP4) e2m1x8_f16(wv, h ? m[j][1] : m[j][0], h ? m[j][1] : m[j][0], t4);
                  else e2m1x8_f16(wv, h ? m[j][2] : m[j][0], h ? m[j][3] : m[j][1], t4);
#pragma unroll
                  for (int p = 0; p < 4; ++p) o[t + 4 * p] = t4[p];
                }
              }
              if (j == 0 && hh == 0) {
                mbar_wait(&a_empty[as], ((ak / kSA) + 1) & 1, abort_flag, g.status);
                tc_fence_after();
              }
              tmem_st16(t_lane + as * kAColsPerUnit + j * kAColsPerStage + 16 * h, o);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    grid_dependency_wait();
    const int q = warp & 3;            // TMEM lane quarter
    const int hr = q * 32 + lane;      // row within each 128-row half
    const int et = threadIdx.x - kWarpEpi0 * 32;  // 0..255
    const int csub = (warp - kWarpEpi0) >> 2;      // which 8-column chunks this warp takes
    const float* gs_tab = reinterpret_cast<const float*>(g.packed + (kG1 ? L.gs13_off : L.gs2_off));
    const uint16_t* bias_tab = reinterpret_cast<const uint16_t*>(g.packed + (kG1 ? L.b13_off : L.b2_off));
    const int Npad = L.Npad;
    const int width = kGated ? 2 * Npad : (kG1 ? Npad : L.K);  // partial row width
    const int bias_stride = kGated ? 2 * Npad : (kG1 ? Npad : L.Kpad2);
    uint32_t ic = 0;
    float vmax = 0.0f;  // largest |value| stored as fp16 (NaN ignored)
    for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
      int b, tile, split;
      decode_item(plan, w, b, tile, split);
      const int e = block_expert(g, b);
      if (e < 0) {  // a block inside n_padded without one of this layer's experts
        if (et == 0 && split == 0) atomicOr(g.status, kStatusRouting);
        continue;
      }
      // everything the item's epilogue reads from global memory is fetched before
      // the accumulator wait, off the critical path
      const int jmax = min(BN, g.block_m);
      named_bar_sync(2, kEpiThreads);  // the previous item's readers of epi_sid are done
      if (et < jmax) {
        const int v = g.sorted_ids[b * g.block_m + et];
        epi_sid[et] = v;
        if ((unsigned)v > (unsigned)g.pairs) atomicOr(g.status, kStatusRouting);  // neither a pair nor padding
      }
      const float gsc = gs_tab[e];
      // feature / output rows held by this thread in half 0 and half 1; for
      // gated GEMM1 both halves hold the same feature (gate and up)
      int row0, row1, col0, col1;  // col*: index in the partial row and in the bias row
      if (kGated) { row0 = tile * 128 + hr; row1 = row0; col0 = row0; col1 = Npad + row0; }
      else { row0 = tile * 256 + hr; row1 = row0 + 128; col0 = row0; col1 = row1; }
      float bias0 = 0.f, bias1 = 0.f;
      if (g.has_bias) {
        bias0 = bf16_bits_to_float(bias_tab[(int64_t)e * bias_stride + col0]);
        bias1 = bf16_bits_to_float(bias_tab[(int64_t)e * bias_stride + col1]);
      }
      const bool ok0 = kG1 || row0 < L.K, ok1 = kG1 || row1 < L.K;
      named_bar_sync(2, kEpiThreads);
      const int accb = ic % kNacc;
      mbar_wait(&acc_full[accb], (ic / kNacc) & 1, abort_flag, g.status);
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + kAccCol0 + accb * 2 * BN;
      bool finish = true;  // this CTA writes final results for the item
      if (plan.S > 1) {
        // split-K: store the fp32 partial of this slice, rows by sorted position
        for (int c0 = 8 * csub; c0 < BN; c0 += kEpiColStep) {
          uint32_t v0[8], v1[8];
          tmem_ld8(tb + c0, v0);
          tmem_ld8(tb + BN + c0, v1);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            if (c0 + jj >= jmax) break;
            float* dst = g.partial + ((int64_t)split * g.split_rows + b * g.block_m + c0 + jj) * width;
            if (ok0) __stcg(dst + col0, __uint_as_float(v0[jj]));
            if (ok1) __stcg(dst + col1, __uint_as_float(v1[jj]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[accb]);
        // the CTA barrier orders every epilogue thread's partial stores before one
        // thread's fence and arrival (release); the last CTA's arriving thread fences
        // again before the barrier that lets the others read the partials (acquire)
        named_bar_sync(1, kEpiThreads);
        if (et == 0) {
          __threadfence();
          const unsigned old = atomicInc(reinterpret_cast<unsigned*>(&g.counters[b * plan.T + tile]),
                                         (unsigned)(plan.S - 1));
          misc[2] = old == (unsigned)(plan.S - 1) ? 1u : 0u;
          __threadfence();
        }
        named_bar_sync(1, kEpiThreads);
        finish = misc[2] != 0;
      }
      if (finish) {
        // This thread's token columns come in batches of 8: c0 = 8 * csub + kEpiColStep * it.
        // Each batch loads its 8 sorted ids at once, computes all 8 values and then
        // stores them, so the columns overlap; the next batch's accumulators are
        // requested from TMEM before this batch's math.
        constexpr int kIters = BN / kEpiColStep;
        uint32_t v0[8], v1[8];
        if (plan.S == 1) {
          tmem_ld8(tb + 8 * csub, v0);
          tmem_ld8(tb + BN + 8 * csub, v1);
        }
#pragma unroll 1
        for (int it = 0; it < kIters; ++it) {
          const int c0 = 8 * csub + kEpiColStep * it;
          float f0[8], f1[8];
          if (plan.S == 1) {
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) { f0[jj] = __uint_as_float(v0[jj]); f1[jj] = __uint_as_float(v1[jj]); }
            if (it + 1 < kIters) {
              tmem_ld8(tb + c0 + kEpiColStep, v0);
              tmem_ld8(tb + BN + c0 + kEpiColStep, v1);
            } else {  // every accumulator column of this thread is in registers
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[accb]);
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) { f0[jj] = 0.f; f1[jj] = 0.f; }
            for (int sp = 0; sp < plan.S; ++sp)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                if (c0 + jj < jmax) {
                  const float* src = g.partial + ((int64_t)sp * g.split_rows + b * g.block_m + c0 + jj) * width;
                  if (ok0) f0[jj] += __ldcg(src + col0);
                  if (ok1) f1[jj] += __ldcg(src + col1);
                }
              }
          }
          const uint4 sa = lds128(epi_sid_s + 4 * c0), sb = lds128(epi_sid_s + 4 * c0 + 16);
          const int sid[8] = {(int)sa.x, (int)sa.y, (int)sa.z, (int)sa.w, (int)sb.x, (int)sb.y, (int)sb.z, (int)sb.w};
          const int pos0 = b * g.block_m + c0;
          if (kGated) {
            float av[8];
            if (g.act_kind == MOE_ACT_SILU_MUL) {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) av[jj] = act_fn(MOE_ACT_SILU_MUL, f0[jj] * gsc + bias0, f1[jj] * gsc + bias1, 0.f, 0.f);
            } else {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                av[jj] = act_fn(MOE_ACT_SIGMOID_ALPHA, f0[jj] * gsc + bias0, f1[jj] * gsc + bias1, g.alpha, g.limit);
            }
            // the warp's 32 features x 8 tokens, transposed: each lane stores 8
            // consecutive features of one token (16 bytes)
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = live_sid(sid[2 * j], g.pairs) ? av[2 * j] : 0.0f;
              const float hi = live_sid(sid[2 * j + 1], g.pairs) ? av[2 * j + 1] : 0.0f;
              vmax = fmax_nan(vmax, fmax_nan(fabsf(lo), fabsf(hi)));
              w[j] = pack_f16x2(lo, hi);
            }
            const uint4 o = transpose8x8_u16(w, lane);
            const int tt = lane & 7;
            if (c0 + tt < jmax) stg128(g.a_out + (int64_t)(pos0 + tt) * Npad + (row0 - hr) + q * 32 + (lane & 24), o);
          } else if (kG1) {  // non-gated: both halves are features, a = relu(h)^2
            uint32_t w0[4], w1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const bool l0 = live_sid(sid[2 * j], g.pairs), l1 = live_sid(sid[2 * j + 1], g.pairs);
              const float h00 = f0[2 * j] * gsc + bias0, h01 = f0[2 * j + 1] * gsc + bias0;
              const float h10 = f1[2 * j] * gsc + bias1, h11 = f1[2 * j + 1] * gsc + bias1;
              const float a00 = l0 ? relu2(h00) : 0.0f, a01 = l1 ? relu2(h01) : 0.0f;
              const float a10 = l0 ? relu2(h10) : 0.0f, a11 = l1 ? relu2(h11) : 0.0f;
              // relu^2 >= 0; h * 0 is NaN exactly when h is not finite (relu2 maps NaN to 0)
              vmax = fmax_nan(vmax, fmax_nan(fmax_nan(a00, a01), fmax_nan(a10, a11)));
              vmax = fmax_nan(vmax, (l0 ? (h00 + h10) * 0.0f : 0.0f) + (l1 ? (h01 + h11) * 0.0f : 0.0f));
              w0[j] = pack_f16x2(a00, a01);
              w1[j] = pack_f16x2(a10, a11);
            }
            const uint4 o0 = transpose8x8_u16(w0, lane), o1 = transpose8x8_u16(w1, lane);
            const int tt = lane & 7;
            if (c0 + tt < jmax) {
              uint16_t* dst = g.a_out + (int64_t)(pos0 + tt) * Npad + (row0 - hr) + q * 32 + (lane & 24);
              stg128(dst, o0);
              stg128(dst + 128, o1);
            }
          } else {
            // fp32 rows by pair: for each token column the warp's 32 lanes hold 32
            // consecutive outputs of one pair, one 128-byte store per half; the
            // column test and ok0/ok1 are warp-uniform (K % 64 == 0 and a warp's
            // 32 rows start on a multiple of 32).  Padding columns are stored by
            // no lane.  y is fp32: only a non-finite value of a live column is an
            // error (NaN, or an infinity from an overflow upstream).
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (c0 + j < jmax && live_sid(sid[j], g.pairs)) {
                float* dst = g.y_out + (int64_t)sid[j] * L.K + row0;
                if (ok0) {
                  const float v = f0[j] * gsc + bias0;
                  vmax = fmax_nan(vmax, v * 0.0f);
                  dst[0] = v;
                }
                if (ok1) {
                  const float v = f1[j] * gsc + bias1;
                  vmax = fmax_nan(vmax, v * 0.0f);
                  dst[128] = v;
                }
              }
            }
          }
        }
      }
      ++ic;
    }
    report_epilogue_status(g, vmax, et == 0, kStatusBlobFlagsTc);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace moe
