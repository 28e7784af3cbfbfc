// Device helpers and the tile-native packed-weight layout shared by the repack
// and GEMM kernels of the W4A16 fused-MoE library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_w4a16.h"

namespace moe {

// ----------------------------------------------------------------------------
// Packed weight layout.
//
// Both grouped GEMMs compute 256 weight rows per CTA tile as two 128-row MMA
// operands ("halves").  GEMM1 tile i holds gate rows [128i, 128i+128) in half 0
// and the matching up rows in half 1, so one TMEM lane holds the gate and up
// value of the same intermediate feature and the activation runs in the GEMM1
// epilogue.  Non-gated experts (relu(h)^2) have no up rows: their GEMM1 tile i
// holds rows [256i, 256i+256) of h, like GEMM2.  GEMM2 tile i holds output
// rows [256i, 256i+256).  N is zero-padded to Npad = roundup(N, 128) (gated)
// or roundup(N, 256) (non-gated), GEMM2's rows to roundup(K, 256) (the pages'
// _pad_w13/_pad_w2 tile padding); padded codes decode to 0 and padded bias
// entries are 0, so padded features of a are 0 under every activation.
//
// Each tile is a sequence of K-stages of 64 reduction elements.  A stage's
// packed codes are 8 KiB: uint4 units [j][r] (j = 0,1, r the tile row), so
// that a thread that owns row r reads units r and 256 + r, both
// conflict-free.  A row's 64 codes in a stage are eight 32-bit words v = 2t + h
// (word v is word v % 4 of unit v / 4), each holding four pairs of consecutive
// reduction elements: pair p of word (t, h) starts at k = 32h + 2t + 8p.  This
// is the register fragment of the m16n8k16 tensor-core instruction: fragment
// lane t of a row finds the pairs it needs for the stage's four 16-element
// K-steps -- (2t, 2t+1) and (2t+8, 2t+9) of each -- in words (t, 0) and (t, 1),
// one 8-byte load.  Inside a word, INT4 puts the first element of pair p at
// bits 4p and the second at bits 16+4p (a mask yields an f16x2 pair); FP4 puts
// pair p in byte p, first element in the low nibble, for the hardware
// E2M1x2 -> f16x2 conversion.
//
// Scales ride in front of the stage that first needs them: INT4 (one bf16 per
// 128 = two stages) only in front of even stages, 256 x bf16; MXFP4 two E8M0
// bytes per row per stage (256 x u16); NVFP4 four E4M3 bytes (256 x u32).
//
// INT4 banks with zero points or groups of 32 / 64 are packed as INT4X: one
// 32-bit entry per row and 32-element half stage, two f16 -- the multiplier m
// (the scale) and x: 1024 + z for integer zero points (1032 without), or
// -z * m for float zero points -- 256 x 2 x u32 in front of every stage.
// Act-order banks store each expert matrix's reduction dimension in
// sort_indices order (groups contiguous) and keep w13's permutation for the
// forward, which applies it to x's columns.
// ----------------------------------------------------------------------------
constexpr int kTileRows = 256;       // weight rows per CTA tile (2 x 128)
constexpr int kStageK = 64;          // reduction elements per stage
constexpr int kPackedStageBytes = kTileRows * kStageK / 2;  // 8192

// Which matmul a GEMM kernel instance computes.
enum GemmStage : int {
  kGemm2 = 0,       // y = gs2 * a . W2^T + b2, fp32 rows by pair
  kGemm1Gated = 1,  // a = act(gate, up) of h = gs13 * x . W13^T + b13, fp16
  kGemm1Relu2 = 2,  // a = relu(h)^2, non-gated experts, fp16
};

// Packed format of INT4 banks with zero points or groups below 128 (internal;
// the public enum has the checkpoint formats).
constexpr int kFmtInt4X = 3;

struct Layout {
  int fmt, E, K, N, group;  // fmt: the packed format (MOE_W_* or kFmtInt4X); group as given (-1: per row)
  int zero_kind;   // INT4: 0 none, 1 integer, 2 float zero points
  int act_order;   // INT4: reduction dims stored in sort_indices order
  int gated;       // 1: GEMM1 tiles pair 128 gate rows with their 128 up rows; 0: 256 rows of h
  int Npad;        // roundup(N, 128) gated, roundup(N, 256) non-gated
  int Kpad2;       // roundup(K, 256)
  int T1, T2;      // GEMM1 tiles (Npad/128 or Npad/256), GEMM2 tiles (Kpad2/256)
  int S1, S2;      // stages per tile: K/64 and Npad/64
  int period;      // stages per scale chunk: 2 (INT4) or 1
  int scale_bytes; // scale bytes per chunk
  int64_t period_bytes;   // scale_bytes + period * 8192
  int64_t tile1_bytes, tile2_bytes;
  int64_t w13_off, w2_off, b13_off, b2_off, gs13_off, gs2_off, shift_off, perm13_off, total;
};

__host__ __device__ inline int64_t round_up64(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

__host__ inline bool make_layout(const moe_layer_desc& d, Layout* L) {
  if (d.fmt < 0 || d.fmt > 2 || d.num_experts <= 0 || d.hidden <= 0 || d.inter <= 0) return false;
  const bool int4 = d.fmt == MOE_W_INT4_U4B8;
  if (int4) {
    const int g = d.group_size;
    if (g != 32 && g != 64 && g != 128 && g != -1) return false;
    if (d.zero_kind < 0 || d.zero_kind > 2 || (d.act_order != 0 && d.act_order != 1)) return false;
    if (d.act_order && g < 0) return false;  // act-order groups have a size
    if (d.hidden % 128 || (g > 0 && d.inter % g)) return false;
  } else {
    if (d.group_size != (d.fmt == MOE_W_MXFP4 ? 32 : 16) || d.zero_kind || d.act_order) return false;
    if (d.hidden % 64 || d.inter % d.group_size) return false;
  }
  if (d.non_gated != 0 && (d.non_gated != 1 || d.w13_interleaved)) return false;
  L->fmt = (int4 && (d.zero_kind != 0 || (d.group_size > 0 && d.group_size < 128))) ? kFmtInt4X : d.fmt;
  L->zero_kind = int4 ? d.zero_kind : 0;
  L->act_order = int4 ? d.act_order : 0;
  L->E = d.num_experts;
  L->K = d.hidden;
  L->N = d.inter;
  L->group = d.group_size;
  L->gated = d.non_gated ? 0 : 1;
  const int f1 = L->gated ? 128 : 256;  // intermediate features per GEMM1 tile
  L->Npad = (int)round_up64(d.inter, f1);
  L->Kpad2 = (int)round_up64(d.hidden, 256);
  L->T1 = L->Npad / f1;
  L->T2 = L->Kpad2 / 256;
  L->S1 = d.hidden / kStageK;
  L->S2 = L->Npad / kStageK;
  L->period = L->fmt == MOE_W_INT4_U4B8 ? 2 : 1;
  L->scale_bytes = kTileRows * (L->fmt == kFmtInt4X ? 8 : (L->fmt == MOE_W_NVFP4 ? 4 : 2));
  L->period_bytes = L->scale_bytes + (int64_t)L->period * kPackedStageBytes;
  L->tile1_bytes = (int64_t)(L->S1 / L->period) * L->period_bytes;
  L->tile2_bytes = (int64_t)(L->S2 / L->period) * L->period_bytes;
  int64_t off = 256;  // 256-byte header (reserved)
  L->w13_off = off;
  off += (int64_t)L->E * L->T1 * L->tile1_bytes;
  L->w2_off = off = round_up64(off, 256);
  off += (int64_t)L->E * L->T2 * L->tile2_bytes;
  L->b13_off = off = round_up64(off, 256);
  if (d.has_bias13) off += (int64_t)L->E * (L->gated ? 2 : 1) * L->Npad * 2;
  L->b2_off = off = round_up64(off, 256);
  if (d.has_bias2) off += (int64_t)L->E * L->Kpad2 * 2;
  L->gs13_off = off = round_up64(off, 256);
  off += (int64_t)L->E * 4;
  L->gs2_off = off = round_up64(off, 256);
  off += (int64_t)L->E * 4;
  L->shift_off = off = round_up64(off, 256);  // int32 [2][E]: scale exponent shift of w13 and w2
  off += (int64_t)2 * L->E * 4;
  L->perm13_off = off = round_up64(off, 256);  // act-order: int32 [E][K], x column of packed column k
  if (L->act_order) off += (int64_t)L->E * L->K * 4;
  L->total = round_up64(off, 256);
  return true;
}

// Byte offset of stage s inside a tile and whether it carries scales.
__host__ __device__ inline int64_t stage_offset(const Layout& L, int s) {
  const int q = s / L.period, r = s % L.period;
  return q * L.period_bytes + (r == 0 ? 0 : L.scale_bytes + (int64_t)r * kPackedStageBytes);
}
__host__ __device__ inline bool stage_has_scales(const Layout& L, int s) { return s % L.period == 0; }

// Compile-time view of one format's packed stages (the Layout fields period,
// scale_bytes and period_bytes as constants): stage ss of a chunk that starts
// on a scale period begins at stage_off(ss); its codes at codes_off(ss).
template <int FMT>
struct PackedFmt {
  static constexpr int kPeriod = FMT == MOE_W_INT4_U4B8 ? 2 : 1;
  static constexpr int kScaleBytes = kTileRows * (FMT == kFmtInt4X ? 8 : (FMT == MOE_W_NVFP4 ? 4 : 2));
  static constexpr int kMaxScaleBytesPerStage = FMT == kFmtInt4X ? 2048 : 1024;  // ring slot sizing
  static constexpr int kSlotBytes(int stages) { return stages * (kPackedStageBytes + kMaxScaleBytesPerStage); }
  static constexpr int kPeriodBytes = kScaleBytes + kPeriod * kPackedStageBytes;
  __host__ __device__ static constexpr int stage_off(int ss) {
    return (ss / kPeriod) * kPeriodBytes + (ss % kPeriod ? kScaleBytes + (ss % kPeriod) * kPackedStageBytes : 0);
  }
  __host__ __device__ static constexpr int codes_off(int ss) { return (ss / kPeriod) * kPeriodBytes + kScaleBytes + (ss % kPeriod) * kPackedStageBytes; }
};

// Epilogue factor applied to fp32 accumulators.  FP4 formats dequantise to
// value * 2^-8 (see dequant below), NVFP4 also carries its global scale.
constexpr float kFp4Unscale = 256.0f;

// ----------------------------------------------------------------------------
// Operand windows of the 16-bit tensor-core path and the per-expert scale shift.
//
// Dequantised weights are fp16 tensor-core operands and must be exact there.
// INT4 (q - 8) * s with a bf16 scale s in [2^e, 2^(e+1)) is exact for
// -13 <= e <= 12 (s / 16, used for the odd nibble pairs, keeps its 8
// significant bits above fp16's 2^-24 quantum, and 8 s < 65504).  An MXFP4
// weight e2m1 * 2^(b - 127), produced as e2m1 * 2^(b - 135), is exact for E8M0
// bytes 112 <= b <= 148 (half of 2^(b - 135) stays on the 2^-24 grid, 6 of it
// below 65504).  NVFP4 weights are exact for every E4M3 scale.  Each expert's
// scales of one matrix are multiplied at repack by a power of two 2^d chosen so
// that they fall into the window (d = 0 when they already do), and the epilogue
// factor of that expert carries 2^-d, so the product is unchanged.  When the
// scales of one expert matrix span more than the window, d keeps the largest
// exact and the packed blob's header records the loss.
// ----------------------------------------------------------------------------
constexpr int kInt4ExpMin = -13, kInt4ExpMax = 12;
constexpr int kE8m0Min = 112, kE8m0Max = 148;

// Packed-blob header (its first 256 bytes): word 0 holds these flags.
constexpr uint32_t kFlagInt4Window = 1u;  // an INT4 scale outside the fp16 window (tcgen05 path only)
constexpr uint32_t kFlagFp16Window = 2u;  // an MXFP4 scale byte, or an INT4 scale of a zero-point /
                                          // small-group bank, outside the fp16 window (both GEMM paths)
constexpr uint32_t kFlagGroups = 4u;      // act-order groups that are not group_size indices each

// ----------------------------------------------------------------------------
// Device status word (first 4 bytes of the forward workspace).
// ----------------------------------------------------------------------------
constexpr unsigned kStatusTimeout = 1u;   // a bounded wait ran out
constexpr unsigned kStatusRange = 2u;     // a value left the 16-bit operand range (see above)
constexpr unsigned kStatusRouting = 4u;   // alignment inputs inconsistent with this layer

// ----------------------------------------------------------------------------
// PTX wrappers.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Test the phase with the given parity; while it is incomplete the thread is
// suspended (it issues nothing) until the phase completes or the hint (ns)
// elapses, so waiting roles do not steal issue slots from working warps.
constexpr uint32_t kSuspendHintNs = 1000000u;  // 1 ms
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, records kStatusTimeout in *status, raises the CTA's abort flag
// and returns false; once the flag is up, later waits return at once, so a CTA
// that lost a producer still leaves in bounded time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      // the predecessor kernel clears the status word: record after it completed
      asm volatile("griddepcontrol.wait;" ::: "memory");
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// End-of-role drain: wait (at most kDrainLimitNs) for the phase with the given
// parity, so that no copy or MMA is in flight when the CTA exits or frees
// tensor memory; a drain that runs out records kStatusTimeout.
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 100 ms
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, unsigned* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainLimitNs) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      atomicOr(status, kStatusTimeout);
      return;
    }
  }
}

// 1-D bulk copy global -> shared, completing on an mbarrier (transaction bytes).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}


// Shared-memory loads through 32-bit shared addresses (ordered after the
// barrier waits like every other volatile access).
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}


__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels of the forward are launched with launch_dependent: a kernel may then
// start (set up barriers, tensor memory, descriptor prefetches) while its
// stream predecessor is still finishing.  It calls grid_dependency_wait()
// before its first access to global memory that the predecessor may read or
// write; the wait returns once the predecessor has completed and its writes
// are visible (at once when there is no programmatic predecessor).
// grid_dependents_launch() lets the next kernel start launching early.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// tcgen05 operations issued from a converged warp by its elected leader
// (elect.sync picks the lowest active lane, so every call in a converged loop
// issues from the same thread, as tcgen05.commit requires).  The operands are
// computed by the whole warp, so they stay warp-uniform.
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
// One 64-K stage of both 128-row halves (8 MMAs: K-steps kk = 0..3, halves
// h = 0, 1) from the elected lane: D_h (+)= A_h[kk] * B[kk], with A_h[kk] at
// TMEM column a + 32h + 8kk, B[kk] described by b_desc advanced 32 bytes per
// K-step and D_h at column d + h * n_cols.  `accumulate` applies to the first
// K-step; the later ones always accumulate.
__device__ __forceinline__ void umma_stage_2x4_elect(uint32_t d, uint32_t n_cols, uint32_t a, uint64_t b_desc,
                                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 d1, a1, a2, a3, a4, a5, a6, a7;\n\t.reg .b64 b1, b2, b3;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "add.u32 d1, %0, %1;\n\t"
      "add.u32 a1, %2, 32;\n\tadd.u32 a2, %2, 8;\n\tadd.u32 a3, %2, 40;\n\t"
      "add.u32 a4, %2, 16;\n\tadd.u32 a5, %2, 48;\n\tadd.u32 a6, %2, 24;\n\tadd.u32 a7, %2, 56;\n\t"
      "add.u64 b1, %3, 2;\n\tadd.u64 b2, %3, 4;\n\tadd.u64 b3, %3, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %3, %4, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [d1], [a1], %3, %4, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b1, %4, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [d1], [a3], b1, %4, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b2, %4, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [d1], [a5], b2, %4, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b3, %4, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [d1], [a7], b3, %4, 1;\n\t}" ::"r"(d),
      "r"(n_cols), "r"(a), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Store 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// 32 TMEM lanes x 16 consecutive 32-bit columns (one per register).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// 32 TMEM lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzled
// canonical layout: rows of 128 bytes (64 bf16 of one K-stage), 8-row atoms of
// 1024 bytes (stride-dimension offset), 16-byte chunk c of row r stored at chunk
// c ^ (r % 8).  The atom base must be 1024-byte aligned; advancing the start
// address by 32 bytes selects the next K=16 slice.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading-dim offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride-dim offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                          // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                          // swizzle: 128 B
  return d;
}

// Instruction descriptor: kind::f16, A and B both fp16 (ab_bf16 = 0) or both
// bf16 (ab_bf16 = 1), D = fp32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, uint32_t ab_bf16) {
  return (1u << 4)                         // D format fp32
         | (ab_bf16 << 7)                  // A format
         | (ab_bf16 << 10)                 // B format
         | ((uint32_t)(N >> 3) << 17)      // N / 8
         | ((uint32_t)(M >> 4) << 24);     // M / 16
}


// ---------------------------------------------------------------- register-fed tensor cores
// D (16 x 8, fp32) += A (16 x 16, fp16, row-major fragment) * B (16 x 8, fp16).
// Fragment of lane (g = lane / 4, t = lane % 4): a0 = A[g][2t..2t+1],
// a1 = A[g+8][2t..2t+1], a2 = A[g][2t+8..2t+9], a3 = A[g+8][2t+8..2t+9];
// b0 = B[2t..2t+1][g], b1 = B[2t+8..2t+9][g]; d0, d1 = D[g][2t..2t+1],
// d2, d3 = D[g+8][2t..2t+1].
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four 8 x 8 16-bit matrices from shared memory; lane l gives the address of
// row l % 8 of matrix l / 8 and receives row l / 4, columns 2(l % 4)..+1 of each.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// max / min that propagate NaN (a running max over stored values then also
// catches NaN, and a clamp keeps a NaN input NaN, as torch's clamp does).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// ---------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ float round_bf16(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

// ---------------------------------------------------------------- dequant
// All tensor-core operands are fp16.  Every dequantised weight is exact in fp16:
// INT4 (q - 8) * s has at most 3 + 8 significant bits; E2M1 times a power of two
// (MXFP4) or times an E4M3 value (NVFP4) at most 2 + 4.  FP4 weights are
// produced as value * scale * 2^-8 (kFp4Unscale restores the 2^8 in the fp32
// epilogue), which keeps large block scales inside the fp16 range.

// 8 INT4 (uint4b8) codes of one word -> its 4 pairs as f16x2.  Word layout from
// the repack: pair p has its first element at bits 4p, its second at 16 + 4p.
// Pairs 0 and 2 are (1024 + q) - 1032; pairs 1 and 3 sit 4 bits higher and
// are (1024 + 16q) - 1152 = 16(q - 8), scaled by s / 16.
__device__ __forceinline__ void int4x8_f16(uint32_t w, uint32_t s2, uint32_t s2_16, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t t[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x64006400u,
                         (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x64006400u};
  const __half2 c1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 c1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 sa = *reinterpret_cast<const __half2*>(&s2), sb = *reinterpret_cast<const __half2*>(&s2_16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&t[i]), (i & 1) ? c1152 : c1032);
    const __half2 r = __hmul2(v, (i & 1) ? sb : sa);
    o[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// 8 E2M1 codes of one word (byte p = pair p, first element in the low nibble)
// -> 4 f16x2 with the hardware conversion; pairs 0, 1 times m01, pairs 2, 3
// times m23.
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t m01, uint32_t m23, uint32_t (&o)[4]) {
  uint32_t v[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t m = i < 2 ? m01 : m23;
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&v[i]), *reinterpret_cast<const __half2*>(&m));
    o[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// 8 INT4 codes of one word with a zero point, from a 32-element half stage's
// entry: low-nibble pairs (1024 + q) - c_lo, high-nibble pairs (1024 + 16q) -
// c_hi, then times m (m / 16 for the high pairs) plus o, in one fused op.  For
// integer zero points c_lo = 1024 + z, c_hi = 1024 + 16z, o = 0 (q - z exact,
// one rounding of (q - z) * m); for float zero points c = 1024 and o = -z * m.
struct Int4ZpConst {
  uint32_t c_lo, c_hi, m, m16, o;  // f16x2 (both halves equal)
};
__device__ __forceinline__ Int4ZpConst int4zp_const(uint32_t entry, int zp_float) {
  const uint32_t m = entry & 0xFFFFu, x = entry >> 16;
  const __half one024 = __ushort_as_half(0x6400);
  const __half hx = __ushort_as_half((uint16_t)x);
  // c_hi = 16 c_lo - 15360 = 1024 + 16 z (exact)
  const __half chi = __hsub(__hmul(hx, __ushort_as_half(0x4C00)), __ushort_as_half(0x7380));
  const uint16_t clo_b = zp_float ? (uint16_t)0x6400 : (uint16_t)x;
  const uint16_t chi_b = zp_float ? (uint16_t)0x6400 : __half_as_ushort(chi);
  const uint16_t o_b = zp_float ? (uint16_t)x : (uint16_t)0;
  const uint16_t m16_b = __half_as_ushort(__hmul(__ushort_as_half((uint16_t)m), __ushort_as_half(0x2C00)));
  (void)one024;
  Int4ZpConst k;
  k.c_lo = (uint32_t)clo_b | ((uint32_t)clo_b << 16);
  k.c_hi = (uint32_t)chi_b | ((uint32_t)chi_b << 16);
  k.m = m | (m << 16);
  k.m16 = (uint32_t)m16_b | ((uint32_t)m16_b << 16);
  k.o = (uint32_t)o_b | ((uint32_t)o_b << 16);
  return k;
}
__device__ __forceinline__ void int4x8_f16_zp(uint32_t w, const Int4ZpConst& k, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t t[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x64006400u,
                         (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x64006400u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t c = (i & 1) ? k.c_hi : k.c_lo, m = (i & 1) ? k.m16 : k.m;
    const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&t[i]), *reinterpret_cast<const __half2*>(&c));
    const __half2 r = __hfma2(v, *reinterpret_cast<const __half2*>(&m), *reinterpret_cast<const __half2*>(&k.o));
    o[i] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Multipliers (as f16 bit patterns, to be paired by the caller).
__device__ __forceinline__ uint32_t bf16_scale_f16(uint32_t sbits) {
  return __half_as_ushort(__float2half_rn(__uint_as_float(sbits << 16)));
}
// Two E8M0 bytes (low = first) -> f16x2 of 2^(b-127) * 2^-8 = 2^(b-135) each:
// normal for b >= 121, a subnormal power of two for 111 <= b <= 120, 0 below
// (the conversion rounds to nearest even); 255 is NaN.  Bytes above 150 do not
// occur: the repack shift keeps them in [112, 148].  The fp32 value 2^(b-127)
// is the byte shifted into the exponent field (b = 0 gives 0; 255 gets a
// mantissa bit, NaN), scaled by 2^-8 exactly.
__device__ __forceinline__ uint32_t e8m0x2_mult_f16(uint32_t two_bytes) {
  const uint32_t b0 = two_bytes & 0xFFu, b1 = (two_bytes >> 8) & 0xFFu;
  const float f0 = __uint_as_float((b0 << 23) | (b0 == 255u ? 0x400000u : 0u)) * 0.00390625f;
  const float f1 = __uint_as_float((b1 << 23) | (b1 == 255u ? 0x400000u : 0u)) * 0.00390625f;
  const __half2 h = __floats2half2_rn(f0, f1);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Two E4M3 bytes (low = first) -> f16x2 of value * 2^-8 (exact).
__device__ __forceinline__ uint32_t e4m3x2_mult_f16(uint32_t two_bytes) {
  uint32_t v;
  asm("{\n\t.reg .b16 h;\n\t"
      "cvt.u16.u32 h, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h;\n\t}"
      : "=r"(v)
      : "r"(two_bytes));
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&v),
                            __halves2half2(__ushort_as_half(0x1C00), __ushort_as_half(0x1C00)));  // 2^-8
  return *reinterpret_cast<const uint32_t*>(&r);
}
// 8 bf16 -> 8 fp16 (round to nearest; exact inside the fp16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  const __half2 h = __floats2half2_rn(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace moe
