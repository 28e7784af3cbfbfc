// Grouped W4A16 GEMM on tcgen05 tensor cores (sm_103a), shared by GEMM1 (w13,
// fused gated activation) and GEMM2 (w2).
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
//   * a persistent grid (one CTA per SM) walks work items (tile, block, K-split)
//     derived on the device from n_padded, splitting K when there are too few
//     items to fill the GPU (decode) and reducing the fp32 partials in fixed
//     split order (bitwise reproducible; the last CTA to arrive on a per-item
//     counter does the reduction, no spinning);
//   * operands: GEMM2 and the INT4 GEMM1 run fp16 x fp16 (every dequantised
//     weight is exact in fp16, and the activation operand keeps 11 significant
//     bits); the FP4 GEMM1 runs bf16 x bf16 on the bf16 input as is (E2M1 times
//     its scale is exact in bf16).  For the INT4 GEMM1 the dequant warps convert
//     the staged bf16 input rows to fp16 in shared memory.  Accumulation, bias,
//     scales and the activation are fp32; only the tensor-core operands are 16-bit;
//   * warp roles: a TMA producer streams each stage's packed codes + scales
//     (one contiguous chunk thanks to the repack) with 1-D bulk copies; a loader
//     warp gathers the block's activation rows with cp.async; eight dequant
//     warps turn 4-bit codes into bf16 in registers and write the 128-byte
//     swizzled K-major operand; one thread issues tcgen05.mma into a
//     double-buffered TMEM accumulator; four epilogue warps read TMEM, add bias,
//     scale, round to bf16 and apply the activation (GEMM1) or scatter rows to
//     their pairs (GEMM2) while the next item's MMAs run.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kSA = 2;                 // dequantised-A ring
constexpr int kSB = 4;                 // activation (B) ring
constexpr int kSP = 8;                 // packed-weight ring
constexpr int kBLoadAhead = 2;         // cp.async groups in flight in the loader
constexpr int kNumDequantWarps = 8;
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpLoader = 2, kWarpDequant0 = 3;
constexpr int kWarpEpi0 = kWarpDequant0 + kNumDequantWarps;  // 11..14
constexpr int kGemmThreads = (kWarpEpi0 + 4) * 32;          // 480
constexpr int kHalfBytes = 128 * 128;                       // one 128-row x 64-K bf16 operand
constexpr int kPackedSlotBytes = kPackedStageBytes + 1024;  // codes + largest scale block

struct GemmArgs {
  Layout L;
  const uint8_t* packed;      // repacked blob
  const uint16_t* act;        // GEMM1: x bf16 [M, K]; GEMM2: a fp16 rows [cap, Npad]
  int act_ld;                 // row stride of act in elements
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* n_padded;
  int pairs;                  // M * top_k (sentinel value)
  int top_k;
  int block_m;
  int has_bias;
  int act_kind;               // moe_act
  float alpha, limit;
  int max_split;
  int split_rows;             // rows of each split-K partial slice
  uint16_t* a_out;            // GEMM1 output, fp16 [cap, Npad]
  float* y_out;               // GEMM2 output, fp32 [pairs, K]
  int32_t* inv_pos;           // GEMM2: pair -> sorted position
  float* partial;             // split-K partials
  int32_t* counters;          // GEMM1 split-K arrival counters [T1 * cap / block_m]
  int32_t* split_used;        // GEMM2: chosen split (read by the combine)
  unsigned* status;
};

template <int BN>
struct GemmSmem {
  static constexpr int kA = 0;
  static constexpr int kB = kA + kSA * 2 * kHalfBytes;
  static constexpr int kP = kB + kSB * BN * 128;
  static constexpr int kBar = kP + kSP * kPackedSlotBytes;
  // barriers: p_full, p_empty, a_full, a_empty, b_full, b_empty, acc_full[2], acc_empty[2], drain
  static constexpr int kNumBars = 2 * kSP + 2 * kSA + 2 * kSB + 4 + 1;
  static constexpr int kRows = kBar + kNumBars * 8;
  static constexpr int kMisc = kRows + BN * 4;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ float act_fn(int kind, float g, float u, float alpha, float limit) {
  if (kind == MOE_ACT_SILU_MUL) return g / (1.0f + __expf(-g)) * u;
  const float gc = fminf(g, limit);
  const float uc = fminf(fmaxf(u, -limit), limit);
  return gc / (1.0f + __expf(-alpha * gc)) * (uc + 1.0f);
}

struct WorkPlan {
  int nb;      // valid blocks
  int T;       // tiles
  int S;       // K splits
  int units;   // scale periods per tile
  int items;
};

__device__ __forceinline__ WorkPlan make_plan(const GemmArgs& g, bool gated) {
  WorkPlan p;
  p.nb = *g.n_padded / g.block_m;
  p.T = gated ? g.L.T1 : g.L.T2;
  const int stages = gated ? g.L.S1 : g.L.S2;
  p.units = stages / g.L.period;
  const int base = p.T * p.nb;
  int S = 1;
  if (base > 0 && base < (int)gridDim.x) {
    S = ((int)gridDim.x + base - 1) / base;
    S = min(S, min(g.max_split, p.units));
    if (p.nb * g.block_m > g.split_rows) S = 1;  // partial slices sized for this bound
  }
  p.S = S;
  p.items = base * S;
  return p;
}

__device__ __forceinline__ void decode_item(const WorkPlan& p, int w, int& b, int& tile, int& split) {
  b = w % p.nb;
  const int r = w / p.nb;
  split = r % p.S;
  tile = r / p.S;
}

template <int FMT, bool GATED, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmArgs g) {
  using SM = GemmSmem<BN>;
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
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  int32_t* row_tab = reinterpret_cast<int32_t*>(smem + SM::kRows);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + SM::kMisc);  // [0] tmem base, [1] abort, [2] last flag
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&misc[1]);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Layout& L = g.L;
  constexpr uint32_t kTmemCols = (4 * BN) < 32 ? 32 : 4 * BN;  // two accumulators of 2*BN columns
  constexpr bool kF16 = (FMT == MOE_W_INT4_U4B8) || !GATED;   // fp16 operands, else bf16
  constexpr bool kConvertB = GATED && FMT == MOE_W_INT4_U4B8;  // bf16 input rows -> fp16 in smem

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSP; ++i) { mbar_init(&p_full[i], 1); mbar_init(&p_empty[i], kNumDequantWarps); }
    for (int i = 0; i < kSA; ++i) { mbar_init(&a_full[i], kNumDequantWarps); mbar_init(&a_empty[i], 1); }
    for (int i = 0; i < kSB; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
    mbar_init(drain_bar, 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&misc[0], kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];

  const WorkPlan plan = make_plan(g, GATED);
  if (GATED == false && blockIdx.x == 0 && threadIdx.x == 0) *g.split_used = plan.S;
  const int64_t tile_bytes = GATED ? L.tile1_bytes : L.tile2_bytes;
  const uint8_t* wbase = g.packed + (GATED ? L.w13_off : L.w2_off);

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t pk = 0;
      for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
        int b, tile, split;
        decode_item(plan, w, b, tile, split);
        const int e = g.expert_ids[b];
        const int s0 = split * plan.units / plan.S * L.period, s1 = (split + 1) * plan.units / plan.S * L.period;
        const uint8_t* tb = wbase + ((int64_t)e * plan.T + tile) * tile_bytes;
        for (int s = s0; s < s1; ++s, ++pk) {
          const int slot = pk % kSP;
          mbar_wait(&p_empty[slot], ((pk / kSP) + 1) & 1, abort_flag, g.status);
          const int bytes = stage_bytes(L, s);
          mbar_arrive_expect_tx(&p_full[slot], bytes);
          bulk_g2s(smem + SM::kP + slot * kPackedSlotBytes, tb + stage_offset(L, s), bytes, &p_full[slot], pol);
        }
      }
      // leave no copy in flight: wait for the last phase of every used slot
      for (uint32_t i = 0; i < kSP && i < pk; ++i) {
        const uint32_t k = pk - 1 - i;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&p_full[k % kSP], (k / kSP) & 1) && global_timer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == kWarpLoader) {
    // ------------------------------------------------------------ activation rows (cp.async)
    uint32_t bk = 0, retired = 0;
    for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
      int b, tile, split;
      decode_item(plan, w, b, tile, split);
      const int s0 = split * plan.units / plan.S * L.period, s1 = (split + 1) * plan.units / plan.S * L.period;
      __syncwarp();
      for (int j = lane; j < BN; j += 32) {
        int row = -1;
        if (j < g.block_m) {
          if (GATED) {
            const int sid = g.sorted_ids[b * g.block_m + j];
            row = sid < g.pairs ? sid / g.top_k : -1;
          } else {
            row = b * g.block_m + j;
          }
        }
        row_tab[j] = row;
      }
      __syncwarp();
      for (int s = s0; s < s1; ++s, ++bk) {
        const int slot = bk % kSB;
        mbar_wait(&b_empty[slot], ((bk / kSB) + 1) & 1, abort_flag, g.status);
        const uint32_t dst0 = smem_u32(smem + SM::kB + slot * BN * 128);
        for (int c = lane; c < BN * 8; c += 32) {
          const int j = c >> 3, ck = c & 7;
          const int row = row_tab[j];
          const uint16_t* src = g.act + (row >= 0 ? (int64_t)row * g.act_ld + s * kStageK + ck * 8 : 0);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst0 + sw128_offset(j, ck)), "l"(src),
                       "r"(row >= 0 ? 16 : 0)
                       : "memory");
        }
        cp_async_commit();
        if (bk + 1 - retired > kBLoadAhead) {
          cp_async_wait<kBLoadAhead>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&b_full[retired % kSB]);
          ++retired;
        }
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    for (; retired < bk; ++retired)
      if (lane == 0) mbar_arrive(&b_full[retired % kSB]);
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, BN, kF16 ? 0u : 1u);
      uint32_t ak = 0, bk = 0, ic = 0;
      const uint32_t a0 = smem_u32(smem + SM::kA), b0 = smem_u32(smem + SM::kB);
      for (int w = blockIdx.x; w < plan.items; w += gridDim.x, ++ic) {
        int b, tile, split;
        decode_item(plan, w, b, tile, split);
        const int s0 = split * plan.units / plan.S * L.period, s1 = (split + 1) * plan.units / plan.S * L.period;
        const int accb = ic & 1;
        mbar_wait(&acc_empty[accb], ((ic >> 1) + 1) & 1, abort_flag, g.status);
        tc_fence_after();
        const uint32_t d0 = tmem_base + accb * 2 * BN;
        for (int s = s0; s < s1; ++s, ++ak, ++bk) {
          const int as = ak % kSA, bs = bk % kSB;
          mbar_wait(&a_full[as], (ak / kSA) & 1, abort_flag, g.status);
          if (!kConvertB) mbar_wait(&b_full[bs], (bk / kSB) & 1, abort_flag, g.status);
          tc_fence_after();
          const uint32_t abase = a0 + as * 2 * kHalfBytes, bbase = b0 + bs * BN * 128;
#pragma unroll
          for (int kk = 0; kk < kStageK / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(bbase + kk * 32);
            const uint32_t acc = (s > s0 || kk > 0) ? 1u : 0u;
            umma_bf16(d0, smem_desc_sw128(abase + kk * 32), bd, idesc, acc);
            umma_bf16(d0 + BN, smem_desc_sw128(abase + kHalfBytes + kk * 32), bd, idesc, acc);
          }
          umma_commit(&a_empty[as]);
          umma_commit(&b_empty[bs]);
        }
        umma_commit(&acc_full[accb]);
      }
      // all issued MMAs complete before TMEM is released
      umma_commit(drain_bar);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp < kWarpEpi0) {
    // ------------------------------------------------------------ dequant warps
    const int r = threadIdx.x - kWarpDequant0 * 32;  // tile row 0..255
    const int half = r >> 7, hr = r & 127;
    uint32_t pk = 0, ak = 0;
    uint32_t mult[4] = {0, 0, 0, 0};  // per-stage multipliers (bf16x2)
    for (int w = blockIdx.x; w < plan.items; w += gridDim.x) {
      int b, tile, split;
      decode_item(plan, w, b, tile, split);
      const int s0 = split * plan.units / plan.S * L.period, s1 = (split + 1) * plan.units / plan.S * L.period;
      for (int s = s0; s < s1; ++s, ++pk, ++ak) {
        const int ps = pk % kSP, as = ak % kSA;
        mbar_wait(&p_full[ps], (pk / kSP) & 1, abort_flag, g.status);
        const unsigned char* slot = smem + SM::kP + ps * kPackedSlotBytes;
        const bool has_sc = stage_has_scales(L, s);
        if (has_sc) {
          if (FMT == MOE_W_INT4_U4B8) {
            const uint32_t sv = reinterpret_cast<const uint16_t*>(slot)[r];
            const uint32_t m = kF16 ? bf16_scale_f16(sv) : sv;
            mult[0] = m | (m << 16);
          } else if (FMT == MOE_W_MXFP4) {
            const uint32_t sv = reinterpret_cast<const uint16_t*>(slot)[r];
            const uint32_t m0 = kF16 ? e8m0_mult_f16(sv & 0xFF) : e8m0_mult_bits(sv & 0xFF);
            const uint32_t m1 = kF16 ? e8m0_mult_f16(sv >> 8) : e8m0_mult_bits(sv >> 8);
            mult[0] = m0 | (m0 << 16);
            mult[1] = m1 | (m1 << 16);
          } else {
            const uint32_t sv = reinterpret_cast<const uint32_t*>(slot)[r];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t b8 = (sv >> (8 * q)) & 0xFF;
              const uint32_t m = kF16 ? e4m3_mult_f16(b8) : e4m3_mult_bits(b8);
              mult[q] = m | (m << 16);
            }
          }
        }
        const uint4* codes = reinterpret_cast<const uint4*>(slot + (has_sc ? L.scale_bytes : 0));
        const uint4 u0 = codes[r], u1 = codes[256 + r];
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_empty[ps]);
        mbar_wait(&a_empty[as], ((ak / kSA) + 1) & 1, abort_flag, g.status);
        const uint32_t words[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const uint32_t dst = smem_u32(smem + SM::kA + as * 2 * kHalfBytes + half * kHalfBytes);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t m2;
          if (FMT == MOE_W_INT4_U4B8) m2 = mult[0];
          else if (FMT == MOE_W_MXFP4) m2 = mult[c >> 2];
          else m2 = mult[c >> 1];
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (FMT == MOE_W_INT4_U4B8)
              o[i] = kF16 ? dq_int4_pair_f16(words[c], i, m2) : dq_int4_pair(words[c], i, m2);
            else
              o[i] = kF16 ? dq_e2m1_pair_f16(words[c], i, m2) : dq_e2m1_pair(words[c], i, m2);
          }
          st_shared_v4(dst + sw128_offset(hr, c), o[0], o[1], o[2], o[3]);
        }
        if (kConvertB) {
          // the staged bf16 input rows of this stage -> fp16, in place
          const int bs = ak % kSB;
          mbar_wait(&b_full[bs], (ak / kSB) & 1, abort_flag, g.status);
          const uint32_t bbase = smem_u32(smem + SM::kB + bs * BN * 128);
          for (int c = r; c < BN * 8; c += 256) {
            const uint32_t addr = bbase + c * 16;
            uint32_t v0, v1, v2, v3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                         : "r"(addr)
                         : "memory");
            st_shared_v4(addr, bf16x2_to_f16x2(v0), bf16x2_to_f16x2(v1), bf16x2_to_f16x2(v2),
                         bf16x2_to_f16x2(v3));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;            // TMEM lane quarter
    const int hr = q * 32 + lane;      // row within each 128-row half
    const int et = threadIdx.x - kWarpEpi0 * 32;  // 0..127
    const float* gs_tab = reinterpret_cast<const float*>(g.packed + (GATED ? L.gs13_off : L.gs2_off));
    const uint16_t* bias_tab = reinterpret_cast<const uint16_t*>(g.packed + (GATED ? L.b13_off : L.b2_off));
    const int Npad = L.Npad;
    uint32_t ic = 0;
    for (int w = blockIdx.x; w < plan.items; w += gridDim.x, ++ic) {
      int b, tile, split;
      decode_item(plan, w, b, tile, split);
      const int e = g.expert_ids[b];
      const float gsc = gs_tab[e];
      const int accb = ic & 1;
      mbar_wait(&acc_full[accb], (ic >> 1) & 1, abort_flag, g.status);
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + accb * 2 * BN;
      // feature / output rows held by this thread in half 0 and half 1
      int row0, row1;
      if (GATED) { row0 = tile * 128 + hr; row1 = row0; }
      else { row0 = tile * 256 + hr; row1 = row0 + 128; }
      float bias0 = 0.f, bias1 = 0.f;
      if (g.has_bias) {
        if (GATED) {
          bias0 = bf16_bits_to_float(bias_tab[(int64_t)e * 2 * Npad + row0]);
          bias1 = bf16_bits_to_float(bias_tab[(int64_t)e * 2 * Npad + Npad + row1]);
        } else {
          bias0 = bf16_bits_to_float(bias_tab[(int64_t)e * L.Kpad2 + row0]);
          bias1 = bf16_bits_to_float(bias_tab[(int64_t)e * L.Kpad2 + row1]);
        }
      }
      const int jmax = min(BN, g.block_m);
      bool finish = true;  // this CTA writes final results for the item
      if (plan.S > 1) {
        // split-K: store the fp32 partial of this slice, rows by sorted position
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tb + c0, v0);
          tmem_ld16(tb + BN + c0, v1);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (c0 + jj >= jmax) break;
            const int pos = b * g.block_m + c0 + jj;
            if (GATED) {
              float* dst = g.partial + ((int64_t)split * g.split_rows + pos) * 2 * Npad;
              __stcg(dst + row0, __uint_as_float(v0[jj]));
              __stcg(dst + Npad + row1, __uint_as_float(v1[jj]));
            } else {
              float* dst = g.partial + ((int64_t)split * g.split_rows + pos) * L.K;
              if (row0 < L.K) __stcg(dst + row0, __uint_as_float(v0[jj]));
              if (row1 < L.K) __stcg(dst + row1, __uint_as_float(v1[jj]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[accb]);
        if (GATED) {
          __threadfence();
          named_bar_sync(1, 128);
          if (et == 0) {
            const unsigned old = atomicInc(reinterpret_cast<unsigned*>(&g.counters[tile * (*g.n_padded / g.block_m) + b]),
                                           (unsigned)(plan.S - 1));
            misc[2] = old == (unsigned)(plan.S - 1) ? 1u : 0u;
          }
          named_bar_sync(1, 128);
          finish = misc[2] != 0;
          if (finish) __threadfence();
        } else {
          finish = false;  // the combine reduces GEMM2 partials
        }
      }
      if (!GATED && tile == 0 && split == 0) {
        for (int j = et; j < g.block_m; j += 128) {
          const int sid = g.sorted_ids[b * g.block_m + j];
          if (sid < g.pairs) g.inv_pos[sid] = b * g.block_m + j;
        }
      }
      if (finish) {
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float f0[16], f1[16];
          if (plan.S == 1) {
            uint32_t v0[16], v1[16];
            tmem_ld16(tb + c0, v0);
            tmem_ld16(tb + BN + c0, v1);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) { f0[jj] = __uint_as_float(v0[jj]); f1[jj] = __uint_as_float(v1[jj]); }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) { f0[jj] = 0.f; f1[jj] = 0.f; }
            for (int sp = 0; sp < plan.S; ++sp)
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                if (c0 + jj >= jmax) break;
                const float* src = g.partial + ((int64_t)sp * g.split_rows + b * g.block_m + c0 + jj) * 2 * Npad;
                f0[jj] += __ldcg(src + row0);
                f1[jj] += __ldcg(src + Npad + row1);
              }
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (c0 + jj >= jmax) break;
            const int pos = b * g.block_m + c0 + jj;
            const int sid = g.sorted_ids[pos];
            if (GATED) {
              const float hg = f0[jj] * gsc + bias0;
              const float hu = f1[jj] * gsc + bias1;
              const float a = sid < g.pairs ? act_fn(g.act_kind, hg, hu, g.alpha, g.limit) : 0.0f;
              g.a_out[(int64_t)pos * Npad + row0] = __half_as_ushort(__float2half_rn(a));
            } else if (sid < g.pairs) {
              float* dst = g.y_out + (int64_t)sid * L.K;
              if (row0 < L.K) dst[row0] = f0[jj] * gsc + bias0;
              if (row1 < L.K) dst[row1] = f1[jj] * gsc + bias1;
            }
          }
        }
        if (plan.S == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[accb]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace moe
