// Host side of the C ABI: argument checks, the launch-configuration chooser,
// the workspace plan and the forward's launch sequence (GEMM1 + activation ->
// GEMM2 -> combine), all enqueued on the caller's stream without host syncs.
#include <cuda.h>
#include <cmath>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "combine.cuh"
#include "gemm_launch.cuh"
#include "prologue.cuh"

namespace moe {

constexpr int64_t kSplitBudgetBytes = 64ll << 20;  // cap on each split-K partial area
constexpr int kMaxSplit = 16;

std::atomic<int> g_test_starve_wait{0};  // moe_set_test_starve_wait

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// Token blocks up to this size run on the register-fed kernel.
constexpr int kSmallBlockMax = 32;

// Everything the forward places in the caller's workspace, in bytes from its start.
struct WsPlan {
  int64_t cap, blocks;
  int grid;
  int max_split1, max_split2, rows1, rows2;
  int64_t status_off, counters1_off, counters2_off, header_bytes, align_off, xh_off, a_off, y_off, part1_off,
      part2_off, total;
};

bool plan_workspace(const Layout& L, int M, int top_k, int block_m, WsPlan* w,
                    int64_t split_budget = kSplitBudgetBytes) {
  const int64_t cap = moe_align_capacity(M, top_k, L.E, block_m);
  if (cap < 0) return false;
  const int grid = device_sm_count();
  if (grid <= 0) return false;
  const int64_t pairs = (int64_t)M * top_k;
  w->cap = cap;
  w->blocks = cap / block_m;
  w->grid = grid;
  int64_t per1, per2;
  if (block_m <= kSmallBlockMax) {
    // register-fed kernels (stream-K, 8- and 16-token blocks): two fp32 partial tiles
    // [256 rows][block_m] per CTA; max_split 2 turns the division on, 1 (no room, or
    // 32-token blocks, which run whole items) falls back to whole items
    w->rows1 = w->rows2 = 0;
    per1 = per2 = block_m < kSmallBlockMax ? (int64_t)2 * grid * kTileRows * block_m * 4 : 0;
    w->max_split1 = w->max_split2 = per1 > 0 && per1 <= split_budget ? 2 : 1;
  } else {
    // split-K only runs while tiles * blocks < grid, so the partial rows stay below this bound
    w->rows1 = (int)std::min<int64_t>(cap, (int64_t)((grid - 1) / L.T1 + 1) * block_m);
    w->rows2 = (int)std::min<int64_t>(cap, (int64_t)((grid - 1) / L.T2 + 1) * block_m);
    // fp32 partial rows: GEMM1 gate and up (or h alone), GEMM2 the output width
    per1 = (int64_t)w->rows1 * (L.gated ? 2 : 1) * L.Npad * 4;
    per2 = (int64_t)w->rows2 * L.K * 4;
    w->max_split1 = (int)std::max<int64_t>(1, std::min<int64_t>(kMaxSplit, per1 ? split_budget / per1 : 1));
    w->max_split2 = (int)std::max<int64_t>(1, std::min<int64_t>(kMaxSplit, per2 ? split_budget / per2 : 1));
  }
  int64_t off = 0;
  w->status_off = off;
  off += 256;
  w->counters1_off = off;
  off += (int64_t)L.T1 * w->blocks * 4;
  w->counters2_off = off;
  off += (int64_t)L.T2 * w->blocks * 4;
  w->header_bytes = off;  // zeroed by the prologue every call
  off = round_up64(off, 256);
  // the alignment, when the forward computes it: sorted [cap], experts [cap/B], n_padded, and each
  // pair's sorted position [pairs]
  w->align_off = off;
  off = round_up64(off + (cap + w->blocks + 1 + pairs) * 4, 256);
  // x as fp16: its own rows [M, K] for the register-fed kernels (block_m <= 32),
  // the routed rows in sorted order [cap, K] for the tcgen05 kernels and for
  // act-order banks (whose x columns follow each expert's order)
  w->xh_off = off;
  off = round_up64(off + (block_m <= 32 && !L.act_order ? (int64_t)M : cap) * L.K * 2, 256);
  w->a_off = off;
  off = round_up64(off + cap * L.Npad * 2, 256);
  w->y_off = off;
  off = round_up64(off + pairs * L.K * 4, 256);  // y, fp32
  // (a GEMM that cannot split, max_split 1, never touches its partial area)
  const bool streamk = block_m <= kSmallBlockMax;
  w->part1_off = off;
  off = round_up64(off + (w->max_split1 > 1 ? (streamk ? 1 : (int64_t)w->max_split1) * per1 : 0), 256);
  w->part2_off = off;
  off = round_up64(off + (w->max_split2 > 1 ? (streamk ? 1 : (int64_t)w->max_split2) * per2 : 0), 256);
  w->total = off;
  return true;
}

cudaError_t launch_gemm(int fmt, bool small, int stage, int bn, const GemmArgs& g, int grid, cudaStream_t st) {
  switch (fmt) {
    case MOE_W_INT4_U4B8: return launch_gemm_int4(small, stage, bn, g, grid, st);
    case MOE_W_MXFP4: return launch_gemm_mxfp4(small, stage, bn, g, grid, st);
    case MOE_W_NVFP4: return launch_gemm_nvfp4(small, stage, bn, g, grid, st);
    case kFmtInt4X: return launch_gemm_int4x(small, stage, bn, g, grid, st);
    default: return cudaErrorInvalidValue;
  }
}


bool valid_block_m(int b) { return b == 8 || b == 16 || b == 32 || b == 64 || b == 128; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A row-major [rows, cols] fp16 matrix as a 2-D map with a one-row box of 64
// columns and the 128-byte swizzle, for four-row TMA gathers.
bool make_gather_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || cols % 64) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64u, 1u};
  const cuuint32_t es[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major [rows, cols] fp16 matrix viewed as [rows][cols / 64][64]: dims (64, rows, cols / 64),
// boxes of 64 x box_rows x box_stages landing as [stage][row][64] with the
// 128-byte swizzle, so one copy brings several 64-column stages.
bool make_act_map3(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int box_rows, int box_stages) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || cols % 64) return false;
  const cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128u};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, (cuuint32_t)box_stages};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaEvent_t g_trace[4] = {nullptr, nullptr, nullptr, nullptr};
bool g_tracing = false;

inline cudaError_t trace(int i, cudaStream_t st) {
  return g_tracing ? cudaEventRecord(g_trace[i], st) : cudaSuccess;
}

}  // namespace moe

using namespace moe;

namespace moe {

// Expected token blocks of size B one expert occupies when its row count is
// Poisson(lambda): the sum over n >= 1 of P(n) * ceil(n / B).
static double expected_blocks(double lambda, int B) {
  if (lambda > 200.0) return lambda / B + 0.5;  // the rounding up adds half a block on average
  double p = std::exp(-lambda), e = 0.0;  // p = P(n), from P(0)
  const int nmax = (int)(lambda + 12.0 * std::sqrt(lambda + 1.0)) + 16;
  for (int n = 1; n <= nmax; ++n) {
    p *= lambda / n;
    e += p * ((n + B - 1) / B);
  }
  return e;
}

}  // namespace moe

extern "C" int moe_choose_block_m(const moe_layer_desc* desc, int M, int top_k, int num_routed_ids) {
  if (!desc || M < 0 || top_k <= 0 || num_routed_ids <= 0) return MOE_ERR_INVALID;
  // expected rows per local expert: routed pairs spread over the routed id range
  const double rows = (double)M * top_k / (double)num_routed_ids;
  // Every token block streams (and dequantises) its expert's weights once, so a
  // block size costs the expected number of blocks (Poisson rows per expert)
  // times one block's cost.  Block costs relative to a 16-token block of the
  // register-fed kernel, measured on GB300 at K = 2880..4096:
  //                      8     16    32 (register-fed)   64    128 (tcgen05)
  //   INT4              0.86  1     1.56                1.32  1.68
  //   MXFP4             0.86  1     1.34                0.93  1.09
  //   NVFP4             0.86  1     1.34                0.94  1.26
  // Below K = 1024 the tcgen05 tiles are too short for those costs: the
  // register-fed sizes serve up to 32 rows and 64-token tiles the rest (with
  // 128-token tiles the epilogue, which does not overlap the next tile's MMAs
  // there, outweighs the better MMA rate).
  const bool int4 = desc->fmt == MOE_W_INT4_U4B8, mx = desc->fmt == MOE_W_MXFP4;
  const int sizes[5] = {8, 16, 32, 64, 128};
  const double cost[5] = {0.86, 1.0, int4 ? 1.56 : 1.34, int4 ? 1.32 : (mx ? 0.93 : 0.94),
                          int4 ? 1.68 : (mx ? 1.09 : 1.26)};
  const bool short_k = desc->hidden < 1024;
  if (short_k && rows > 32.0) return 64;
  int best = 8;
  double best_cost = 0.0;
  for (int i = 0; i < (short_k ? 3 : 5); ++i) {
    const double c = cost[i] * expected_blocks(rows, sizes[i]);
    if (i == 0 || c < best_cost) {
      best = sizes[i];
      best_cost = c;
    }
  }
  return best;
}

extern "C" int64_t moe_workspace_size(const moe_layer_desc* desc, int M, int top_k, int block_m) {
  Layout L;
  WsPlan w;
  if (!desc || !make_layout(*desc, &L) || M < 0 || top_k <= 0 || !valid_block_m(block_m)) return -1;
  if (!plan_workspace(L, M, top_k, block_m, &w)) return -1;
  return w.total;
}

namespace moe {

// Argument rules shared by both forward entry points (everything but the workspace).
static int check_forward_args(const moe_layer_desc* desc, const void* packed, const void* x, int M, int top_k,
                              const int32_t* topk_ids, const float* topk_weights, const int32_t* sorted_ids,
                              const int32_t* expert_ids, const int32_t* n_padded, int block_m, int act,
                              const void* post_norm_w, const void* out, Layout* L) {
  if (!desc || !make_layout(*desc, L)) return MOE_ERR_INVALID;
  if (M < 0 || top_k <= 0 || top_k > 16 || !valid_block_m(block_m)) return MOE_ERR_INVALID;
  if (desc->num_experts > 1024) return MOE_ERR_INVALID;  // moe_align's limit: no alignment exists for more
  // gated experts take a gated activation, non-gated ones relu^2
  if (L->gated ? (act != MOE_ACT_SILU_MUL && act != MOE_ACT_SIGMOID_ALPHA) : act != MOE_ACT_RELU2)
    return MOE_ERR_INVALID;
  if ((int64_t)M * top_k >= (int64_t)1 << 31) return MOE_ERR_INVALID;
  if (M == 0) return MOE_OK;
  if (!packed || !x || !topk_ids || !topk_weights || !out) return MOE_ERR_INVALID;
  // the alignment comes from moe_align (all three) or from the forward itself (none)
  const int given = (sorted_ids != nullptr) + (expert_ids != nullptr) + (n_padded != nullptr);
  if (given != 0 && given != 3) return MOE_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(packed) & 255) || (reinterpret_cast<uintptr_t>(x) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15) || (reinterpret_cast<uintptr_t>(post_norm_w) & 15))
    return MOE_ERR_INVALID;
  return MOE_OK;
}

// The launch sequence on a checked argument set and a workspace laid out by `w`.
static int forward_impl(const moe_layer_desc* desc, const Layout& L, const WsPlan& w, const void* packed,
                        const void* x, int M, int top_k, const int32_t* topk_ids, const float* topk_weights,
                        int expert_base, const int32_t* sorted_ids, const int32_t* expert_ids,
                        const int32_t* n_padded, int block_m, int act, float alpha, float limit,
                        float routed_scaling_factor, const void* post_norm_w, float norm_eps, void* out,
                        void* workspace, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  const bool small = block_m <= kSmallBlockMax;
  const int bn = block_m;  // token columns per tile

  // The alignment: the caller's (from moe_align, two launches back by the time
  // the GEMMs start) or computed here by the prologue into the workspace.
  const bool own_align = sorted_ids == nullptr;
  if (own_align) {
    int32_t* base = reinterpret_cast<int32_t*>(ws + w.align_off);
    sorted_ids = base;
    expert_ids = base + w.cap;
    n_padded = base + w.cap + w.blocks;
  }

  GemmArgs g{};
  // GEMM1's activation rows: the register-fed kernel gathers x's rows (fp16) by
  // token, the tcgen05 kernel reads them in sorted order; GEMM2 reads GEMM1's
  // fp16 output in sorted order
  CUtensorMap map2;
  const bool gather_rows = small && !L.act_order;  // else x's routed rows in sorted order
  if (gather_rows ? !make_gather_map(&g.tmap_b, ws + w.xh_off, L.K, M)
                  : !make_act_map3(&g.tmap_b, ws + w.xh_off, L.K, w.cap, bn, small ? kSmallChunk : kSup))
    return MOE_ERR_CUDA;
  if (!make_act_map3(&map2, ws + w.a_off, L.Npad, w.cap, bn, small ? kSmallChunk : kSup)) return MOE_ERR_CUDA;

  // prologue: [alignment,] x to fp16 (rows or sorted order), status word and split-K counters to zero.
  // Aligning in a launch of its own lets the GEMMs find the alignment two
  // launches back and stream weights while the prologue runs, which is worth
  // more than one launch less for decode-sized blocks and for short batches
  // (measured on GB300).  Large batches on the tcgen05 path align and place
  // x's routed rows in one launch (no second pass over the sorted slots).
  const bool split_align = own_align && (small || (int64_t)M * top_k * L.K < ((int64_t)1 << 25));
  PrologueArgs pa{};
  pa.pairs = M * top_k;
  pa.cap = w.cap;
  if (split_align) {
    PrologueArgs al{};
    al.topk_ids = topk_ids;
    al.pairs = M * top_k;
    al.expert_base = expert_base;
    al.E = L.E;
    al.block_m = block_m;
    al.cap = w.cap;
    al.sorted_ids = const_cast<int32_t*>(sorted_ids);
    al.expert_ids = const_cast<int32_t*>(expert_ids);
    al.n_padded = const_cast<int32_t*>(n_padded);
    if (launch_prologue(al, 0, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (own_align && !split_align) {
    pa.topk_ids = topk_ids;
    pa.expert_base = expert_base;
    pa.E = L.E;
    pa.block_m = block_m;
    pa.sorted_ids = const_cast<int32_t*>(sorted_ids);
    pa.expert_ids = const_cast<int32_t*>(expert_ids);
    pa.n_padded = const_cast<int32_t*>(n_padded);
    pa.pair_pos = const_cast<int32_t*>(n_padded) + 1;
    if (!small) pa.align_ctas = align_copy_ctas(M * top_k, L.K, w.grid);
  } else {
    pa.given_sorted = sorted_ids;
    pa.given_expert_ids = expert_ids;
    pa.given_n_padded = n_padded;
    pa.block_m = block_m;
    pa.E = L.E;
  }
  pa.x = static_cast<const uint16_t*>(x);
  pa.M = M;
  pa.K = L.K;
  pa.top_k = top_k;
  if (gather_rows) pa.xh = reinterpret_cast<uint16_t*>(ws + w.xh_off);
  else pa.xs = reinterpret_cast<uint16_t*>(ws + w.xh_off);
  if (L.act_order) pa.perm13 = reinterpret_cast<const int32_t*>(pk + L.perm13_off);
  pa.zero = reinterpret_cast<uint32_t*>(ws);
  pa.zero_words = w.header_bytes / 4;
  if (launch_prologue(pa, w.grid, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (trace(0, st) != cudaSuccess) return MOE_ERR_CUDA;

  g.L = L;
  g.packed = pk;
  g.sorted_ids = sorted_ids;
  g.expert_ids = expert_ids;
  g.n_padded = n_padded;
  g.cap = w.cap;
  g.pairs = M * top_k;
  g.top_k = top_k;
  g.align_early = (own_align && !split_align) ? 0 : 1;
  g.zp_float = L.zero_kind == 2;
  g.gemm1_rows_sorted = gather_rows ? 0 : 1;
  g.block_m = block_m;
  g.act_kind = act;
  g.alpha = alpha;
  g.limit = limit;
  g.a_out = reinterpret_cast<uint16_t*>(ws + w.a_off);
  g.y_out = reinterpret_cast<float*>(ws + w.y_off);
  g.status = reinterpret_cast<unsigned*>(ws + w.status_off);
  g.test_starve_wait = g_test_starve_wait.load(std::memory_order_relaxed);

  // GEMM1 + activation
  g.has_bias = desc->has_bias13 != 0;
  g.max_split = w.max_split1;
  g.split_rows = w.rows1;
  g.partial = reinterpret_cast<float*>(ws + w.part1_off);
  g.counters = reinterpret_cast<int32_t*>(ws + w.counters1_off);
  if (launch_gemm(L.fmt, small, L.gated ? kGemm1Gated : kGemm1Relu2, bn, g, w.grid, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (trace(1, st) != cudaSuccess) return MOE_ERR_CUDA;

  // GEMM2
  g.tmap_b = map2;
  g.has_bias = desc->has_bias2 != 0;
  g.max_split = w.max_split2;
  g.split_rows = w.rows2;
  g.partial = reinterpret_cast<float*>(ws + w.part2_off);
  g.counters = reinterpret_cast<int32_t*>(ws + w.counters2_off);
  if (launch_gemm(L.fmt, small, kGemm2, bn, g, w.grid, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (trace(2, st) != cudaSuccess) return MOE_ERR_CUDA;

  // combine
  CombineArgs c{};
  c.M = M;
  c.top_k = top_k;
  c.K = L.K;
  c.expert_base = expert_base;
  c.E = L.E;
  c.topk_ids = topk_ids;
  c.topk_weights = topk_weights;
  c.y = reinterpret_cast<const float*>(ws + w.y_off);
  c.post_norm_w = static_cast<const uint16_t*>(post_norm_w);
  c.norm_eps = norm_eps;
  c.rsf = routed_scaling_factor;
  c.out = static_cast<uint16_t*>(out);
  if (launch_combine(c, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (trace(3, st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_w4a16_forward(const moe_layer_desc* desc, const void* packed, const void* x, int M, int top_k,
                                 const int32_t* topk_ids, const float* topk_weights, int expert_base,
                                 const int32_t* sorted_ids, const int32_t* expert_ids, const int32_t* n_padded,
                                 int block_m, int act, float alpha, float limit, float routed_scaling_factor,
                                 const void* post_norm_w, float norm_eps, void* out, void* workspace,
                                 int64_t workspace_bytes, void* stream) {
  Layout L;
  const int rc = check_forward_args(desc, packed, x, M, top_k, topk_ids, topk_weights, sorted_ids, expert_ids,
                                    n_padded, block_m, act, post_norm_w, out, &L);
  if (rc != MOE_OK || M == 0) return rc;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return MOE_ERR_INVALID;
  WsPlan w;
  if (!plan_workspace(L, M, top_k, block_m, &w)) return MOE_ERR_CUDA;
  if (workspace_bytes < w.total) return MOE_ERR_WORKSPACE;
  return forward_impl(desc, L, w, packed, x, M, top_k, topk_ids, topk_weights, expert_base, sorted_ids, expert_ids,
                      n_padded, block_m, act, alpha, limit, routed_scaling_factor, post_norm_w, norm_eps, out,
                      workspace, stream);
}

// Allocation-free variant.  Some callers cannot hand over device memory of
// their own: code that runs inside a stream that a framework is recording into
// a graph, where a cudaMalloc would break the recording, or plugins of an
// engine that owns every device allocation.  For them the workspace is a fixed
// array in this library's device image, reserved by the CUDA runtime when the
// module loads, so no call here allocates.  One array per device and process:
// two calls in flight at once (two streams, two host threads) share it and
// race.  The prologue kernel zeroes the status word and the split-K counters
// on every call, so the array needs no initialisation.
namespace moe {

constexpr int64_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
// smaller split-K partial areas than the caller-workspace path so that the
// usual shapes fit in the fixed array
constexpr int64_t kNoAllocSplitBudget = 4ll << 20;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device, looked up once per device.
void* noalloc_scratch() {
  static std::atomic<void*> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace moe

extern "C" int moe_w4a16_forward_noalloc(const moe_layer_desc* desc, const void* packed, const void* x, int M,
                                         int top_k, const int32_t* topk_ids, const float* topk_weights,
                                         int expert_base, const int32_t* sorted_ids, const int32_t* expert_ids,
                                         const int32_t* n_padded, int block_m, int act, float alpha, float limit,
                                         float routed_scaling_factor, const void* post_norm_w, float norm_eps,
                                         void* out, void* stream) {
  Layout L;
  const int rc = check_forward_args(desc, packed, x, M, top_k, topk_ids, topk_weights, sorted_ids, expert_ids,
                                    n_padded, block_m, act, post_norm_w, out, &L);
  if (rc != MOE_OK || M == 0) return rc;
  WsPlan w;
  if (!plan_workspace(L, M, top_k, block_m, &w, kNoAllocSplitBudget)) return MOE_ERR_CUDA;
  if (w.total > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = noalloc_scratch();
  if (!scratch) return MOE_ERR_CUDA;
  return forward_impl(desc, L, w, packed, x, M, top_k, topk_ids, topk_weights, expert_base, sorted_ids, expert_ids,
                      n_padded, block_m, act, alpha, limit, routed_scaling_factor, post_norm_w, norm_eps, out,
                      scratch, stream);
}

extern "C" int moe_set_trace_events(void* const* events, int n) {
  if (!events || n == 0) {
    g_tracing = false;
    return MOE_OK;
  }
  if (n != 4) return MOE_ERR_INVALID;
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return MOE_ERR_INVALID;
    g_trace[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_tracing = true;
  return MOE_OK;
}

extern "C" int moe_get_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(workspace, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & kStatusTimeout) return MOE_ERR_TIMEOUT;
  if (v & kStatusRouting) return MOE_ERR_INVALID;
  if (v & kStatusRange) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

extern "C" int moe_set_test_starve_wait(int on) {
  g_test_starve_wait.store(on ? 1 : 0, std::memory_order_relaxed);
  return MOE_OK;
}

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}
