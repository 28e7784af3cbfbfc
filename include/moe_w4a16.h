/*
 * moe_w4a16.h -- C ABI of the GB300 (sm_103a) weight-only 4-bit fused
 * Mixture-of-Experts layer.
 *
 * The layer is the expert computation of SGLang's Marlin MoE runner as the
 * source pages describe it:
 *   - "013-moe-middle-tiles.py" (open-kernel-challenge), kernel_fn: routing
 *     alignment (moe_align_block_size) -> grouped GEMM1 against packed 4-bit
 *     w13 -> silu_and_mul -> grouped GEMM2 against w2 -> post-expert-norm
 *     weighted sum; Weights / Inputs / Config give the tensor layouts;
 *   - "Marlin MoE kernel occupancy ..." (sglang PR #31552): the fused op
 *     fused_marlin_moe(...) with per-expert bias (kHasBias) and the
 *     expert-parallel block filter (kIsEP), and the per-expert reference loop of
 *     test_fused_marlin_moe_large_non_ep_schedule (top-k weights applied in the
 *     combine, tolerance |out - ref| <= 0.06 + 0.04 |ref|), including its
 *     non-gated experts (is_gated=False, activation "relu2");
 *   - "SM120 MXFP4 MoE ... Marlin" (sglang PR #28231): MXFP4 weights with GPT-OSS
 *     interleaved gate/up rows (deinterleave_moe_mxfp4_w13_for_marlin), zero
 *     padding of the intermediate dimension (_pad_w13/_pad_w2), the sigmoid-alpha
 *     activation (swiglu_gpt_oss_sigmoid_alpha_contiguous) and the shape rule of
 *     check_moe_marlin_supports_layer(allow_tile_padding): hidden % 64 == 0 and
 *     intermediate % group_size == 0.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to memory the current CUDA
 *     device can access; the caller owns all memory.  The library never
 *     allocates device memory and never synchronises the stream, except where an
 *     entry point says so.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All device work is enqueued on it, in order.
 *   - Every entry point returns a moe_status (size queries return -1 for
 *     invalid arguments, the status-name lookup a string).  Argument errors that the host can
 *     see are returned synchronously and nothing is enqueued.  Errors found on the
 *     device (a bounded wait that ran out) are recorded in the workspace status
 *     word and reported by moe_get_status().
 *   - Tensors are dense, row-major, with the shapes given below.
 *   - bf16 values are passed as their 16-bit patterns.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID = -1,      /* bad argument (null pointer, shape, enum, alignment) */
    MOE_ERR_UNSUPPORTED = -2,  /* valid request this build does not implement */
    MOE_ERR_CUDA = -3,         /* a CUDA runtime call failed */
    MOE_ERR_TIMEOUT = -4,      /* a device-side bounded wait ran out */
    MOE_ERR_WORKSPACE = -5     /* workspace too small */
} moe_status;

/* Weight formats.  Codes are 4 bits, two per byte, element 2j in the low nibble
 * and element 2j+1 in the high nibble of byte j of a row.
 *   INT4_U4B8: code q stands for q - 8 ("uint4b8"), or q - z with a zero point z
 *              (moe_layer_desc.zero_kind); one bf16 scale per group of
 *              group_size (32, 64, 128, or -1: one group per row) along the
 *              reduction dimension, groups given per reduction index by g_idx
 *              when act_order (the w*_zeros / is_zp_float / g_idx /
 *              sort_indices / group_blocks of fused_marlin_moe and the Marlin
 *              template, "Marlin MoE kernel occupancy ..." (sglang PR #31552)).
 *   MXFP4:     E2M1 codes; one E8M0 scale byte (2^(b-127)) per 32.
 *   NVFP4:     E2M1 codes; one FP8 E4M3 scale per 16, times one fp32 global
 *              scale per expert (the same for gate and up rows). */
typedef enum moe_wfmt { MOE_W_INT4_U4B8 = 0, MOE_W_MXFP4 = 1, MOE_W_NVFP4 = 2 } moe_wfmt;

/* Activations.  Gated experts: gate = first N outputs of GEMM1, up = the next N.
 *   SILU_MUL:      silu(gate) * up                         (silu_and_mul)
 *   SIGMOID_ALPHA: g = min(gate, limit), u = clamp(up, -limit, limit),
 *                  g * sigmoid(alpha * g) * (u + 1)         (GPT-OSS)
 * Non-gated experts (moe_layer_desc.non_gated = 1): GEMM1 has N outputs h.
 *   RELU2:         relu(h)^2   (activation="relu2", is_gated=False of the
 *                  large-M schedule test in "Marlin MoE kernel occupancy ...",
 *                  sglang PR #31552) */
typedef enum moe_act { MOE_ACT_SILU_MUL = 0, MOE_ACT_SIGMOID_ALPHA = 1, MOE_ACT_RELU2 = 2 } moe_act;

/* Shape of one layer's expert bank held by this GPU. */
typedef struct moe_layer_desc {
    int32_t fmt;              /* moe_wfmt */
    int32_t num_experts;      /* E: experts held here, local ids 0..E-1 */
    int32_t hidden;           /* K: model width (GEMM1 reduction, GEMM2 output); % 64 == 0, and
                                 % 128 == 0 for INT4 */
    int32_t inter;            /* N: expert intermediate width; % group_size == 0 */
    int32_t group_size;       /* INT4: 32, 64, 128 or -1 (one group per row); MXFP4 32; NVFP4 16 */
    int32_t w13_interleaved;  /* 1: w13 rows stored gate0, up0, gate1, up1, ... (GPT-OSS) */
    int32_t has_bias13;       /* 1: per-expert bf16 bias on GEMM1 outputs */
    int32_t has_bias2;        /* 1: per-expert bf16 bias on GEMM2 outputs */
    int32_t non_gated;        /* 0: w13 holds gate and up rows (2N); 1: w13 holds N rows and
                                 the activation is MOE_ACT_RELU2 (w13_interleaved must be 0) */
    int32_t zero_kind;        /* INT4 only: 0 none (uint4b8); 1 integer zero points, one byte
                                 0..15 per (row, group); 2 float zero points (is_zp_float),
                                 one bf16 per (row, group); W = (q - z) * s */
    int32_t act_order;        /* INT4 only: 1 = both matrices carry g_idx / sort_indices
                                 (groups of group_size indices each; group_size 32..128) */
} moe_layer_desc;

/* ------------------------------------------------------------------ repack
 * Load-time conversion of checkpoint tensors into the kernels' tile-native
 * layout ("013-moe-middle-tiles.py", prepare(): prepare_moe_nvfp4_layer_for_marlin;
 * PR #28231: deinterleave, _pad_w13/_pad_w2).  One device pass; the output is an
 * opaque blob of moe_repack_size() bytes that moe_w4a16_forward reads.
 *
 * Inputs (device pointers):
 *   w13    uint8 [E, R, K/2]    packed codes; R = 2N gated (gate rows then up rows, or
 *                               interleaved), R = N non-gated
 *   w13_s  [E, R, K/g]          bf16 (INT4) | uint8 E8M0 (MXFP4) | uint8 E4M3 (NVFP4)
 *   w13_gs fp32 [E]             NVFP4 only, else NULL
 *   b13    bf16 [E, R]          when has_bias13, else NULL (same row order as w13)
 *   w2     uint8 [E, K, N/2];  w2_s [E, K, N/g];  w2_gs fp32 [E] (NVFP4);
 *   b2     bf16 [E, K]          when has_bias2, else NULL
 *   packed device buffer of moe_repack_size() bytes, 256-byte aligned.
 * Returns MOE_ERR_INVALID for shapes outside the rules above or non_gated
 * together with w13_interleaved.  (The ValueError cases of
 * deinterleave_moe_mxfp4_w13_for_marlin -- an odd row count, scale or bias rows
 * not matching the weight rows -- cannot arise here: every row count derives
 * from desc, 2N for interleaved banks.)
 * Each expert matrix's scales are stored shifted by a power of two into the
 * kernels' exact fp16 window, the shift undone by the expert's fp32 factor (see
 * "Operand range" at moe_w4a16_forward); a matrix whose scales spread wider
 * than the window marks the blob, and forwards on it report
 * MOE_ERR_UNSUPPORTED through moe_get_status. */
int64_t moe_repack_size(const moe_layer_desc* desc);
int moe_repack_weights(const moe_layer_desc* desc, const void* w13, const void* w13_s,
                       const float* w13_gs, const void* b13, const void* w2, const void* w2_s,
                       const float* w2_gs, const void* b2, void* packed, void* stream);

/* The checkpoint tensors of one bank, for moe_repack_weights_ex (device
 * pointers; those a bank does not have are NULL). */
typedef struct moe_repack_tensors {
    const void* w13;              /* uint8 [E, R, K/2] */
    const void* w13_s;            /* [E, R, K/g] */
    const float* w13_gs;          /* fp32 [E] (NVFP4) */
    const void* b13;              /* bf16 [E, R] */
    const void* w13_zeros;        /* [E, R, K/g]: uint8 (zero_kind 1) or bf16 (zero_kind 2) */
    const int32_t* w13_g_idx;     /* int32 [E, K]: group of each reduction index (act_order) */
    const int32_t* w13_sort_indices; /* int32 [E, K]: reduction indices by ascending group */
    const void* w2;               /* uint8 [E, K, N/2] */
    const void* w2_s;             /* [E, K, N/g] */
    const float* w2_gs;           /* fp32 [E] (NVFP4) */
    const void* b2;               /* bf16 [E, K] */
    const void* w2_zeros;         /* [E, K, N/g] */
    const int32_t* w2_g_idx;      /* int32 [E, N] */
    const int32_t* w2_sort_indices;  /* int32 [E, N] */
} moe_repack_tensors;

/* moe_repack_weights with the INT4 variants: zero points (desc->zero_kind),
 * act-order (desc->act_order) and group sizes 32 / 64 / 128 / -1.  With
 * act_order the reduction dimension of each expert matrix is stored in
 * sort_indices order, so that its groups are contiguous; w2's order is folded
 * into the order of w13's output features (and their bias), so GEMM1 writes
 * the activations in the order GEMM2 reads them, and the forward permutes x's
 * columns per expert as it places the routed rows.  The groups must hold
 * group_size indices each (g_idx[sort_indices[k]] == k / group_size); a bank
 * that breaks this marks the blob, and forwards on it report
 * MOE_ERR_UNSUPPORTED.  Arithmetic: with integer zero points (q - z) * s may
 * need 12 significant bits and is rounded once to fp16 (relative error <=
 * 2^-12); with float zero points q * s - z * s is formed in fp16 (z * s rounded
 * at repack, one more rounding in the product).  Returns MOE_ERR_INVALID for a
 * missing tensor the descriptor requires. */
int moe_repack_weights_ex(const moe_layer_desc* desc, const moe_repack_tensors* t, void* packed, void* stream);

/* ------------------------------------------------------------------ align
 * Routing alignment ("013-moe-middle-tiles.py", kernel_fn: moe_align_block_size;
 * the -1 block marker of the PR #31552 kIsEP block filter).  Pair p = t*top_k + j
 * with routed id topk_ids[p] is local when expert_base <= id < expert_base + E.
 * Outputs (device):
 *   sorted_ids int32 [cap]        local pairs grouped by expert (ascending local id),
 *                                 ascending p within an expert, each expert's run
 *                                 padded to a multiple of block_m with the sentinel
 *                                 M*top_k; empty experts take no block; entries at
 *                                 or past n_padded are the sentinel;
 *   expert_ids int32 [cap/block_m] local expert of each block, -1 past n_padded;
 *   n_padded   int32 [1]           sum over experts of ceil(count/block_m)*block_m.
 * cap = moe_align_capacity(M, top_k, E, block_m) = roundup(M*top_k +
 * min(E, M*top_k)*(block_m-1), block_m), the worst case over all routings.
 * block_m must be 8, 16, 32, 64 or 128; E <= 1024; M*top_k < 2^31.
 * topk_ids: int32 [M, top_k] device. */
int64_t moe_align_capacity(int M, int top_k, int num_experts, int block_m);
int moe_align(const int32_t* topk_ids, int M, int top_k, int expert_base, int num_experts,
              int block_m, int32_t* sorted_ids, int32_t* expert_ids, int32_t* n_padded,
              void* stream);

/* Launch-configuration choice (host only, no device sync): the block_m the
 * forward runs best with for this problem, from the token count, top_k, the
 * number of experts routed ids range over and the layer shape.  Replaces the
 * page's candidate loop ("013-moe-middle-tiles.py", BLOCK_SIZE_M_CANDIDATES). */
int moe_choose_block_m(const moe_layer_desc* desc, int M, int top_k, int num_routed_ids);

/* ------------------------------------------------------------------ forward
 * Workspace bytes moe_w4a16_forward needs for (desc, M, top_k, block_m); 256-byte
 * aligned device memory owned by the caller; its contents need no initialisation. */
int64_t moe_workspace_size(const moe_layer_desc* desc, int M, int top_k, int block_m);

/* The layer ("013-moe-middle-tiles.py" kernel_fn after alignment; PR #31552
 * fused_marlin_moe and the per-expert reference loop of its large-M test):
 *   for every local pair p = (t, j) with expert e:
 *     h = gs13[e] * x[t] . W13[e]^T + b13[e]                  [2N] ([N] non-gated)
 *     a = act(h[:N], h[N:])   (relu(h)^2 non-gated)            [N]
 *     y = gs2[e] * a . W2[e]^T + b2[e]                         [K]
 *   out[t] = bf16(rsf * sum_j topk_weights[t,j] * y_(t,j))      (post_norm_w == NULL)
 *   out[t] = bf16(rsf * sum_j topk_weights[t,j] * inv_j * z_j),  z = y * nw,
 *            nw = bf16(fp32(1 + post_norm_w)), inv = 1/sqrt(mean(z^2) + norm_eps)
 *            (_expert_norm_factors / _expert_norm_sum, weight_first)
 * Non-local pairs contribute nothing.  Arithmetic: fp32 accumulation, scales,
 * bias, activation and combine; the tensor-core operands are fp16 (weights
 * dequantised exactly, x converted to fp16 -- exact inside its range -- and a
 * rounded to fp16); a is kept as fp16 and y as fp32 between the kernels; the
 * combine sums in fp32 and writes out as bf16.
 * Arguments (device unless said): packed from moe_repack_weights for `desc`;
 * x bf16 [M, K]; topk_ids int32 [M, top_k]; topk_weights fp32 [M, top_k];
 * sorted_ids / expert_ids / n_padded from moe_align with the same M, top_k,
 * expert_base, E and block_m -- or all three NULL: the forward then aligns the
 * routing itself, in its first kernel, into the workspace (one launch fewer,
 * the same result bit for bit); act a moe_act (MOE_ACT_RELU2 exactly when
 * desc->non_gated); alpha, limit (host) for
 * SIGMOID_ALPHA (limit = +inf: no clamp); post_norm_w bf16 [K] or NULL;
 * out bf16 [M, K]; workspace of at least moe_workspace_size() bytes.  packed and
 * workspace must be 256-byte aligned; x, out and post_norm_w 16-byte aligned.
 * E <= 1024 (the alignment's limit).
 * Operand range: the tensor-core operands are fp16 and a is kept as fp16, so
 * x and the activations a must stay inside the fp16 range (|v| < 65504; values
 * below 2^-14 keep fewer significant bits).
 * A value that leaves it (or is not a number) is not an argument error: the
 * forward completes and records MOE_ERR_UNSUPPORTED for moe_get_status.
 * Dequantised weights are exact fp16 operands for every scale within these
 * windows, per expert and matrix (w13 or w2): the scales are shifted at repack
 * by a power of two into the window and the expert's fp32 epilogue factor
 * undoes the shift, so only the spread of one expert matrix's scales matters:
 *   INT4:  largest / smallest nonzero |scale| below 2^26 (binary exponents
 *          spanning at most 26 values);
 *   MXFP4: E8M0 bytes spanning at most 37 values (largest - smallest <= 36);
 *   NVFP4: any E4M3 scale.
 * A wider spread keeps the largest scales exact and rounds the smallest blocks;
 * moe_repack_weights marks the packed blob and every forward on it records
 * MOE_ERR_UNSUPPORTED (INT4: only forwards with block_m >= 64, whose kernel
 * dequantises with fp16 scales; the block_m <= 32 kernel applies INT4 scales
 * in fp32).
 * Alignment arguments: sorted_ids, expert_ids and n_padded are validated on the
 * device as they are read -- n_padded outside [0, moe_align_capacity(M, top_k,
 * E, block_m)] or not a multiple of block_m, an expert id outside [0, E), a
 * sorted id outside [0, M*top_k) -- and never lead to an access outside the
 * workspace, packed or out; such blocks and slots are skipped and
 * moe_get_status reports MOE_ERR_INVALID afterwards.
 * M == 0 is a no-op. */
int moe_w4a16_forward(const moe_layer_desc* desc, const void* packed, const void* x, int M,
                      int top_k, const int32_t* topk_ids, const float* topk_weights,
                      int expert_base, const int32_t* sorted_ids, const int32_t* expert_ids,
                      const int32_t* n_padded, int block_m, int act, float alpha, float limit,
                      float routed_scaling_factor, const void* post_norm_w, float norm_eps,
                      void* out, void* workspace, int64_t workspace_bytes, void* stream);

/* Allocation-free forward.  Not part of the method: the pages have no
 * counterpart; it exists for callers that cannot pass device memory of their
 * own, such as code running on a stream that a framework is recording into a
 * CUDA graph (an allocation there breaks the recording) or plugins of an engine
 * that owns every device allocation.
 *   Same computation, arguments and rules as moe_w4a16_forward, without
 * workspace / workspace_bytes.  The workspace is instead a fixed array of
 * MOE_NOALLOC_SCRATCH_BYTES in this library's device image, one per device and
 * process, reserved by the CUDA runtime when the module loads; no call here
 * allocates device memory.  Its partial areas (split-K, and the balanced
 * division of 8- and 16-token blocks) are smaller than those
 * moe_w4a16_forward plans, so this entry point can split K less, or run whole
 * items only; results match moe_w4a16_forward's within the layer's tolerance,
 * not bit for bit.
 *   Size limit: returns MOE_ERR_WORKSPACE (nothing launched) when the shape's
 * workspace would exceed MOE_NOALLOC_SCRATCH_BYTES; moe_w4a16_forward with a
 * caller workspace handles such shapes.
 *   Start state: none needed.  The prologue kernel zeroes the status word and
 * the split-K counters at the start of every call.
 *   Concurrency: calls on one device share the array, so two calls in flight
 * at once (two streams, or two host threads without ordering) race and give
 * undefined results; the caller serialises them.
 *   Setup: the first call on a device looks up the array's address
 * (cudaGetSymbolAddress, which can load the module) and the tensor-map
 * encoder; make one call on each device before any stream capture.  Nothing
 * is claimed about behaviour under capture.
 *   Status: device-side reports (a wait that runs out, a value outside the fp16
 * operand range, inconsistent alignment inputs) are recorded in the array's
 * status word, which this entry point does not report; callers that need them
 * use moe_w4a16_forward and moe_get_status.  Decode-sized shapes may run with
 * fewer K splits (down to none, whole items) than moe_w4a16_forward would choose.
 *   Lifetime: the array's device address is looked up once per device and
 * cached; the library must not be used across a reset of the device
 * (cudaDeviceReset), after which the cached address is stale. */
#define MOE_NOALLOC_SCRATCH_BYTES ((int64_t)64 << 20)
int moe_w4a16_forward_noalloc(const moe_layer_desc* desc, const void* packed, const void* x,
                              int M, int top_k, const int32_t* topk_ids,
                              const float* topk_weights, int expert_base,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* n_padded, int block_m, int act, float alpha,
                              float limit, float routed_scaling_factor, const void* post_norm_w,
                              float norm_eps, void* out, void* stream);

/* Synchronises `stream`, returns the device status recorded in `workspace` by
 * the last forward on it and clears it: MOE_OK; MOE_ERR_TIMEOUT (a device wait
 * ran out); MOE_ERR_INVALID (alignment inputs inconsistent with the call);
 * MOE_ERR_UNSUPPORTED (a value outside the fp16 operand range, see
 * moe_w4a16_forward), in that order of precedence.  Each forward clears the word
 * in its first kernel. */
int moe_get_status(void* workspace, void* stream);

/* Tracing hook.  With events != NULL and n == 4, every later moe_w4a16_forward
 * records, on its stream, events[0] before GEMM1, events[1] between GEMM1 and
 * GEMM2, events[2] between GEMM2 and the combine and events[3] after the
 * combine, so a caller can time each kernel with cudaEventElapsedTime.
 * events are cudaEvent_t handles created and owned by the caller; the table is
 * copied.  NULL / 0 turns tracing off.  Process-wide, not thread-safe.
 * Returns MOE_ERR_INVALID for any other n. */
int moe_set_trace_events(void* const* events, int n);

/* Test hook of the device failure path.  With on != 0, every later forward
 * whose GEMMs run the register-fed kernel (block_m 8, 16 or 32) makes CTA 0 of
 * each GEMM end with a bounded wait on a barrier nothing arrives on: the wait
 * gives up after its limit (2 s), records MOE_ERR_TIMEOUT in the workspace
 * status word and the kernel ends normally, so moe_get_status reports the
 * timeout and the context stays usable.  Outputs are computed as usual.  0
 * turns it off.  Process-wide, not thread-safe; returns MOE_OK. */
int moe_set_test_starve_wait(int on);

/* Short English name of a status code (static storage). */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4A16_H */
