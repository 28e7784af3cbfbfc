/*
 * moe_requant.h -- C ABI of the FP8 activation requantisation kernel of the
 * W4AFP8 expert path (GB300, sm_103a), a companion of moe_w4a16.h: the
 * per-token -> per-tensor requantisation that "W4AFP8 requant ..." (sglang PR
 * #35760: _fp8_per_token_quant_to_per_tensor_quant_kernel, _requant_row,
 * requant_launch_geometry) runs on the low-latency dispatcher's output before
 * the W4A8 grouped GEMM.
 *
 * Conventions as in moe_w4a16.h: device pointers owned by the caller, no
 * allocation, no synchronisation, `stream` a cudaStream_t passed as void*,
 * return values from moe_status.
 */
#ifndef MOE_REQUANT_H
#define MOE_REQUANT_H

#include <stdint.h>

#include "moe_w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Requantise every valid row of an expert-major FP8 payload from its
 * per-token, per-group scales to one per-tensor scale.
 *   x            uint8 FP8 E4M3 [E, max_m, K] (16-byte aligned); expert e's
 *                rows m < min(masked_m[e], max_m) are valid
 *   scale        fp32; the scale of row m of expert e, column group g (columns
 *                [g*group, (g+1)*group)) at scale[e*scale_stride_e +
 *                g*scale_stride_g + m*scale_stride_m]: the dispatcher's
 *                column-major layout [E, K/group, max_m] is (K/group*max_m,
 *                max_m, 1), a row-major [E, max_m, K/group] (max_m*K/group,
 *                1, K/group)
 *   masked_m     int32 [E] valid rows per expert (values outside [0, max_m]
 *                are clamped)
 *   group        a power of two >= 16 dividing K (128 on the page)
 *   tensor_scale fp32 [1]: S, the per-tensor scale of the output
 *   out          uint8 FP8 E4M3 [E, max_m, K] (16-byte aligned; may be x)
 *   expected_rows  a launch hint, the caller's estimate of valid rows per
 *                expert (<= 0: unknown); any value gives the same bytes
 * Each valid element becomes e4m3(fp32(fp32(x * s) * r)), r = fp32(1 / S):
 * two fp32 multiplies, each rounded to nearest, then E4M3 rounding to nearest
 * (ties to even) that saturates at +-448 (NaN stays NaN).  Rows at or past
 * masked_m are not written.  E <= 1024.  Returns MOE_ERR_INVALID for bad
 * arguments (nothing launched), MOE_ERR_CUDA if the launch fails. */
int moe_requant_fp8(const void* x, const float* scale, int64_t scale_stride_e, int64_t scale_stride_g,
                    int64_t scale_stride_m, const int32_t* masked_m, int num_experts, int max_m, int K, int group,
                    const float* tensor_scale, void* out, int expected_rows, void* stream);

/* The launch geometry moe_requant_fp8 uses (host only): CTAs and threads per
 * CTA for num_experts experts of K columns, the row estimate expected_rows
 * (<= 0: unknown) and sm_count SMs.  One warp streams one row at a time,
 * 16 bytes per lane whatever K is; the grid covers E * floor_pow2(expected_rows)
 * rows with one warp each, at least 1 and at most 8 CTAs per SM (the whole
 * machine when the estimate is unknown).  Returns MOE_OK or MOE_ERR_INVALID. */
int moe_requant_launch_geometry(int num_experts, int K, int expected_rows, int sm_count, int* ctas, int* threads);

#ifdef __cplusplus
}
#endif
#endif /* MOE_REQUANT_H */
