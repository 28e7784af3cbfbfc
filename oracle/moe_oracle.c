/*
 * CPU oracle for the weight-only 4-bit fused Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: it is used by tests/, by the smoke check and by the timed
 * CPU baseline of the benchmark.  It shares no code, header, table or helper
 * with the CUDA library.
 *
 * What it computes (plain definitions, written out, fp64 accumulation):
 *
 *   decode      the 4-bit codes and scale bytes from their bit-level definitions
 *               (uint4b8 of "Marlin MoE kernel occupancy ..." (sglang PR #31552),
 *               test_fused_marlin_moe_large_non_ep_schedule: quant_type uint4b8;
 *               E2M1 / E8M0 / E4M3 from the OCP microscaling and FP8 formats, which
 *               the pages name but do not define);
 *   dequant     W = (q-8)*s (int4, group along the reduction dim), or with the INT4
 *               variants W = (q - z)*s, z an integer or bf16 zero point per group,
 *               groups of 32 / 64 / 128 / a whole row, or given per reduction index
 *               by g_idx (act-order),
 *               W = e2m1*2^(b-127) (MXFP4, one E8M0 byte per 32),
 *               W = e2m1*e4m3*gs[e] (NVFP4, one E4M3 per 16, one fp32 global
 *               scale per expert shared by gate and up: "013-moe-middle-tiles.py",
 *               Weights and _marlin_layer);
 *   deinterleave  GPT-OSS w13 rows [g0,u0,g1,u1,...] -> gate i = row 2i, up i = row
 *               2i+1 ("SM120 MXFP4 MoE ... Marlin" (sglang PR #28231),
 *               deinterleave_moe_mxfp4_w13_for_marlin);
 *   align       sort the local (token, slot) pairs by expert and pad each expert's
 *               run to block_m ("013-moe-middle-tiles.py", kernel_fn:
 *               moe_align_block_size(local_ids, block_size_m, ...));
 *   FFN         per local pair p=(t,j) with expert e:
 *                 h = gs13 * sum_k x[t,k] W13[e,r,k] + b13[e,r]       r < 2N
 *                 a = act(h[n], h[N+n])     gate = first half, up = second
 *                 y = gs2 * sum_n a[n] W2[e,c,n] + b2[e,c]            c < K
 *               act = silu(g)*u (silu_and_mul) or
 *                     g' = min(g, L), u' = clamp(u,-L,L), g'*sigmoid(alpha*g')*(u'+1)
 *               (swiglu_gpt_oss_sigmoid_alpha_contiguous of PR #28231);
 *               non-gated experts (w1 has N rows, is_gated=False): a = relu(h)^2
 *               (activation="relu2" of the PR #31552 large-M test, whose reference
 *               loop computes torch.square(torch.relu(intermediate)));
 *   combine     out[t] = bf16(rsf * sum_j w[t,j] * y[t,j]) over local slots
 *               (the per-expert reference loop of the PR #31552 test), or with the
 *               post-expert norm of "013-moe-middle-tiles.py" (_expert_norm_factors,
 *               _expert_norm_sum, weight_first):
 *                 z = y * nw,  nw = bf16(fp32(1 + w_norm)),
 *                 inv = 1 / sqrt(sum_c z^2 / K + eps),
 *                 out[t] = bf16(rsf * sum_j w[t,j] * inv_j * z_j).
 *
 *   requant     the W4AFP8 activation requantisation of "W4AFP8 requant ..." (sglang
 *               PR #35760, _fp8_per_token_quant_to_per_tensor_quant_kernel and
 *               _requant_row): every valid row m < masked_m[e] of each expert's FP8
 *               payload, quantised with one fp32 scale per (row, 128-group), is
 *               re-quantised to one per-tensor scale S:
 *                 out = e4m3(fp32(fp32(x * s[e, g, m]) * r)),  r = fp32(1 / S),
 *               two fp32 multiplies per element as the page states, e4m3 rounding
 *               to nearest (ties to even) and saturating at +-448, NaN -> 0x7F;
 *               rows at or past masked_m are left untouched.
 *
 * h, a and y are carried exactly (fp64); the only rounding is the bf16 output.
 * The bf16 intermediates of kernel_fn (cache1 / cache2 / cache3) are that
 * implementation's storage, not part of the layer's definition, which is the
 * per-expert matmul chain combined in fp32 of the PR #31552 reference loop.
 * Non-local pairs contribute nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_INT4 = 0, ORC_MXFP4 = 1, ORC_NVFP4 = 2 };
enum { ORC_SILU_MUL = 0, ORC_SIGMOID_ALPHA = 1, ORC_RELU2 = 2 };

/* ------------------------------------------------------------------ formats */

/* bf16 is the high half of an IEEE binary32. */
double orc_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, ties to even),
 * keeping bf16 subnormals (quantum 2^-133) and overflowing to infinity. */
uint16_t orc_bf16_round(double x) {
    if (isnan(x)) return 0x7FC0;
    int neg = signbit(x) != 0;
    double a = fabs(x);
    if (a == 0.0) return neg ? 0x8000 : 0x0000;
    int ex;
    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;           /* a in [2^e, 2^(e+1)) */
    double quantum = (e < -126) ? ldexp(1.0, -133) : ldexp(1.0, e - 7);
    double r = nearbyint(a / quantum) * quantum;  /* default mode: ties to even */
    float f;
    if (r > 3.3895313892515355e38) {              /* largest finite bf16 */
        f = INFINITY;
    } else {
        f = (float)r;                               /* exact: r has <= 8 bits */
    }
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t b = (uint16_t)(u >> 16);
    return neg ? (uint16_t)(b | 0x8000) : b;
}

/* E2M1: sign | 2-bit exponent (bias 1) | 1-bit mantissa; exponent 0 is subnormal. */
double orc_e2m1_value(unsigned code) {
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* E8M0: a bare biased exponent, 2^(b-127); 0xFF is NaN. */
double orc_e8m0_value(unsigned b) {
    b &= 0xFFu;
    if (b == 0xFFu) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* E4M3 (fn variant): sign | 4-bit exponent (bias 7) | 3-bit mantissa,
 * subnormals m/8 * 2^-6, S.1111.111 is NaN, no infinities. */
double orc_e4m3_value(unsigned b) {
    b &= 0xFFu;
    unsigned s = b >> 7, e = (b >> 3) & 15u, m = b & 7u;
    if (e == 15u && m == 7u) return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* uint4b8: a 4-bit unsigned code q standing for q - 8. */
double orc_int4_value(unsigned q) { return (double)((int)(q & 15u) - 8); }

/* Element c of a packed row: byte c/2, low nibble for even c, high for odd. */
static unsigned nibble(const uint8_t* row, long c) {
    uint8_t b = row[c >> 1];
    return (c & 1) ? (unsigned)(b >> 4) : (unsigned)(b & 15u);
}

static double code_value(int fmt, unsigned q) {
    return fmt == ORC_INT4 ? orc_int4_value(q) : orc_e2m1_value(q);
}

/* Scale value of entry idx of a scale array in format fmt. */
static double scale_value(int fmt, const void* scales, long idx) {
    if (fmt == ORC_INT4) return orc_bf16_value(((const uint16_t*)scales)[idx]);
    if (fmt == ORC_MXFP4) return orc_e8m0_value(((const uint8_t*)scales)[idx]);
    return orc_e4m3_value(((const uint8_t*)scales)[idx]);
}


/*
 * Dequantise logical rows [0, rows) of one expert's matrix, cols along the
 * reduction dimension, into out[rows][cols] (without the NVFP4 global scale,
 * which the caller applies to the fp64 sum).  row_map[r] gives the stored row
 * of logical row r (identity when NULL); it is how interleaved gate/up rows are
 * read.
 *
 * INT4 variants (the w*_zeros, is_zp_float, g_idx and group_blocks of
 * fused_marlin_moe / the Marlin template in "Marlin MoE kernel occupancy ..."
 * (sglang PR #31552)): element c of a row belongs to group gidx[c] when gidx
 * is given (act-order), else to c / group; group <= 0 means one group per row
 * (channelwise).  With zero_kind 0 the code is uint4b8, W = (q - 8) * s; with
 * zero_kind 1 the group's zero point is an integer byte z, W = (q - z) * s;
 * with zero_kind 2 a bf16 value z, W = (q - z) * s.  zeros hold one entry per
 * (row, group), like the scales.  Every product is exact in binary32 except
 * float zeros, whose (q - z) * s is rounded once to binary32.
 */
void orc_dequant_ex(int fmt, const uint8_t* codes, const void* scales, const void* zeros, int zero_kind,
                    const int32_t* gidx, int rows, int cols, int group, const int32_t* row_map, float* out) {
    long bpr = cols / 2;
    if (group <= 0) group = cols;
    long spr = cols / group;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        long sr = row_map ? row_map[r] : r;
        const uint8_t* crow = codes + sr * bpr;
        for (long c = 0; c < cols; ++c) {
            long g = gidx ? (long)gidx[c] : c / group;
            double sv = scale_value(fmt, scales, sr * spr + g);
            unsigned q = nibble(crow, c);
            double v;
            if (fmt != ORC_INT4 || zero_kind == 0) {
                v = code_value(fmt, q) * sv;
            } else if (zero_kind == 1) {
                v = ((double)q - (double)((const uint8_t*)zeros)[sr * spr + g]) * sv;
            } else {
                v = ((double)q - orc_bf16_value(((const uint16_t*)zeros)[sr * spr + g])) * sv;
            }
            out[(long)r * cols + c] = (float)v;
        }
    }
}

void orc_dequant(int fmt, const uint8_t* codes, const void* scales, int rows, int cols, int group,
                 const int32_t* row_map, float* out) {
    orc_dequant_ex(fmt, codes, scales, NULL, 0, NULL, rows, cols, group, row_map, out);
}

/* ------------------------------------------------------------------ align */

/* Worst-case number of sorted slots: every non-empty expert wastes at most
 * block_m - 1 slots, and at most min(E, M*k) experts are non-empty. */
long orc_align_capacity(int M, int top_k, int num_experts, int block_m) {
    long pairs = (long)M * top_k;
    long busy = pairs < num_experts ? pairs : num_experts;
    long n = pairs + busy * (block_m - 1);
    return (n + block_m - 1) / block_m * block_m;
}

/*
 * Align the local pairs to block_m.  A pair is the flat index p = t*k + j; its
 * routed id topk_ids[p] is local when base <= id < base + E.
 *   - experts appear in ascending local id, empty experts get no block;
 *   - within an expert the pairs are in ascending p;
 *   - each expert's run is padded to a multiple of block_m with the sentinel M*k;
 *   - n_padded = sum_e ceil(count_e / block_m) * block_m;
 *   - sorted_ids[n_padded, cap) = sentinel, expert_ids[b] = expert of block b,
 *     -1 for blocks at or past n_padded / block_m.
 * Returns 0, or -1 on bad arguments.
 */
int orc_align(const int32_t* topk_ids, int M, int top_k, int base, int num_experts, int block_m,
              int32_t* sorted_ids, long cap, int32_t* expert_ids, int32_t* n_padded) {
    if (M < 0 || top_k <= 0 || num_experts <= 0 || block_m <= 0) return -1;
    long pairs = (long)M * top_k;
    int32_t sentinel = (int32_t)pairs;
    long* count = (long*)calloc((size_t)num_experts, sizeof(long));
    long* start = (long*)calloc((size_t)num_experts, sizeof(long));
    if (!count || !start) { free(count); free(start); return -1; }
    for (long p = 0; p < pairs; ++p) {
        long e = (long)topk_ids[p] - base;
        if (e >= 0 && e < num_experts) count[e]++;
    }
    long total = 0;
    for (int e = 0; e < num_experts; ++e) {
        start[e] = total;
        total += (count[e] + block_m - 1) / block_m * block_m;
    }
    if (total > cap) { free(count); free(start); return -1; }
    for (long i = 0; i < cap; ++i) sorted_ids[i] = sentinel;
    for (long b = 0; b < cap / block_m; ++b) expert_ids[b] = -1;
    long* fill = (long*)calloc((size_t)num_experts, sizeof(long));
    for (long p = 0; p < pairs; ++p) {
        long e = (long)topk_ids[p] - base;
        if (e >= 0 && e < num_experts) sorted_ids[start[e] + fill[e]++] = (int32_t)p;
    }
    for (int e = 0; e < num_experts; ++e)
        for (long b = start[e] / block_m; b < (start[e] + (count[e] + block_m - 1) / block_m * block_m) / block_m; ++b)
            expert_ids[b] = e;
    *n_padded = (int32_t)total;
    free(count); free(start); free(fill);
    return 0;
}

/* ------------------------------------------------------------------ forward */

typedef struct {
    int fmt, num_experts, hidden, inter, group, interleaved;
    const uint8_t* w13;   /* [E, R, K/2], R = 2N gated (gate rows then up rows), N non-gated */
    const void* w13_s;    /* [E, R, K/g] */
    const float* w13_gs;  /* [E] or NULL */
    const uint16_t* b13;  /* [E, R] bf16 or NULL */
    const uint8_t* w2;    /* [E, K, N/2] */
    const void* w2_s;     /* [E, K, N/g] */
    const float* w2_gs;   /* [E] or NULL */
    const uint16_t* b2;   /* [E, K] bf16 or NULL */
    int gated;            /* 1: gate and up rows, act on (gate, up); 0: N rows, relu^2 */
    int zero_kind;        /* INT4 zero points: 0 none (uint4b8), 1 integer bytes, 2 bf16 values */
    const void* w13_z;    /* [E, R, K/g] zero points, or NULL */
    const void* w2_z;     /* [E, K, N/g] */
    const int32_t* w13_gidx;  /* [E, K] group of each reduction index (act-order), or NULL */
    const int32_t* w2_gidx;   /* [E, N] */
} orc_layer;

/* Groups per row of a matrix with `cols` reduction elements (group <= 0: one). */
static long n_groups(int group, int cols) { return group <= 0 ? 1 : cols / group; }

/* Dequantised w13 (logical rows, gate block then up block) and w2 of expert e. */
static void dequant_expert(const orc_layer* L, int e, const int32_t* rmap, float* W13, float* W2) {
    const int K = L->hidden, N = L->inter, R = L->gated ? 2 * N : N;
    const long sb = L->fmt == ORC_INT4 ? 2 : 1;                 /* scale bytes */
    const long zb = L->zero_kind == 2 ? 2 : 1;                  /* zero bytes */
    const long g13 = n_groups(L->group, K), g2 = n_groups(L->group, N);
    orc_dequant_ex(L->fmt, L->w13 + (long)e * R * (K / 2), (const uint8_t*)L->w13_s + (long)e * R * g13 * sb,
                   L->w13_z ? (const uint8_t*)L->w13_z + (long)e * R * g13 * zb : NULL, L->zero_kind,
                   L->w13_gidx ? L->w13_gidx + (long)e * K : NULL, R, K, L->group, rmap, W13);
    orc_dequant_ex(L->fmt, L->w2 + (long)e * K * (N / 2), (const uint8_t*)L->w2_s + (long)e * K * g2 * sb,
                   L->w2_z ? (const uint8_t*)L->w2_z + (long)e * K * g2 * zb : NULL, L->zero_kind,
                   L->w2_gidx ? L->w2_gidx + (long)e * N : NULL, K, N, L->group, NULL, W2);
}

typedef struct {
    int M, top_k, expert_base, act;
    double alpha, limit, rsf, norm_eps;
    const uint16_t* x;            /* [M, K] bf16 */
    const int32_t* topk_ids;      /* [M, k] */
    const float* topk_weights;    /* [M, k] */
    const uint16_t* post_norm_w;  /* [K] bf16 raw w (applied as 1 + w) or NULL */
} orc_batch;

static double round_bf16(double v) { return orc_bf16_value(orc_bf16_round(v)); }

static double activation(int act, double g, double u, double alpha, double limit) {
    if (act == ORC_RELU2) return g > 0.0 ? g * g : 0.0;  /* non-gated: u unused */
    if (act == ORC_SILU_MUL) return g / (1.0 + exp(-g)) * u;
    double gc = g < limit ? g : limit;
    double uc = u > limit ? limit : (u < -limit ? -limit : u);
    return gc * (1.0 / (1.0 + exp(-alpha * gc))) * (uc + 1.0);
}

/* y[K] of one pair whose expert weights are already dequantised. */
static void ffn_pair(const orc_layer* L, const orc_batch* X, int e, int t, const float* W13,
                     const float* W2, double* h, double* a, double* y) {
    const int K = L->hidden, N = L->inter, R = L->gated ? 2 * N : N;
    const uint16_t* xr = X->x + (long)t * K;
    double gs13 = L->w13_gs ? (double)L->w13_gs[e] : 1.0;
    double gs2 = L->w2_gs ? (double)L->w2_gs[e] : 1.0;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        const float* wr = W13 + (long)r * K;
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += orc_bf16_value(xr[c]) * (double)wr[c];
        long br = (L->gated && L->interleaved) ? (long)2 * (r % N) + (r / N) : r;
        double b = L->b13 ? orc_bf16_value(L->b13[(long)e * R + br]) : 0.0;
        h[r] = gs13 * acc + b;
    }
    for (int n = 0; n < N; ++n)
        a[n] = L->gated ? activation(X->act, h[n], h[N + n], X->alpha, X->limit)
                        : activation(ORC_RELU2, h[n], 0.0, X->alpha, X->limit);
#pragma omp parallel for schedule(static)
    for (int c = 0; c < K; ++c) {
        const float* wr = W2 + (long)c * N;
        double acc = 0.0;
        for (int n = 0; n < N; ++n) acc += a[n] * (double)wr[n];
        double b = L->b2 ? orc_bf16_value(L->b2[(long)e * K + c]) : 0.0;
        y[c] = gs2 * acc + b;
    }
}

/*
 * Output rows of the tokens listed in tokens[0, n_tokens) (each 0 <= t < M):
 * out_bf16[i][K] gets token tokens[i]; out_acc (optional, [n_tokens][K]) gets the
 * same value before its final bf16 rounding.  Only experts touched by those
 * tokens are dequantised, one at a time.  Returns 0, or -1 on bad arguments or
 * allocation failure.
 */
int orc_forward(const orc_layer* L, const orc_batch* X, const int32_t* tokens, int n_tokens,
                uint16_t* out_bf16, double* out_acc) {
    const int K = L->hidden, N = L->inter, E = L->num_experts, k = X->top_k;
    const int R = L->gated ? 2 * N : N;  /* rows of w13 */
    if (K <= 0 || N <= 0 || E <= 0 || k <= 0 || L->group == 0) return -1;
    if (!L->gated && X->act != ORC_RELU2) return -1;
    if (L->gated && X->act == ORC_RELU2) return -1;
    if ((L->group > 0 && (K % L->group || N % L->group)) || K % 2 || N % 2) return -1;
    if (L->fmt != ORC_INT4 && (L->zero_kind || L->w13_gidx || L->w2_gidx || L->group < 0)) return -1;
    if (L->zero_kind && (!L->w13_z || !L->w2_z)) return -1;
    double* acc_out = (double*)calloc((size_t)n_tokens * K, sizeof(double));
    double* nsq = (double*)calloc((size_t)n_tokens * k, sizeof(double));
    float* W13 = (float*)malloc(sizeof(float) * (size_t)R * K);
    float* W2 = (float*)malloc(sizeof(float) * (size_t)K * N);
    int32_t* rmap = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
    double* h = (double*)malloc(sizeof(double) * (size_t)R);
    double* a = (double*)malloc(sizeof(double) * (size_t)N);
    double* y = (double*)malloc(sizeof(double) * (size_t)K);
    double* nw = (double*)malloc(sizeof(double) * (size_t)K);
    if (!acc_out || !nsq || !W13 || !W2 || !rmap || !h || !a || !y || !nw) {
        free(acc_out); free(nsq); free(W13); free(W2); free(rmap); free(h); free(a); free(y); free(nw);
        return -1;
    }
    for (int r = 0; r < R; ++r)  /* logical row r -> stored row */
        rmap[r] = (L->gated && L->interleaved) ? 2 * (r % N) + (r / N) : r;
    if (X->post_norm_w)
        for (int c = 0; c < K; ++c) {
            float s = (float)(1.0 + orc_bf16_value(X->post_norm_w[c]));  /* fp32 add, as torch */
            nw[c] = round_bf16((double)s);
        }
    for (int e = 0; e < E; ++e) {
        int touched = 0;
        for (int i = 0; i < n_tokens && !touched; ++i)
            for (int j = 0; j < k; ++j)
                if (X->topk_ids[(long)tokens[i] * k + j] - X->expert_base == e) { touched = 1; break; }
        if (!touched) continue;
        dequant_expert(L, e, rmap, W13, W2);
        for (int i = 0; i < n_tokens; ++i) {
            int t = tokens[i];
            for (int j = 0; j < k; ++j) {
                if (X->topk_ids[(long)t * k + j] - X->expert_base != e) continue;
                ffn_pair(L, X, e, t, W13, W2, h, a, y);
                double w = (double)X->topk_weights[(long)t * k + j];
                double* acc = acc_out + (long)i * K;
                if (X->post_norm_w) {
                    double ss = 0.0;
                    for (int c = 0; c < K; ++c) { double z = y[c] * nw[c]; ss += z * z; }
                    double inv = 1.0 / sqrt(ss / K + X->norm_eps);
                    for (int c = 0; c < K; ++c) acc[c] += w * inv * (y[c] * nw[c]);
                } else {
                    for (int c = 0; c < K; ++c) acc[c] += w * y[c];
                }
            }
        }
    }
    for (long i = 0; i < (long)n_tokens * K; ++i) {
        double v = X->rsf * acc_out[i];
        if (out_acc) out_acc[i] = v;
        if (out_bf16) out_bf16[i] = orc_bf16_round(v);
    }
    free(acc_out); free(nsq); free(W13); free(W2); free(rmap); free(h); free(a); free(y); free(nw);
    return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Intermediates of one pair (token t on local expert e): h[2N], a[N], y[K]
 * as the forward computes them.  Returns 0 or -1. */
int orc_ffn_pair(const orc_layer* L, const orc_batch* X, int e, int t, double* h, double* a, double* y) {
    const int K = L->hidden, N = L->inter, R = L->gated ? 2 * N : N;
    if (e < 0 || e >= L->num_experts || t < 0 || t >= X->M) return -1;
    float* W13 = (float*)malloc(sizeof(float) * (size_t)R * K);
    float* W2 = (float*)malloc(sizeof(float) * (size_t)K * N);
    int32_t* rmap = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
    if (!W13 || !W2 || !rmap) { free(W13); free(W2); free(rmap); return -1; }
    for (int r = 0; r < R; ++r) rmap[r] = (L->gated && L->interleaved) ? 2 * (r % N) + (r / N) : r;
    dequant_expert(L, e, rmap, W13, W2);
    ffn_pair(L, X, e, t, W13, W2, h, a, y);
    free(W13); free(W2); free(rmap);
    return 0;
}

/* ------------------------------------------------------------------ requant */

/* fp32 -> FP8 E4M3 (fn): the nearest of the 126 positive finite values (and 0),
 * ties to the even code (the even mantissa), magnitudes of 448 and above
 * saturating to 448, the sign kept (negative values that round to zero give
 * 0x80), NaN giving 0x7F.  A brute-force search over the format's own values. */
uint8_t orc_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int best = 0;
    double bd = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_value((unsigned)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) { best = c; bd = d; }
    }
    return (uint8_t)(sign | best);
}

/*
 * Per-token -> per-tensor requantisation of an expert-major FP8 payload.
 *   x        uint8 E4M3 [E, max_m, K]
 *   scale    fp32, entry (e, g, m) at e*se + g*sg + m*sm (g = k / group)
 *   masked_m int32 [E]: valid rows of each expert (clamped to [0, max_m])
 *   tensor_scale: S; out = e4m3((x * s) * (1 / S)) in fp32 steps
 *   out      uint8 [E, max_m, K]; rows at or past masked_m are not written.
 * Returns 0, or -1 on bad arguments.
 */
int orc_requant(const uint8_t* x, const float* scale, long se, long sg, long sm, const int32_t* masked_m,
                int E, int max_m, int K, int group, float tensor_scale, uint8_t* out) {
    if (E < 0 || max_m < 0 || K <= 0 || group <= 0 || K % group) return -1;
    const float r = 1.0f / tensor_scale;
    for (int e = 0; e < E; ++e) {
        int rows = masked_m[e] < 0 ? 0 : (masked_m[e] > max_m ? max_m : masked_m[e]);
        for (int m = 0; m < rows; ++m) {
            const uint8_t* xr = x + ((long)e * max_m + m) * K;
            uint8_t* orow = out + ((long)e * max_m + m) * K;
            for (int k = 0; k < K; ++k) {
                float s = scale[e * se + (long)(k / group) * sg + m * sm];
                float t = (float)orc_e4m3_value(xr[k]);
                t = t * s;
                t = t * r;
                orow[k] = orc_e4m3_encode(t);
            }
        }
    }
    return 0;
}
