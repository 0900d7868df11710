/*
 * oracle.c -- plain CPU reference for the MoE combine/finalize step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests/, the smoke check and the bench's
 * CPU-baseline leg can compare the CUDA path against an obviously correct,
 * slow implementation.  It shares no code, header, table or constant with
 * norm_quant_gb300/csrc.
 *
 * Arithmetic: fp64 everywhere the method accumulates, in a fixed order
 * (ascending top-k slot j, then the shared-expert row, then the residual).
 * Where a floating-point value decides an integer code (the UE8M0 / e4m3
 * block scales and the e4m3 / e2m1 element codes) the value is first taken
 * to fp32, the precision the CUDA kernels decide in, and every further step
 * is an exact function of that fp32 value or an fp32-rounded quotient /
 * product (computed in double, then rounded once to float: for +,-,*,/ of
 * float operands that double rounding is innocuous, since 53 >= 2*24+2).
 *
 * Sources (page title, section):
 *  - Struct_ep_combine_skip_a2a, "execute": the weighted sum of routed
 *    expert outputs per token; args router_weights [num_tokens, top_k],
 *    topk_ids [num_tokens, top_k], src_info (origin of each received row),
 *    recv_count_ptrs (tokens received per expert); parameter
 *    fused_shared_expert (the shared expert's output is added).
 *  - flashinfer.megamoe.nvfp4_mega_moe, parameter num_tokens: short ranks
 *    are padded with rows routed to -1; parameter
 *    cumulative_local_expert_recv_stats: int32 receive count per expert.
 *  - flashinfer.comm.trtllm_moe_allreduce_fusion, parameters residual_in,
 *    residual_out, rms_gamma, rms_eps, norm_out, weight_bias (gamma + bias,
 *    None means 0; 1.0 is the Gemma form), scale_factor, quant_out,
 *    scale_out, layout_code.
 *  - flashinfer.comm.moe_a2a_combine, parameters output_dtype (bf16 or
 *    float8_e4m3fn), output_scales (UE8M0 in uint8, vector size 32),
 *    output_scalar_scale (per-tensor global scale applied before FP4 block
 *    scaling), sf_layout (linear default, or swizzled).
 *
 * Readings where the pages are silent (the plainest one the rest supports):
 *  R1 rows of one expert are stored in ascending (token, slot) order;
 *  R2 ids outside [-1, E) are treated as padding and reported;
 *  R4 router weights are used as given (no renormalisation); a padded slot
 *     contributes nothing whatever its weight;
 *  R5 the shared row has weight 1; x = (routed + shared) + residual; the
 *     norm and the quantiser see the unrounded x, not bf16(residual_out);
 *  R6 y = x / sqrt(mean(x^2) + eps) * (gamma + weight_bias);
 *  R7 MXFP8 block exponent: the smallest e with amax <= 448 * 2^e, stored as
 *     clamp(e + 127, 0, 254); amax == 0 stores 0;
 *  R9 NVFP4 block scale s = e4m3(amax(g*y) / 6); each element is divided
 *     by the block scale, q = e2m1(fp32(fp32(g*y) / s)), q = 0 when s == 0;
 *     element 2i in the low nibble;
 *  R10 the 128x4 swizzled scale layout of the cuBLAS block-scaling format;
 *  R16 MXFP4 block exponent: the smallest e with amax <= 6 * 2^e, like R7;
 *     fp16 I/O and bf16 / fp16 router weights decode exactly to fp64;
 *  R15 the slot-major layout (trtllm_moe_allreduce_fusion,
 *     moe_reduction_active_experts_token_input / moe_reduction_scale_input /
 *     moe_reduction_token_input): expert rows as [k, T, H], one per slot, the
 *     per-(token, slot) scale in the router-weight layout [T, k], and the
 *     token input added like the shared-expert row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_INVALID_EXPERT 4

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bf16: the upper half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Exact value -> bf16, round to nearest, ties to even.  bf16 keeps 8
 * significant bits; normal exponents run down to 2^-126, below which the
 * quantum is fixed at 2^-133 (subnormals).  Values that round past the
 * largest finite bf16 become infinity, as IEEE rounding does. */
uint16_t oracle_f64_to_bf16(double d)
{
    if (isnan(d))
        return 0x7FC0;
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int p;
    frexp(a, &p);            /* a in [2^(p-1), 2^p) */
    int q = p - 8;           /* quantum giving 8 significant bits */
    if (q < -133)
        q = -133;
    double m = nearbyint(ldexp(a, -q)); /* ties to even (default mode) */
    double r = ldexp(m, q);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)r;      /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* IEEE binary16: s.eeeee.mmmmmmmmmm, bias 15, subnormals m * 2^-24. */
double oracle_f16_to_f64(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

/* Exact value -> binary16, round to nearest, ties to even: 11 significant
 * bits, normal exponents down to 2^-14, fixed quantum 2^-24 below that;
 * values that round past 65504 become infinity. */
uint16_t oracle_f64_to_f16(double d)
{
    if (isnan(d))
        return 0x7E00;
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (a == 0.0)
        return sign;
    int p;
    frexp(a, &p);           /* a in [2^(p-1), 2^p) */
    int q = p - 11;         /* quantum giving 11 significant bits */
    if (q < -24)
        q = -24;
    double m = nearbyint(ldexp(a, -q));
    double r = ldexp(m, q);
    if (r > 65504.0)
        return sign | 0x7C00;
    /* encode the exact binary16 value r */
    if (r < ldexp(1.0, -14))
        return sign | (uint16_t)(r * ldexp(1.0, 24));
    int pe;
    double f = frexp(r, &pe); /* r = f * 2^pe, f in [0.5, 1) */
    int e = pe - 1 + 15;
    uint16_t man = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(e << 10) | man;
}

/* float8 e4m3 ("fn": finite, no infinity): s.eeee.mmm, bias 7; exponent
 * field 0 holds subnormals m * 2^-9; s.1111.111 is NaN; largest finite 448. */
double oracle_e4m3_to_f64(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* Round to nearest e4m3, ties to the even code, saturating to +-448.  The
 * non-negative finite codes 0x00..0x7E are in increasing order of value and
 * a code's lowest bit is its mantissa's lowest bit, so "even code" is
 * "even mantissa". */
uint8_t oracle_e4m3_from_f64(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_to_f64((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - oracle_e4m3_to_f64((uint8_t)lo);
    double dhi = oracle_e4m3_to_f64((uint8_t)hi) - a;
    int code = (dlo < dhi) ? lo : (dhi < dlo) ? hi : ((lo & 1) ? hi : lo);
    return sign | (uint8_t)code;
}

/* fp4 e2m1: s.ee.m, bias 1; exponent field 0 holds the subnormal m * 0.5.
 * Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_to_f64(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Round to nearest e2m1, ties to the even code, saturating to +-6. */
uint8_t oracle_e2m1_from_f64(double x)
{
    uint8_t sign = signbit(x) ? 0x8 : 0;
    double a = fabs(x);
    if (a >= 6.0)
        return sign | 0x7;
    int lo = 0;
    while (lo < 7 && oracle_e2m1_to_f64((uint8_t)(lo + 1)) <= a)
        lo++;
    int hi = lo + 1;
    double dlo = a - oracle_e2m1_to_f64((uint8_t)lo);
    double dhi = oracle_e2m1_to_f64((uint8_t)hi) - a;
    int code = (dlo < dhi) ? lo : (dhi < dlo) ? hi : ((lo & 1) ? hi : lo);
    return sign | (uint8_t)code;
}

/* UE8M0 block scale for MXFP8 (reading R7): the smallest integer e with
 * amax <= 448 * 2^e, so that no element of the block saturates, biased by
 * 127 and clamped to the finite byte range [0, 254].  amax == 0 -> 0. */
uint8_t oracle_ue8m0_for_amax(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int p;
    frexp(amax, &p);
    int e = p - 9; /* a first guess, then adjust to the definition */
    while (ldexp(448.0, e) < amax)
        e++;
    while (ldexp(448.0, e - 1) >= amax)
        e--;
    int b = e + 127;
    if (b < 0)
        b = 0;
    if (b > 254)
        b = 254;
    return (uint8_t)b;
}

/* UE8M0 block scale for MXFP4 (reading R16): the smallest integer e with
 * amax <= 6 * 2^e (6 is the largest e2m1 magnitude), biased by 127 and
 * clamped to [0, 254].  amax == 0 -> 0. */
uint8_t oracle_ue8m0_fp4_for_amax(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int p;
    frexp(amax, &p);
    int e = p - 3;
    while (ldexp(6.0, e) < amax)
        e++;
    while (ldexp(6.0, e - 1) >= amax)
        e--;
    int b = e + 127;
    if (b < 0)
        b = 0;
    if (b > 254)
        b = 254;
    return (uint8_t)b;
}

/* Byte offset of scale (row r, column c) in a scale matrix of C columns.
 * layout 0: linear, row-major.  layout 1: 128x4 swizzle (reading R10):
 * 128-row x 4-column tiles of 512 bytes, tiles ordered row-tile major with
 * column tiles fastest; inside a tile, row r sits at (r % 32) * 16 +
 * ((r % 128) / 32) * 4 and column c at c % 4. */
int64_t oracle_sf_offset(int64_t r, int64_t c, int64_t C, int32_t layout)
{
    if (layout == 0)
        return r * C + c;
    int64_t Cp = (C + 3) / 4 * 4;
    return (r / 128) * (Cp / 4) * 512 + (c / 4) * 512 + (r % 32) * 16 +
           ((r % 128) / 32) * 4 + (c % 4);
}

/* out[r * C + c] = oracle_sf_offset(r, c, C, layout) for r < T, c < C. */
void oracle_sf_offsets(int64_t T, int64_t C, int32_t layout, int64_t *out)
{
    for (int64_t r = 0; r < T; r++)
        for (int64_t c = 0; c < C; c++)
            out[r * C + c] = oracle_sf_offset(r, c, C, layout);
}

/* Size in bytes of the scale matrix for T rows and H elements per row. */
int64_t oracle_scales_bytes(int64_t T, int32_t H, int32_t quant, int32_t layout)
{
    int64_t vec = (quant == 2) ? 16 : 32;  /* NVFP4 16; MXFP8 and MXFP4 32 */
    int64_t C = H / vec;
    if (layout == 0)
        return T * C;
    int64_t Tp = (T + 127) / 128 * 128, Cp = (C + 3) / 4 * 4;
    return Tp * Cp;
}

/* ------------------------------------------------------------------------ */
/* Routing: counts, offsets, row_map, src_row                                */
/* ------------------------------------------------------------------------ */

/* topk_ids is [T, k] row-major; -1 marks a padded slot (nvfp4_mega_moe,
 * num_tokens).  counts[e] is the number of slots routed to expert e (the
 * per-expert receive count of nvfp4_mega_moe /
 * Struct_ep_combine_skip_a2a recv_count_ptrs), offsets the exclusive prefix
 * sum over experts (E + 1 entries), and row_map[t, j] the row of the
 * expert-grouped buffer holding token t's output from slot j, -1 for padding.
 * Inside one expert the rows follow ascending (t, j) (reading R1).
 * src_row[row] = t * k + j is the single-GPU form of src_info.
 * Ids outside [-1, E) are treated as padding and make the call return
 * ORACLE_ERR_INVALID_EXPERT (reading R2).  src_row may be NULL. */
int oracle_build_row_map(const int32_t *topk_ids, int64_t T, int32_t k, int32_t E,
                         int32_t *counts, int32_t *offsets, int32_t *row_map,
                         int32_t *src_row)
{
    if (T < 0 || k < 1 || E < 1)
        return ORACLE_ERR_INVALID_ARG;
    int status = ORACLE_OK;
    int64_t N = T * (int64_t)k;
    for (int32_t e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t i = 0; i < N; i++) {
        int32_t e = topk_ids[i];
        if (e >= 0 && e < E)
            counts[e]++;
        else if (e != -1)
            status = ORACLE_ERR_INVALID_EXPERT;
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!seen)
        return ORACLE_ERR_INVALID_ARG;
    for (int64_t i = 0; i < N; i++) {
        int32_t e = topk_ids[i];
        if (e >= 0 && e < E) {
            int32_t row = offsets[e] + seen[e]++;
            row_map[i] = row;
            if (src_row)
                src_row[row] = (int32_t)i;
        } else {
            row_map[i] = -1;
        }
    }
    free(seen);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Combine, residual, RMSNorm, quantisation                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t T;
    int32_t H, k;
    const uint16_t *expert_out; /* bf16 [n_rows, H], grouped by expert */
    int64_t n_rows;
    const int32_t *row_map;     /* [T, k], -1 = padded slot */
    const float *weights;       /* fp32 [T, k] router weights */
    const uint16_t *shared;     /* bf16 [T, H] or NULL */
    const uint16_t *residual;   /* bf16 [T, H] or NULL */
    const uint16_t *gamma;      /* bf16 [H] or NULL: no RMSNorm */
    float eps, weight_bias;
    int32_t quant;              /* 0 none, 1 MXFP8 e4m3/UE8M0/32, 2 NVFP4 e2m1/e4m3/16 */
    int32_t sf_layout;          /* 0 linear, 1 128x4 swizzled */
    float global_scale;         /* NVFP4 per-tensor scale g */
    uint16_t *combined_out;     /* bf16 [T, H] or NULL */
    uint16_t *residual_out;     /* bf16 [T, H] or NULL */
    uint16_t *norm_out;         /* bf16 [T, H] or NULL */
    uint8_t *quant_out;         /* [T, H] (MXFP8) or [T, H/2] (NVFP4) or NULL */
    uint8_t *scales_out;        /* oracle_scales_bytes(...) bytes or NULL */
    double *y_out;              /* fp64 [T, H] quantiser input, or NULL */
    int32_t expert_layout;      /* 0: rows grouped by expert, found through row_map;
                                   1: slot-major [k, T, H], row of (t, j) at j * T + t,
                                      row_map unused (reading R15) */
    int32_t io_dtype;           /* 16-bit tensors in and out: 0 bf16, 1 fp16 */
    int32_t weight_dtype;       /* router weights: 0 fp32, 1 bf16, 2 fp16 */
    int32_t pad0;
} oracle_combine_args;

int oracle_combine_args_size(void) { return (int)sizeof(oracle_combine_args); }

/* MXFP8 (moe_a2a_combine output_dtype float8_e4m3fn with UE8M0
 * output_scales, vector size 32) of one row already rounded to fp32. */
static void quant_mxfp8_row(const float *y32, int32_t H, int64_t t, int32_t layout,
                            uint8_t *q, uint8_t *scales)
{
    int64_t C = H / 32;
    for (int64_t c = 0; c < C; c++) {
        double amax = 0.0;
        for (int i = 0; i < 32; i++) {
            double v = fabs((double)y32[c * 32 + i]);
            if (v > amax)
                amax = v;
        }
        uint8_t b = oracle_ue8m0_for_amax(amax);
        scales[oracle_sf_offset(t, c, C, layout)] = b;
        for (int i = 0; i < 32; i++)
            q[c * 32 + i] = oracle_e4m3_from_f64(ldexp((double)y32[c * 32 + i], 127 - b));
    }
}

/* MXFP4 (moe_a2a_combine: the MXFP4 path, which ignores
 * output_scalar_scale) of one row already rounded to fp32: UE8M0 scale per
 * 32 elements (reading R16), e2m1 codes of y * 2^-e, element 2i in the low
 * nibble. */
static void quant_mxfp4_row(const float *y32, int32_t H, int64_t t, int32_t layout, uint8_t *q,
                            uint8_t *scales)
{
    int64_t C = H / 32;
    for (int64_t c = 0; c < C; c++) {
        double amax = 0.0;
        for (int i = 0; i < 32; i++) {
            double v = fabs((double)y32[c * 32 + i]);
            if (v > amax)
                amax = v;
        }
        uint8_t b = oracle_ue8m0_fp4_for_amax(amax);
        scales[oracle_sf_offset(t, c, C, layout)] = b;
        for (int i = 0; i < 32; i += 2) {
            uint8_t lo = oracle_e2m1_from_f64(ldexp((double)y32[c * 32 + i], 127 - b));
            uint8_t hi = oracle_e2m1_from_f64(ldexp((double)y32[c * 32 + i + 1], 127 - b));
            q[c * 16 + i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* NVFP4 (trtllm_moe_allreduce_fusion quant_out / scale_out with
 * scale_factor; moe_a2a_combine output_scalar_scale) of one row already
 * rounded to fp32.  Reading R9. */
static void quant_nvfp4_row(const float *y32, int32_t H, int64_t t, int32_t layout,
                            float g, uint8_t *q, uint8_t *scales)
{
    int64_t C = H / 16;
    for (int64_t c = 0; c < C; c++) {
        float v[16];
        double amax = 0.0;
        for (int i = 0; i < 16; i++) {
            v[i] = (float)((double)g * (double)y32[c * 16 + i]); /* fp32 product */
            if (fabs((double)v[i]) > amax)
                amax = fabs((double)v[i]);
        }
        float sdiv = (float)(amax / 6.0);                 /* fp32 quotient */
        uint8_t sc = oracle_e4m3_from_f64((double)sdiv);
        double s = oracle_e4m3_to_f64(sc);
        scales[oracle_sf_offset(t, c, C, layout)] = sc;
        for (int i = 0; i < 16; i += 2) {
            uint8_t lo = 0, hi = 0;
            if (s != 0.0) {                               /* fp32 quotients v / s */
                lo = oracle_e2m1_from_f64((double)(float)((double)v[i] / s));
                hi = oracle_e2m1_from_f64((double)(float)((double)v[i + 1] / s));
            }
            q[c * 8 + i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* A 16-bit input element of the combine (bf16 or fp16, io_dtype). */
static double in16(const oracle_combine_args *a, uint16_t v)
{
    return a->io_dtype == 1 ? oracle_f16_to_f64(v) : oracle_bf16_to_f64(v);
}

/* A 16-bit output element (bf16 or fp16), round to nearest even. */
static uint16_t out16(const oracle_combine_args *a, double v)
{
    return a->io_dtype == 1 ? oracle_f64_to_f16(v) : oracle_f64_to_bf16(v);
}

/* Router weight (t, j) as fp32 (Struct_ep_combine_skip_a2a,
 * router_weights_dtype): stored as fp32, bf16 or fp16. */
static double weight_at(const oracle_combine_args *a, int64_t idx)
{
    if (a->weight_dtype == 1)
        return oracle_bf16_to_f64(((const uint16_t *)a->weights)[idx]);
    if (a->weight_dtype == 2)
        return oracle_f16_to_f64(((const uint16_t *)a->weights)[idx]);
    return (double)a->weights[idx];
}

int oracle_combine(const oracle_combine_args *a)
{
    if (!a || a->T < 0 || a->H < 1 || a->k < 1)
        return ORACLE_ERR_INVALID_ARG;
    if ((a->quant == 1 || a->quant == 3) && a->H % 32)
        return ORACLE_ERR_INVALID_ARG;
    if (a->quant == 2 && a->H % 16)
        return ORACLE_ERR_INVALID_ARG;
    int32_t H = a->H, k = a->k;
    double *s = (double *)malloc(sizeof(double) * (size_t)H);
    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    float *y32 = (float *)malloc(sizeof(float) * (size_t)H);
    if (!s || !x || !y32) {
        free(s); free(x); free(y32);
        return ORACLE_ERR_INVALID_ARG;
    }
    int status = ORACLE_OK;
    if (a->quant && a->scales_out && a->sf_layout == 1)
        memset(a->scales_out, 0, (size_t)oracle_scales_bytes(a->T, H, a->quant, 1));

    for (int64_t t = 0; t < a->T; t++) {
        /* routed sum, ascending slot j (Struct_ep_combine_skip_a2a, execute) */
        for (int32_t h = 0; h < H; h++)
            s[h] = 0.0;
        for (int32_t j = 0; j < k; j++) {
            /* slot-major: every slot of every token has its row
             * (trtllm_moe_allreduce_fusion, moe_reduction_active_experts_token_input) */
            int64_t r = a->expert_layout == 1 ? (int64_t)j * a->T + t : a->row_map[t * k + j];
            if (r < 0)
                continue; /* padded slot: contributes nothing */
            if (r >= a->n_rows) {
                status = ORACLE_ERR_INVALID_ARG;
                continue;
            }
            double w = weight_at(a, t * k + j);
            const uint16_t *row = a->expert_out + (int64_t)r * H;
            for (int32_t h = 0; h < H; h++)
                s[h] += w * in16(a, row[h]);
        }
        /* fused shared expert, weight 1 */
        if (a->shared)
            for (int32_t h = 0; h < H; h++)
                s[h] += in16(a, a->shared[t * H + h]);
        if (a->combined_out)
            for (int32_t h = 0; h < H; h++)
                a->combined_out[t * H + h] = out16(a, s[h]);
        /* residual add (trtllm_moe_allreduce_fusion residual_in / residual_out) */
        for (int32_t h = 0; h < H; h++)
            x[h] = s[h] + (a->residual ? in16(a, a->residual[t * H + h]) : 0.0);
        if (a->residual_out)
            for (int32_t h = 0; h < H; h++)
                a->residual_out[t * H + h] = out16(a, x[h]);
        /* RMSNorm with weight_bias (trtllm_moe_allreduce_fusion rms_gamma,
         * rms_eps, weight_bias) */
        if (a->gamma) {
            double ss = 0.0;
            for (int32_t h = 0; h < H; h++)
                ss += x[h] * x[h];
            double rinv = 1.0 / sqrt(ss / (double)H + (double)a->eps);
            for (int32_t h = 0; h < H; h++) {
                double g = in16(a, a->gamma[h]) + (double)a->weight_bias;
                x[h] = x[h] * rinv * g;
            }
            if (a->norm_out)
                for (int32_t h = 0; h < H; h++)
                    a->norm_out[t * H + h] = out16(a, x[h]);
        }
        if (a->y_out)
            for (int32_t h = 0; h < H; h++)
                a->y_out[t * H + h] = x[h];
        /* quantisation of the (normed) row, decided in fp32 */
        if (a->quant && a->quant_out && a->scales_out) {
            for (int32_t h = 0; h < H; h++)
                y32[h] = (float)x[h];
            if (a->quant == 1)
                quant_mxfp8_row(y32, H, t, a->sf_layout, a->quant_out + t * H, a->scales_out);
            else if (a->quant == 3)
                quant_mxfp4_row(y32, H, t, a->sf_layout, a->quant_out + t * (H / 2), a->scales_out);
            else
                quant_nvfp4_row(y32, H, t, a->sf_layout, a->global_scale,
                                a->quant_out + t * (H / 2), a->scales_out);
        }
    }
    free(s);
    free(x);
    free(y32);
    return status;
}

/* ------------------------------------------------------------------------ */
/* Dispatch-side permute                                                     */
/* ------------------------------------------------------------------------ */

/* The step before the expert computation, the inverse of the combine's
 * gather (flashinfer.comm.moe_a2a_combine: combine is the inverse of
 * moe_a2a_dispatch): token t's row x[t] is copied to every expert-grouped
 * row row_map[t, j] >= 0.  Rows of x_grouped that no slot names are left as
 * they are.  Returns ORACLE_ERR_INVALID_ARG if a row_map entry is >= n_rows
 * (that slot is skipped). */
int oracle_dispatch_permute(const uint16_t *x, int64_t T, int32_t H, const int32_t *row_map, int32_t k,
                            uint16_t *x_grouped, int64_t n_rows)
{
    int status = ORACLE_OK;
    for (int64_t t = 0; t < T; t++)
        for (int32_t j = 0; j < k; j++) {
            int32_t r = row_map[t * k + j];
            if (r < 0)
                continue;
            if (r >= n_rows) {
                status = ORACLE_ERR_INVALID_ARG;
                continue;
            }
            memcpy(x_grouped + (int64_t)r * H, x + t * H, sizeof(uint16_t) * (size_t)H);
        }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation (the formats' definitions), for comparisons in tests       */
/* ------------------------------------------------------------------------ */

/* out[t, h] = e4m3(q[t, h]) * 2^(scale - 127) */
void oracle_dequant_mxfp8(const uint8_t *q, const uint8_t *scales, int64_t T, int32_t H,
                          int32_t layout, double *out)
{
    int64_t C = H / 32;
    for (int64_t t = 0; t < T; t++)
        for (int32_t h = 0; h < H; h++) {
            uint8_t b = scales[oracle_sf_offset(t, h / 32, C, layout)];
            out[t * H + h] = ldexp(oracle_e4m3_to_f64(q[t * H + h]), (int)b - 127);
        }
}

/* out[t, h] = e2m1(q) * 2^(scale - 127) */
void oracle_dequant_mxfp4(const uint8_t *q, const uint8_t *scales, int64_t T, int32_t H, int32_t layout,
                          double *out)
{
    int64_t C = H / 32;
    for (int64_t t = 0; t < T; t++)
        for (int32_t h = 0; h < H; h++) {
            uint8_t byte = q[t * (H / 2) + h / 2];
            uint8_t code = (h & 1) ? (byte >> 4) : (byte & 15);
            uint8_t b = scales[oracle_sf_offset(t, h / 32, C, layout)];
            out[t * H + h] = ldexp(oracle_e2m1_to_f64(code), (int)b - 127);
        }
}

/* out[t, h] = e2m1(q) * e4m3(scale) / g */
void oracle_dequant_nvfp4(const uint8_t *q, const uint8_t *scales, int64_t T, int32_t H,
                          int32_t layout, float g, double *out)
{
    int64_t C = H / 16;
    for (int64_t t = 0; t < T; t++)
        for (int32_t h = 0; h < H; h++) {
            uint8_t byte = q[t * (H / 2) + h / 2];
            uint8_t code = (h & 1) ? (byte >> 4) : (byte & 15);
            double s = oracle_e4m3_to_f64(scales[oracle_sf_offset(t, h / 16, C, layout)]);
            out[t * H + h] = oracle_e2m1_to_f64(code) * s / (double)g;
        }
}
