/*
 * dsv4_oracle.c -- plain, slow CPU oracle of the DeepSeek-V4 attention
 * O-projection hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: every step below is written out from the definitions on the
 * pages it cites.
 *
 * Pages cited:
 *   [grouped_wo_a]  vLLM docs, models/deepseek_v4/common/grouped_wo_a,
 *                   class DeepseekV4GroupedWoA (grouped_input, grouped_forward)
 *   [o_proj]        vLLM docs, models/deepseek_v4/nvidia/ops/o_proj,
 *                   compute_fp8_einsum_recipe, deep_gemm_fp8_o_proj,
 *                   rope_quant_attn_out
 *   [fused_quant]   vLLM docs, models/deepseek_v4/common/ops/
 *                   fused_inv_rope_fp8_quant (signature, parameter table,
 *                   shape asserts, derived sizes)
 *   [sglang_v4]     sglang python/sglang/srt/models/deepseek_v4.py,
 *                   MQALayer.forward (O-projection section), _dequant_fp8,
 *                   the rotary_emb construction (is_neox_style=False)
 *
 * Precision.  Where floating point only feeds a sum (the GEMMs) the oracle
 * works in fp64.  Where it decides an integer (the FP8 code and the UE8M0
 * exponent of a block) both sides must take the decision in the same
 * precision; the pages leave the kernel's precision open, so the rotated
 * value is formed in fp32 with one fixed operation order (see
 * oracle_inv_rope_pair) and everything after it is exact.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared
 *        -fPIC  (no -ffast-math: fmaf and the exact conversions rely on IEEE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_SHAPE (-1)
#define OR_ERR_NULL (-2)
#define OR_ERR_RANGE (-8)

/* Largest finite float8_e4m3fn value (torch.finfo(float8_e4m3fn).max), the
 * fp8_max the [fused_quant] wrapper passes to its kernel. */
#define E4M3_MAX 448.0

/* Floor on a block's amax before its scale is chosen.  The pages are silent on
 * all-zero blocks; this reading keeps the UE8M0 byte finite (it gives 105,
 * i.e. 2^-22, for an all-zero block). */
#define AMAX_FLOOR 1e-4f

/* Threads the oracle's parallel loops use (for reporting its timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the thread count of the parallel loops (timing only: every result is
 * the same at any thread count, each output element being computed whole by
 * one thread). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 -> float: a bf16 is the top half of an IEEE binary32. Exact. */
float oracle_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* double -> bf16, round to nearest, ties to even, taken directly from the
 * double (no intermediate float, so there is no double rounding).  bf16 has
 * 8 significant bits, exponent range of binary32, subnormal quantum 2^-133. */
uint16_t oracle_bf16_from_double(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0) return sign;
    int e;
    (void)frexp(ax, &e);          /* ax = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;             /* quantum of an 8-significant-bit value  */
    if (qexp < -133) qexp = -133; /* bf16 subnormal quantum                 */
    double r = ldexp(nearbyint(ldexp(ax, -qexp)), qexp); /* RNE (default mode) */
    if (r >= 0x1p128) return sign | 0x7F80;              /* overflow -> inf    */
    float rf = (float)r;          /* exact: r has <= 8 significant bits     */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* OCP FP8 E4M3 ("fn" variant, the float8_e4m3fn of the pages): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits, no infinities, NaN = S.1111.111.
 * Normal: 2^(E-7) * (1 + M/8), E in 1..15.  Subnormal: 2^-6 * M/8. */
double oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 0xF, M = c & 7;
    double v;
    if (E == 15 && M == 7) return NAN;
    if (E == 0) v = ldexp((double)M, -9);
    else v = ldexp(8.0 + M, E - 10);
    return s ? -v : v;
}

/* Nearest E4M3 value of q, ties to the even mantissa, saturating to +-448
 * ("satfinite"); the sign of q is kept, so -0 and negative values that round
 * to zero encode as 0x80.  Works from the format definition: in the binade
 * of q the spacing is 2^(E-10) (normal) or 2^-9 (subnormal). */
uint8_t oracle_e4m3_encode(double q)
{
    if (isnan(q)) return 0x7F;
    uint8_t sign = signbit(q) ? 0x80 : 0;
    double a = fabs(q);
    if (a >= E4M3_MAX) return sign | 0x7E; /* satfinite: 448 = E15 M6 */
    int e;
    (void)frexp(a, &e);           /* a = f * 2^e, f in [0.5,1); unbiased exponent e-1 */
    int E = (a == 0.0) ? 0 : (e - 1) + 7;
    int qexp = (E >= 1) ? (e - 1) - 3 : -9; /* spacing in this binade */
    double n = nearbyint(ldexp(a, -qexp));  /* RNE on the integer significand */
    double r = ldexp(n, qexp);
    if (r > E4M3_MAX) r = E4M3_MAX;         /* cannot happen below 448, kept for clarity */
    /* re-encode r (exactly representable) into bits */
    if (r == 0.0) return sign;
    int er;
    (void)frexp(r, &er);
    int Eb = (er - 1) + 7;
    uint8_t bits;
    if (Eb <= 0) {                          /* subnormal: r = M * 2^-9 */
        bits = (uint8_t)ldexp(r, 9);
    } else {
        int M = (int)(ldexp(r, -(er - 1)) * 8.0) - 8; /* r = 2^(er-1)*(1+M/8) */
        bits = (uint8_t)((Eb << 3) | M);
    }
    return sign | bits;
}

/* UE8M0 block exponent ([o_proj] compute_fp8_einsum_recipe: "SM100 uses packed
 * per-row E8M0 scales"; [fused_quant] parameter table: INT32 packed UE8M0).
 * The scale is the power of two 2^e; the plain definition of "block-scaled
 * with fp8_max" is: the smallest integer e with amax <= fp8_max * 2^e, so that
 * every scaled element fits the format.  amax is floored first (AMAX_FLOOR).
 * Written as the definition: start well below and step up; fp64 makes the
 * comparison exact (448 * 2^e and a binary32 amax are both exact doubles). */
int oracle_ue8m0_exponent(float amax)
{
    double a = (double)(amax > AMAX_FLOOR ? amax : AMAX_FLOOR);
    int e = ilogb(a) - 10;        /* certainly too small: 448*2^e < 2^(e+9) <= a */
    while (!(a <= ldexp(E4M3_MAX, e))) e++;
    return e;
}

void oracle_ue8m0_exponent_array(const float* amax, int64_t n, int32_t* e_out)
{
    for (int64_t i = 0; i < n; i++) e_out[i] = oracle_ue8m0_exponent(amax[i]);
}

void oracle_e4m3_encode_array(const double* q, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(q[i]);
}

void oracle_bf16_from_double_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_bf16_from_double(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Inverse RoPE                                                              */
/* ------------------------------------------------------------------------ */

/* One rotary pair, GPT-J / interleaved convention: sglang builds the rotary
 * embedding with is_neox_style=False, so lanes (2i, 2i+1) of the rope slice form
 * the complex number a + ib.  The inverse rotation ([sglang_v4]
 * fused_rope_inplace(..., inverse=True) on o[..., -rope_dim:]) multiplies by
 * conj(e^{i theta}) = c - i s:
 *     y0 = a*c + b*s,   y1 = b*c - a*s.
 * fp32 operation order (a reading: the vLLM kernel body is not shown): each
 * cross product is rounded to fp32 first and the other product is fused,
 *     y0 = fmaf(a, c, fl(b*s)),   y1 = fmaf(b, c, -fl(a*s)). */
void oracle_inv_rope_pair(float a, float b, float c, float s, float* y0, float* y1)
{
    float bs = b * s;   /* rounded product (no contraction: -ffp-contract=off) */
    float as = a * s;
    *y0 = fmaf(a, c, bs);
    *y1 = fmaf(b, c, -as);
}

/* The forward rotation, multiplication by e^{i theta} = c + i s; used only by
 * the round-trip pin (rotate, then inverse-rotate). */
void oracle_fwd_rope_pair(float a, float b, float c, float s, float* y0, float* y1)
{
    float bs = b * s;
    float as = a * s;
    *y0 = fmaf(a, c, -bs);
    *y1 = fmaf(b, c, as);
}

void oracle_inv_rope_pairs(const float* a, const float* b, const float* c, const float* s,
                           int64_t n, float* y0, float* y1)
{
    for (int64_t i = 0; i < n; i++) oracle_inv_rope_pair(a[i], b[i], c[i], s[i], &y0[i], &y1[i]);
}

void oracle_fwd_rope_pairs(const float* a, const float* b, const float* c, const float* s,
                           int64_t n, float* y0, float* y1)
{
    for (int64_t i = 0; i < n; i++) oracle_fwd_rope_pair(a[i], b[i], c[i], s[i], &y0[i], &y1[i]);
}

/* ------------------------------------------------------------------------ */
/* Layout rules                                                              */
/* ------------------------------------------------------------------------ */

/* get_tma_aligned_size(T, 4) ([fused_quant] derived sizes; [o_proj]
 * rope_quant_attn_out): the token extent of the MN-major scale tensor padded
 * so that a row of int32 is a whole number of 16-byte TMA units. */
int64_t oracle_tma_aligned_tokens(int64_t T)
{
    const int64_t per16 = 16 / 4;
    return (T + per16 - 1) / per16 * per16;
}

/* [fused_quant] shape asserts, in the order the wrapper states them. */
int oracle_check_quant_shapes(int64_t num_heads, int64_t head_dim, int64_t n_groups,
                              int64_t heads_per_group, int64_t nope_dim, int64_t rope_dim,
                              int64_t quant_group_size, int64_t cache_last_dim)
{
    if (n_groups <= 0 || heads_per_group <= 0 || quant_group_size <= 0) return OR_ERR_SHAPE;
    if (num_heads != n_groups * heads_per_group) return OR_ERR_SHAPE;
    if (head_dim != nope_dim + rope_dim) return OR_ERR_SHAPE;
    if (head_dim % quant_group_size != 0) return OR_ERR_SHAPE;
    if (nope_dim % quant_group_size != quant_group_size - rope_dim) return OR_ERR_SHAPE;
    if (rope_dim % 2 != 0) return OR_ERR_SHAPE;
    if (cache_last_dim != rope_dim) return OR_ERR_SHAPE;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* O-1: fused inverse RoPE + block-scaled FP8 quantisation                   */
/* ------------------------------------------------------------------------ */

/*
 * [fused_quant] fused_inv_rope_fp8_quant, tma_aligned_scales=True branch
 * (SM100 layout, [o_proj] compute_fp8_einsum_recipe for cap.major >= 10).
 *
 *   o          bf16 bits [T, H, head_dim], H = n_groups * heads_per_group
 *   positions  int64 [T], each in [0, max_pos)
 *   cache      fp32 [max_pos, rope_dim]: cos in [0, rope_dim/2), sin after
 *   out_fp8    e4m3 bits, physical [G][T][D], D = heads_per_group * head_dim
 *              (the returned view is [T, G, D] with strides (D, T*D, 1))
 *   out_scale  int32, physical [G][PK][T_al], PK = ceil(NB/4), NB = D/qgs,
 *              T_al = tma-aligned T (the view is [T, G, PK], strides
 *              (1, PK*T_al, T_al)); block kb of (t, g) is byte kb%4 of
 *              int32 kb/4 (little-endian byte order: a reading).
 *              Pad columns [T, T_al) are left untouched.
 *
 * Steps for every token t and group g (one row of D values):
 *   1. x = float(o[t, g*hpg + j/head_dim, j%head_dim])                (exact)
 *   2. the last rope_dim lanes of each head are inverse-rotated with row
 *      positions[t] of the cache; the other lanes pass through.
 *   3. for each block of qgs consecutive values: amax = max |y|,
 *      e = oracle_ue8m0_exponent(amax), byte = e + 127.
 *   4. code = e4m3(y * 2^-e)  (the scaling is exact in fp64).
 */
int oracle_inv_rope_fp8_quant(const uint16_t* o, const int64_t* positions, const float* cache,
                              int64_t T, int64_t max_pos, int64_t n_groups, int64_t heads_per_group,
                              int64_t nope_dim, int64_t rope_dim, int64_t quant_group_size,
                              uint8_t* out_fp8, int32_t* out_scale)
{
    const int64_t head_dim = nope_dim + rope_dim;
    const int64_t H = n_groups * heads_per_group;
    int rc = oracle_check_quant_shapes(H, head_dim, n_groups, heads_per_group, nope_dim, rope_dim,
                                       quant_group_size, rope_dim);
    if (rc != OR_OK) return rc;
    if (T < 0 || max_pos <= 0) return OR_ERR_SHAPE;
    if (T == 0) return OR_OK;
    if (!o || !positions || !cache || !out_fp8 || !out_scale) return OR_ERR_NULL;
    for (int64_t t = 0; t < T; t++)
        if (positions[t] < 0 || positions[t] >= max_pos) return OR_ERR_RANGE;

    const int64_t D = heads_per_group * head_dim;
    const int64_t NB = D / quant_group_size;
    const int64_t PK = (NB + 3) / 4;
    const int64_t T_al = oracle_tma_aligned_tokens(T);
    const int64_t half = rope_dim / 2;
    if (PK > 64) return OR_ERR_SHAPE; /* this oracle's per-row pack buffer */

#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        float* y = (float*)malloc(sizeof(float) * (size_t)D);
        const float* crow = cache + positions[t] * rope_dim;
        for (int64_t g = 0; g < n_groups; g++) {
            /* 1-2. load, rotate the rope lanes of every head of the group */
            for (int64_t hh = 0; hh < heads_per_group; hh++) {
                const uint16_t* src = o + (t * H + g * heads_per_group + hh) * head_dim;
                float* dst = y + hh * head_dim;
                for (int64_t j = 0; j < head_dim; j++) dst[j] = oracle_bf16_to_float(src[j]);
                for (int64_t i = 0; i < half; i++) {
                    float a = dst[nope_dim + 2 * i], b = dst[nope_dim + 2 * i + 1];
                    oracle_inv_rope_pair(a, b, crow[i], crow[half + i],
                                         &dst[nope_dim + 2 * i], &dst[nope_dim + 2 * i + 1]);
                }
            }
            /* 3-4. per-block scale and codes */
            uint8_t* qrow = out_fp8 + (g * T + t) * D;
            uint32_t packed[64];
            memset(packed, 0, sizeof packed);
            for (int64_t kb = 0; kb < NB; kb++) {
                float amax = 0.0f;
                for (int64_t j = 0; j < quant_group_size; j++) {
                    float v = fabsf(y[kb * quant_group_size + j]);
                    if (v > amax) amax = v;
                }
                int e = oracle_ue8m0_exponent(amax);
                uint32_t byte = (uint32_t)(e + 127);
                packed[kb / 4] |= byte << (8 * (kb % 4));
                for (int64_t j = 0; j < quant_group_size; j++) {
                    double q = ldexp((double)y[kb * quant_group_size + j], -e);
                    qrow[kb * quant_group_size + j] = oracle_e4m3_encode(q);
                }
            }
            for (int64_t p = 0; p < PK; p++)
                out_scale[(g * PK + p) * T_al + t] = (int32_t)packed[p];
        }
        free(y);
    }
    return OR_OK;
}

/*
 * The quantize=False variant ([grouped_wo_a] grouped_input: "The BF16
 * inverse-rotated groups, [num_tokens, n_groups, group_dim]"; [o_proj]
 * deep_gemm_fp8_o_proj passes quantize=use_fp8): steps 1-2 of O-1, then every
 * value rounded to bf16 (nearest, ties to even).  Nope lanes come back exactly.
 * out_bf16 physical [G][T][D], the same group-major layout as the FP8 codes.
 */
int oracle_inv_rope_bf16(const uint16_t* o, const int64_t* positions, const float* cache,
                         int64_t T, int64_t max_pos, int64_t n_groups, int64_t heads_per_group,
                         int64_t nope_dim, int64_t rope_dim, uint16_t* out_bf16)
{
    const int64_t head_dim = nope_dim + rope_dim;
    const int64_t H = n_groups * heads_per_group;
    if (n_groups <= 0 || heads_per_group <= 0 || nope_dim < 0 || rope_dim <= 0 || rope_dim % 2)
        return OR_ERR_SHAPE;
    if (T < 0 || max_pos <= 0) return OR_ERR_SHAPE;
    if (T == 0) return OR_OK;
    if (!o || !positions || !cache || !out_bf16) return OR_ERR_NULL;
    for (int64_t t = 0; t < T; t++)
        if (positions[t] < 0 || positions[t] >= max_pos) return OR_ERR_RANGE;
    const int64_t D = heads_per_group * head_dim;
    const int64_t half = rope_dim / 2;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        const float* crow = cache + positions[t] * rope_dim;
        for (int64_t h = 0; h < H; h++) {
            const int64_t g = h / heads_per_group, hh = h % heads_per_group;
            const uint16_t* src = o + (t * H + h) * head_dim;
            uint16_t* dst = out_bf16 + (g * T + t) * D + hh * head_dim;
            for (int64_t j = 0; j < nope_dim; j++) dst[j] = src[j];
            for (int64_t i = 0; i < half; i++) {
                float y0, y1;
                oracle_inv_rope_pair(oracle_bf16_to_float(src[nope_dim + 2 * i]),
                                     oracle_bf16_to_float(src[nope_dim + 2 * i + 1]), crow[i],
                                     crow[half + i], &y0, &y1);
                dst[nope_dim + 2 * i] = oracle_bf16_from_double((double)y0);
                dst[nope_dim + 2 * i + 1] = oracle_bf16_from_double((double)y1);
            }
        }
    }
    return OR_OK;
}

/*
 * The bf16 grouped product ([o_proj] deep_gemm_fp8_o_proj when wo_a is not
 * FP8: torch.bmm of the [G, T, D] groups with wo_a.weight viewed [G, R, D],
 * transposed):  z[t, g, n] = sum_k x[g][t][k] * W[g*R + n][k], fp64 sum,
 * bf16 result.   x_bf16 physical [G][T][D], w_bf16 [G*R][D], z [T][G][R].
 */
int oracle_grouped_gemm_bf16(const uint16_t* x_bf16, const uint16_t* w_bf16, int64_t T, int64_t G,
                             int64_t D, int64_t R, double* z64, uint16_t* z_bf16)
{
    if (T < 0 || G <= 0 || D <= 0 || R <= 0) return OR_ERR_SHAPE;
    if (T == 0) return OR_OK;
    if (!x_bf16 || !w_bf16 || !z_bf16) return OR_ERR_NULL;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t tg = 0; tg < T * G; tg++) {
        const int64_t t = tg / G, g = tg % G;
        const uint16_t* xr = x_bf16 + (g * T + t) * D;
        for (int64_t n = 0; n < R; n++) {
            const uint16_t* wr = w_bf16 + (g * R + n) * D;
            double acc = 0.0;
            for (int64_t k = 0; k < D; k++)
                acc += (double)oracle_bf16_to_float(xr[k]) * (double)oracle_bf16_to_float(wr[k]);
            if (z64) z64[(t * G + g) * R + n] = acc;
            z_bf16[(t * G + g) * R + n] = oracle_bf16_from_double(acc);
        }
    }
    return OR_OK;
}

/* The same steps without rotation, on a plain [T, C] bf16 matrix: the per-token
 * 1 x qgs block quantisation that the FP8 wo_b projection applies to the
 * flattened bf16 z ([o_proj] deep_gemm_fp8_o_proj returns wo_b(z.flatten(1));
 * [sglang_v4] builds wo_b with the FP8 block quant_config; the activation
 * quantisation inside that linear is not printed, so it is read as the same
 * per-128 UE8M0 rule).  Output layout matches O-1 with G = 1:
 * out_fp8 [T][C], out_scale [PK][T_al]. */
int oracle_block_quant_rows(const uint16_t* x, int64_t T, int64_t C, int64_t quant_group_size,
                            uint8_t* out_fp8, int32_t* out_scale)
{
    if (T < 0 || C <= 0 || quant_group_size <= 0 || C % quant_group_size) return OR_ERR_SHAPE;
    if (T == 0) return OR_OK;
    if (!x || !out_fp8 || !out_scale) return OR_ERR_NULL;
    const int64_t NB = C / quant_group_size, PK = (NB + 3) / 4;
    const int64_t T_al = oracle_tma_aligned_tokens(T);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        for (int64_t p = 0; p < PK; p++) out_scale[p * T_al + t] = 0;
        for (int64_t kb = 0; kb < NB; kb++) {
            const uint16_t* src = x + t * C + kb * quant_group_size;
            float amax = 0.0f;
            for (int64_t j = 0; j < quant_group_size; j++) {
                float v = fabsf(oracle_bf16_to_float(src[j]));
                if (v > amax) amax = v;
            }
            int e = oracle_ue8m0_exponent(amax);
            out_scale[(kb / 4) * T_al + t] |= (int32_t)((uint32_t)(e + 127) << (8 * (kb % 4)));
            for (int64_t j = 0; j < quant_group_size; j++)
                out_fp8[t * C + kb * quant_group_size + j] =
                    oracle_e4m3_encode(ldexp((double)oracle_bf16_to_float(src[j]), -e));
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* O-2 / O-3: block-scaled FP8 (grouped) GEMM                               */
/* ------------------------------------------------------------------------ */

/*
 * z[t, g, n] = sum_k dq_x[t, g, k] * dq_w[g*R + n, k]
 *
 * [grouped_wo_a]: group g meets only wo_a rows g*R:(g+1)*R.
 * [o_proj] deep_gemm_fp8_o_proj: fp8_einsum("bhr,hdr->bhd") over the quantised
 * groups and wo_a.weight viewed [G, R, D]; the bf16 fallback is the same
 * product as torch.bmm.  z is allocated bf16.
 * [sglang_v4] _dequant_fp8: weight block (sn, sk) of 128 x 128 is multiplied by
 * scale[sn, sk].
 *
 *   x_fp8    e4m3 physical [G][T][D]        (O-1's out_fp8)
 *   x_scale  int32 physical [G][PK][T_al]   (O-1's out_scale)
 *   w_fp8    e4m3 [G*R, D] row-major
 *   w_scale  UE8M0 bytes [G*R/128, D/128] row-major
 *   z64      optional fp64 [T][G][R] (the exact-sum reference, before rounding)
 *   z_bf16   bf16 bits [T][G][R]: z64 rounded to nearest even
 *
 * Dequantised values are exact in fp64; the sum is accumulated in fp64 in
 * increasing k.  With G = 1 this is also the dense wo_b projection
 * out[t, h] = sum_c dq(zq)[t, c] * dq(Wb)[h, c].
 */
int oracle_grouped_gemm(const uint8_t* x_fp8, const int32_t* x_scale, int64_t T, int64_t G,
                        int64_t D, int64_t R, const uint8_t* w_fp8, const uint8_t* w_scale,
                        double* z64, uint16_t* z_bf16)
{
    if (T < 0 || G <= 0 || D <= 0 || R <= 0 || D % 128 || R % 128) return OR_ERR_SHAPE;
    if (T == 0) return OR_OK;
    if (!x_fp8 || !x_scale || !w_fp8 || !w_scale || !z_bf16) return OR_ERR_NULL;
    const int64_t NB = D / 128, PK = (NB + 3) / 4, T_al = oracle_tma_aligned_tokens(T);
    const int64_t KB = D / 128; /* weight scale columns */

    double lut[256];
    for (int c = 0; c < 256; c++) lut[c] = oracle_e4m3_decode((uint8_t)c);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t tg = 0; tg < T * G; tg++) {
        const int64_t t = tg / G, g = tg % G;
        double* xs = (double*)malloc(sizeof(double) * (size_t)D);
        const uint8_t* xrow = x_fp8 + (g * T + t) * D;
        for (int64_t k = 0; k < D; k++) {
            int64_t kb = k / 128;
            uint32_t word = (uint32_t)x_scale[(g * PK + kb / 4) * T_al + t];
            int e = (int)((word >> (8 * (kb % 4))) & 0xFF) - 127;
            xs[k] = ldexp(lut[xrow[k]], e);
        }
        for (int64_t n = 0; n < R; n++) {
            const int64_t row = g * R + n;
            const uint8_t* wrow = w_fp8 + row * D;
            const uint8_t* srow = w_scale + (row / 128) * KB;
            double acc = 0.0;
            for (int64_t kb = 0; kb < KB; kb++) {
                const double sc = ldexp(1.0, (int)srow[kb] - 127); /* exact power of two */
                for (int64_t k = kb * 128; k < kb * 128 + 128; k++)
                    acc += xs[k] * (lut[wrow[k]] * sc);          /* exact product terms */
            }
            if (z64) z64[(t * G + g) * R + n] = acc;
            z_bf16[(t * G + g) * R + n] = oracle_bf16_from_double(acc);
        }
        free(xs);
    }
    return OR_OK;
}

/*
 * The whole O-projection for a set of tokens ([o_proj] deep_gemm_fp8_o_proj):
 * O-1 quantisation, the grouped wo_a GEMM into bf16 z [T, G, R], the per-128
 * re-quantisation of z.flatten(1) and the dense wo_b GEMM into bf16 out
 * [T, hidden].  Scratch is allocated here (this is a test oracle).
 * Optional outputs (may be NULL): z_bf16 [T][G][R], out64 [T][hidden].
 */
int oracle_o_proj(const uint16_t* o, const int64_t* positions, const float* cache, int64_t T,
                  int64_t max_pos, int64_t n_groups, int64_t heads_per_group, int64_t nope_dim,
                  int64_t rope_dim, int64_t quant_group_size, int64_t o_lora_rank, int64_t hidden,
                  const uint8_t* wo_a, const uint8_t* wo_a_scale, const uint8_t* wo_b,
                  const uint8_t* wo_b_scale, uint16_t* z_bf16_out, double* out64,
                  uint16_t* out_bf16)
{
    if (T < 0 || hidden <= 0 || hidden % 128 || o_lora_rank <= 0 || o_lora_rank % 128)
        return OR_ERR_SHAPE;
    if (quant_group_size != 128) return OR_ERR_SHAPE;
    if (T == 0) return OR_OK;
    const int64_t head_dim = nope_dim + rope_dim;
    const int64_t D = heads_per_group * head_dim;
    const int64_t NB = D / quant_group_size, PK = (NB + 3) / 4;
    const int64_t T_al = oracle_tma_aligned_tokens(T);
    const int64_t C = n_groups * o_lora_rank;
    const int64_t PKC = (C / 128 + 3) / 4;
    int rc;
    uint8_t* xq = (uint8_t*)malloc((size_t)(n_groups * T * D));
    int32_t* xs = (int32_t*)calloc((size_t)(n_groups * PK * T_al), sizeof(int32_t));
    uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * C));
    uint8_t* zq = (uint8_t*)malloc((size_t)(T * C));
    int32_t* zs = (int32_t*)calloc((size_t)(PKC * T_al), sizeof(int32_t));
    if (!xq || !xs || !z || !zq || !zs) { rc = OR_ERR_SHAPE; goto done; }
    rc = oracle_inv_rope_fp8_quant(o, positions, cache, T, max_pos, n_groups, heads_per_group,
                                   nope_dim, rope_dim, quant_group_size, xq, xs);
    if (rc != OR_OK) goto done;
    rc = oracle_grouped_gemm(xq, xs, T, n_groups, D, o_lora_rank, wo_a, wo_a_scale, NULL, z);
    if (rc != OR_OK) goto done;
    if (z_bf16_out) memcpy(z_bf16_out, z, sizeof(uint16_t) * (size_t)(T * C));
    rc = oracle_block_quant_rows(z, T, C, 128, zq, zs);
    if (rc != OR_OK) goto done;
    rc = oracle_grouped_gemm(zq, zs, T, 1, C, hidden, wo_b, wo_b_scale, out64, out_bf16);
done:
    free(xq); free(xs); free(z); free(zq); free(zs);
    return rc;
}
