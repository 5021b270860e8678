/*
 * fp8bs_oracle.c -- plain, slow CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * Only tests/, the smoke check and the benchmark's CPU-baseline leg use this
 * file.  It shares no code, table or constant generator with the CUDA
 * library: everything here is derived from the definitions it cites.
 *
 * Parity pins for each function live in tests/test_oracle_*.py.
 */
#include "fp8bs_oracle.h"

#include <assert.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define TILE 128   /* Atlas quantize_fp8_bs.rs: FP8_BLOCK = 128, both axes   */
#define MXG 32     /* FreeToken issue #624: one e8m0 scale per 32 elements   */
#define E4M3_MAX 448.0

/* ---------------------------------------------------------------------
 * e4m3fn ("E4M3 FN": 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, so the largest finite value is
 * 1.75 * 2^8 = 448).  This is the OCP 8-bit floating point E4M3 encoding
 * the pages call "e4m3" / "FP8 E4M3".
 * ------------------------------------------------------------------- */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);          /* subnormal: m/8 * 2^(1-7) */
    else
        mag = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7)     */
    return sign ? -mag : mag;
}

/*
 * Round to the nearest finite e4m3fn value by brute force: scan all 127
 * non-negative finite magnitudes (codes 0x00..0x7E, increasing in value) and
 * keep the closest; on a tie between two neighbours keep the one whose code
 * is even (even mantissa LSB = round-half-to-even).  |v| >= 448 saturates to
 * 448 ("satfinite").  The sign is reattached, so -0.0 and tiny negatives give
 * 0x80.
 *
 * Exactness of the distances: callers pass either a binary32 value or a
 * binary64 value with at most 8 significant bits.  For |v| >= 2^-10 both
 * |dec - |v|| are exact in binary64 (their bits span at most 2^8..2^-33);
 * below 2^-10 the nearest value is 0, whose distance |v| is exact, and every
 * other distance exceeds 2^-10 by far more than its rounding error.
 */
/* the 127 non-negative finite magnitudes, decoded once */
static double g_mag[0x7F];
static int g_mag_ready;

static void init_magnitudes(void)
{
    int c;
    if (g_mag_ready)
        return;
    for (c = 0; c < 0x7F; ++c)
        g_mag[c] = oracle_e4m3_decode((uint8_t)c);
    g_mag_ready = 1;
}

uint8_t oracle_e4m3_encode(double v)
{
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    int best = 0;
    double bestd;
    int c;
    assert(!isnan(v) && !isinf(v));
    if (a >= E4M3_MAX)
        return (uint8_t)(0x7E | (neg << 7));
    init_magnitudes();
    bestd = a; /* distance to code 0x00 (= 0.0) */
    for (c = 1; c <= 0x7E; ++c) {
        double d = fabs(g_mag[c] - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(best | (neg << 7));
}

void oracle_e4m3_encode_f32_array(const float *v, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode((double)v[i]);
}

/* ---------------------------------------------------------------------
 * bf16: the top 16 bits of an IEEE binary32.
 * ------------------------------------------------------------------- */
static float bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double oracle_bf16_to_double(uint16_t bits)
{
    return (double)bf16_to_float(bits);
}

/*
 * Round a double to bf16 (8 significant bits, exponent range of binary32,
 * subnormal quantum 2^-133), ties to even, overflow to infinity.
 */
uint16_t oracle_double_to_bf16(double v)
{
    int e2;
    double a, q, fl, frac, r;
    float f;
    uint32_t u;
    int neg = signbit(v) ? 1 : 0;
    if (isnan(v))
        return 0x7FC0;
    a = fabs(v);
    if (isinf(a) || a == 0.0) {
        r = a;
    } else {
        /* a = f * 2^e2 with f in [0.5, 1): the leading bit has weight
         * 2^(e2-1); bf16 keeps 8 bits, so the quantum is 2^(e2-8), but
         * never below the subnormal quantum 2^-133. */
        frexp(a, &e2);
        if (e2 - 8 < -133)
            e2 = -133 + 8;
        q = ldexp(a, -(e2 - 8));      /* exact: power-of-two scaling */
        fl = floor(q);
        frac = q - fl;                /* exact: q < 2^9 */
        if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
            fl += 1.0;
        r = ldexp(fl, e2 - 8);
        /* largest finite bf16 is (2 - 2^-7) * 2^127 */
        if (r > ldexp(255.0, 120))
            r = INFINITY;
    }
    f = (float)r; /* exact: r is a bf16 value (or inf) */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | (neg ? 0x8000u : 0u));
}

/* ---------------------------------------------------------------------
 * Block-FP8 quantization (128 x 128 tiles, fp32 scales).
 * ------------------------------------------------------------------- */
static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

void oracle_block_quantize_tile(const uint16_t *w, int64_t n, int64_t k,
                                int64_t bn, int64_t bk,
                                uint8_t *codes, float *scales)
{
    int64_t kb = cdiv(k, TILE);
    int64_t r0 = bn * TILE, c0 = bk * TILE;
    int64_t r1 = r0 + TILE < n ? r0 + TILE : n;
    int64_t c1 = c0 + TILE < k ? c0 + TILE : k;
    int64_t r, c;
    float amax = 0.0f, s;

    /* amax over the real elements of the tile only (ragged edge tiles) */
    for (r = r0; r < r1; ++r)
        for (c = c0; c < c1; ++c) {
            float a = fabsf(bf16_to_float(w[r * k + c]));
            assert(!isnan(a) && !isinf(a));
            if (a > amax)
                amax = a;
        }
    /* s = amax / 448 in binary32; an all-zero tile takes s = 1 */
    s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    scales[bn * kb + bk] = s;
    for (r = r0; r < r1; ++r)
        for (c = c0; c < c1; ++c) {
            float q = bf16_to_float(w[r * k + c]) / s; /* binary32 quotient */
            codes[r * k + c] = oracle_e4m3_encode((double)q);
        }
}

void oracle_block_quantize(const uint16_t *w, int64_t n, int64_t k,
                           uint8_t *codes, float *scales)
{
    int64_t bn, bk;
    for (bn = 0; bn < cdiv(n, TILE); ++bn)
        for (bk = 0; bk < cdiv(k, TILE); ++bk)
            oracle_block_quantize_tile(w, n, k, bn, bk, codes, scales);
}

/* ---------------------------------------------------------------------
 * MXFP8 quantization (groups of 32 consecutive K elements, e8m0 scales).
 * ------------------------------------------------------------------- */
static int mx_exponent(double amax)
{
    int e, E;
    if (amax == 0.0)
        return 127;
    /* smallest integer e with 448 * 2^e >= amax, by exact comparisons */
    frexp(amax, &e);
    e -= 9;
    while (ldexp(E4M3_MAX, e) < amax)
        ++e;
    while (ldexp(E4M3_MAX, e - 1) >= amax)
        --e;
    E = e + 127;
    if (E < 0)
        E = 0;
    if (E > 254)
        E = 254;
    return E;
}

static void mx_quantize_row(const uint16_t *w, int64_t k, int64_t r,
                            uint8_t *codes, uint8_t *e8m0)
{
    int64_t G = cdiv(k, MXG), g, c;
    for (g = 0; g < G; ++g) {
        int64_t c0 = g * MXG, c1 = c0 + MXG < k ? c0 + MXG : k;
        double amax = 0.0, scale;
        int E;
        for (c = c0; c < c1; ++c) {
            double a = fabs(oracle_bf16_to_double(w[r * k + c]));
            assert(!isnan(a) && !isinf(a));
            if (a > amax)
                amax = a;
        }
        E = mx_exponent(amax);
        e8m0[r * G + g] = (uint8_t)E;
        scale = ldexp(1.0, E - 127);
        for (c = c0; c < c1; ++c) /* w / 2^(E-127): exact in binary64 */
            codes[r * k + c] =
                oracle_e4m3_encode(oracle_bf16_to_double(w[r * k + c]) / scale);
    }
}

void oracle_mx_quantize(const uint16_t *w, int64_t n, int64_t k,
                        uint8_t *codes, uint8_t *e8m0)
{
    int64_t r;
    for (r = 0; r < n; ++r)
        mx_quantize_row(w, k, r, codes, e8m0);
}

void oracle_mx_quantize_rows(const uint16_t *w, int64_t n, int64_t k,
                             const int64_t *rows, int64_t nrows,
                             uint8_t *codes, uint8_t *e8m0)
{
    int64_t j;
    (void)n;
    for (j = 0; j < nrows; ++j)
        mx_quantize_row(w, k, rows[j], codes, e8m0);
}

/* ---------------------------------------------------------------------
 * W8A16 GEMV, y = x . dequant(W)^T, in binary64.  dec(q) * s is exact in
 * binary64 (4 + 24 significant bits) and so is each product with a bf16 x
 * (8 more bits); only the K-term sum rounds, at binary64 precision.
 * ------------------------------------------------------------------- */
void oracle_block_gemv(const uint16_t *x, int64_t m, const uint8_t *codes,
                       const float *scales, int64_t n, int64_t k,
                       const int64_t *rows, int64_t nrows, double *y64)
{
    double dec[256];
    int64_t kb = cdiv(k, TILE), mi, j, c;
    int i;
    if (rows == NULL)
        nrows = n;
    for (i = 0; i < 256; ++i)
        dec[i] = oracle_e4m3_decode((uint8_t)i);
    for (mi = 0; mi < m; ++mi)
        for (j = 0; j < nrows; ++j) {
            int64_t r = rows ? rows[j] : j;
            double sum = 0.0;
            for (c = 0; c < k; ++c) {
                double s = (double)scales[(r / TILE) * kb + c / TILE];
                double wq = dec[codes[r * k + c]] * s;
                sum += oracle_bf16_to_double(x[mi * k + c]) * wq;
            }
            y64[mi * nrows + j] = sum;
        }
}

void oracle_mx_gemv(const uint16_t *x, int64_t m, const uint8_t *codes,
                    const uint8_t *e8m0, int64_t n, int64_t k,
                    const int64_t *rows, int64_t nrows, double *y64)
{
    double dec[256];
    int64_t G = cdiv(k, MXG), mi, j, c;
    int i;
    if (rows == NULL)
        nrows = n;
    for (i = 0; i < 256; ++i)
        dec[i] = oracle_e4m3_decode((uint8_t)i);
    for (mi = 0; mi < m; ++mi)
        for (j = 0; j < nrows; ++j) {
            int64_t r = rows ? rows[j] : j;
            double sum = 0.0;
            for (c = 0; c < k; ++c) {
                double s = ldexp(1.0, (int)e8m0[r * G + c / MXG] - 127);
                double wq = dec[codes[r * k + c]] * s;
                sum += oracle_bf16_to_double(x[mi * k + c]) * wq;
            }
            y64[mi * nrows + j] = sum;
        }
}

/* ---------------------------------------------------------------------
 * Per-row and per-tensor FP8 (one fp32 scale per output row, or one for
 * the whole weight).  FreeToken PR #389 "load-time per-tensor FP8 dense
 * projections" (What this adds: e4m3 with one fp32 scale per weight; Why:
 * the per-row W8A16 route of its decode table).  The scale follows the
 * same rule as the 128x128 tiles: s = amax/448 in binary32 over the real
 * elements of the row (or tensor), s = 1 when they are all zero, and
 * q = e4m3(w/s) with the quotient formed in binary32.
 * ------------------------------------------------------------------- */
static float amax_of_rows(const uint16_t *w, int64_t k, int64_t r0, int64_t r1)
{
    float amax = 0.0f;
    int64_t i;
    for (i = r0 * k; i < r1 * k; ++i) {
        float a = fabsf(bf16_to_float(w[i]));
        assert(!isnan(a) && !isinf(a));
        if (a > amax)
            amax = a;
    }
    return amax;
}

static float scale_of_amax(float amax)
{
    return (amax == 0.0f) ? 1.0f : amax / 448.0f;
}

static void encode_row(const uint16_t *w, int64_t k, int64_t r, float s,
                       uint8_t *codes)
{
    int64_t c;
    for (c = 0; c < k; ++c) {
        float q = bf16_to_float(w[r * k + c]) / s; /* binary32 quotient */
        codes[r * k + c] = oracle_e4m3_encode((double)q);
    }
}

void oracle_row_quantize_rows(const uint16_t *w, int64_t n, int64_t k,
                              const int64_t *rows, int64_t nrows,
                              uint8_t *codes, float *scales)
{
    int64_t j;
    if (rows == NULL)
        nrows = n;
    for (j = 0; j < nrows; ++j) {
        int64_t r = rows ? rows[j] : j;
        float s = scale_of_amax(amax_of_rows(w, k, r, r + 1));
        scales[r] = s;
        encode_row(w, k, r, s, codes);
    }
}

void oracle_row_quantize(const uint16_t *w, int64_t n, int64_t k,
                         uint8_t *codes, float *scales)
{
    oracle_row_quantize_rows(w, n, k, NULL, 0, codes, scales);
}

void oracle_tensor_quantize_rows(const uint16_t *w, int64_t n, int64_t k,
                                 const int64_t *rows, int64_t nrows,
                                 uint8_t *codes, float *scale)
{
    int64_t j;
    float s = scale_of_amax(amax_of_rows(w, k, 0, n));
    *scale = s;
    if (rows == NULL)
        nrows = n;
    for (j = 0; j < nrows; ++j)
        encode_row(w, k, rows ? rows[j] : j, s, codes);
}

void oracle_tensor_quantize(const uint16_t *w, int64_t n, int64_t k,
                            uint8_t *codes, float *scale)
{
    oracle_tensor_quantize_rows(w, n, k, NULL, 0, codes, scale);
}

/* y64[mi, j] = sum_k x[mi,k] * dec(q[r,k]) * scales[r * scale_stride] with
 * r = rows[j], in binary64 (exact products, as for the block form). */
void oracle_row_gemv(const uint16_t *x, int64_t m, const uint8_t *codes,
                     const float *scales, int64_t scale_stride, int64_t n,
                     int64_t k, const int64_t *rows, int64_t nrows,
                     double *y64)
{
    double dec[256];
    int64_t mi, j, c;
    int i;
    if (rows == NULL)
        nrows = n;
    for (i = 0; i < 256; ++i)
        dec[i] = oracle_e4m3_decode((uint8_t)i);
    for (mi = 0; mi < m; ++mi)
        for (j = 0; j < nrows; ++j) {
            int64_t r = rows ? rows[j] : j;
            double s = (double)scales[r * scale_stride];
            double sum = 0.0;
            for (c = 0; c < k; ++c)
                sum += oracle_bf16_to_double(x[mi * k + c]) * (dec[codes[r * k + c]] * s);
            y64[mi * nrows + j] = sum;
        }
}

/* ---------------------------------------------------------------------
 * W8A8 (FreeToken PR #389, What this adds: a dynamic per-tensor activation
 * scale -- an amax pass, then the cast -- and a GEMM of the e4m3
 * activations with the per-tensor e4m3 weight, scaled by both scales).
 * The activation quantizer is oracle_tensor_quantize applied to x.
 * y64[mi, j] = sx * sw * sum_k dec(qx[mi,k]) * dec(qw[r,k]), r = rows[j]:
 * every product of two e4m3 values is exact in binary64, as is the
 * multiplication by the two binary32 scales of an exact sum.
 * ------------------------------------------------------------------- */
void oracle_w8a8_gemv(const uint8_t *xcodes, int64_t m, float sx,
                      const uint8_t *wcodes, float sw, int64_t n, int64_t k,
                      const int64_t *rows, int64_t nrows, double *y64)
{
    double dec[256];
    int64_t mi, j, c;
    int i;
    if (rows == NULL)
        nrows = n;
    for (i = 0; i < 256; ++i)
        dec[i] = oracle_e4m3_decode((uint8_t)i);
    for (mi = 0; mi < m; ++mi)
        for (j = 0; j < nrows; ++j) {
            int64_t r = rows ? rows[j] : j;
            double sum = 0.0;
            for (c = 0; c < k; ++c)
                sum += dec[xcodes[mi * k + c]] * dec[wcodes[r * k + c]];
            y64[mi * nrows + j] = sum * (double)sx * (double)sw;
        }
}

/* ---------------------------------------------------------------------
 * Grouped MoE GEMV (Atlas quantize_fp8_bs.rs, module notes: block-scaled
 * FP8 experts read by a grouped MoE GEMM with [N/128, K/128] fp32 scales).
 * Each (token t, slot j) output is the block GEMV of x[t] with expert
 * ids[t*topk + j]; an id outside [0, num_experts) leaves its row at 0.
 * y64 layout [m, topk, nrows].
 * ------------------------------------------------------------------- */
void oracle_moe_gemv(const uint16_t *x, int64_t m, const int32_t *ids,
                     int64_t topk, const uint8_t *codes, const float *scales,
                     int64_t num_experts, int64_t n, int64_t k,
                     const int64_t *rows, int64_t nrows, double *y64)
{
    int64_t nb = cdiv(n, TILE), kb = cdiv(k, TILE), t, j, r;
    if (rows == NULL)
        nrows = n;
    for (t = 0; t < m; ++t)
        for (j = 0; j < topk; ++j) {
            int32_t e = ids[t * topk + j];
            double *out = y64 + (t * topk + j) * nrows;
            if (e < 0 || e >= num_experts) {
                for (r = 0; r < nrows; ++r)
                    out[r] = 0.0;
                continue;
            }
            oracle_block_gemv(x + t * k, 1, codes + (int64_t)e * n * k,
                              scales + (int64_t)e * nb * kb, n, k, rows, nrows, out);
        }
}

/* ---------------------------------------------------------------------
 * FP8 E4M3 KV cache (InfiniLM PR #586, Summary: an F8 cache with per-layer
 * F32 k_scale / v_scale for paged attention; Benchmark: split-KV decode).
 * Paged layout: cache [num_blocks, page_size, num_kv_heads, head_dim] e4m3;
 * token i of sequence b lives in block block_table[b][i / page_size] at
 * offset i % page_size.  Appending quantizes like the per-tensor rule with
 * the given (static) scale: code = e4m3(x / scale), binary32 quotient.
 * ------------------------------------------------------------------- */
void oracle_kv_append(const uint16_t *x, int64_t num_tokens, int64_t kv_heads,
                      int64_t head_dim, const int32_t *slots, float scale,
                      uint8_t *cache)
{
    int64_t t, i, row = kv_heads * head_dim;
    for (t = 0; t < num_tokens; ++t)
        for (i = 0; i < row; ++i) {
            float q = bf16_to_float(x[t * row + i]) / scale; /* binary32 quotient */
            cache[(int64_t)slots[t] * row + i] = oracle_e4m3_encode((double)q);
        }
}

/* Decode attention over the cache, in binary64:
 *   s_l = sm_scale * sum_d q[b,h,d] * dec(K[l,g,d]) * k_scale   (g = h / (Hq/Hkv))
 *   p_l = exp(s_l - max s) / sum exp(s - max s)
 *   o[b,h,:] = sum_l p_l * dec(V[l,g,:]) * v_scale
 * over the seq_lens[b] tokens of sequence b.  o64 [batch, q_heads, head_dim];
 * an empty sequence gives zeros. */
void oracle_kv_attention(const uint16_t *q, int64_t batch, int64_t q_heads,
                         int64_t kv_heads, int64_t head_dim,
                         const uint8_t *k_cache, const uint8_t *v_cache,
                         float k_scale, float v_scale, const int32_t *block_table,
                         int64_t max_blocks, const int32_t *seq_lens,
                         int64_t page_size, double sm_scale, double *o64)
{
    double dec[256];
    int64_t b, h, l, d, group = q_heads / kv_heads, row = kv_heads * head_dim;
    int i;
    for (i = 0; i < 256; ++i)
        dec[i] = oracle_e4m3_decode((uint8_t)i);
    for (b = 0; b < batch; ++b)
        for (h = 0; h < q_heads; ++h) {
            int64_t g = h / group, len = seq_lens[b];
            const uint16_t *qv = q + (b * q_heads + h) * head_dim;
            double *out = o64 + (b * q_heads + h) * head_dim;
            double *s = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
            double mx = -INFINITY, sum = 0.0;
            for (d = 0; d < head_dim; ++d)
                out[d] = 0.0;
            for (l = 0; l < len; ++l) {
                int64_t slot = (int64_t)block_table[b * max_blocks + l / page_size] * page_size + l % page_size;
                const uint8_t *kr = k_cache + slot * row + g * head_dim;
                double dot = 0.0;
                for (d = 0; d < head_dim; ++d)
                    dot += oracle_bf16_to_double(qv[d]) * (dec[kr[d]] * (double)k_scale);
                s[l] = sm_scale * dot;
                if (s[l] > mx)
                    mx = s[l];
            }
            for (l = 0; l < len; ++l) {
                int64_t slot = (int64_t)block_table[b * max_blocks + l / page_size] * page_size + l % page_size;
                const uint8_t *vr = v_cache + slot * row + g * head_dim;
                double p = exp(s[l] - mx);
                sum += p;
                for (d = 0; d < head_dim; ++d)
                    out[d] += p * (dec[vr[d]] * (double)v_scale);
            }
            if (len > 0)
                for (d = 0; d < head_dim; ++d)
                    out[d] /= sum;
            free(s);
        }
}
