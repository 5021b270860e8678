/*
 * fp8bs_oracle.h -- plain, slow CPU oracle for block-scaled FP8 / MXFP8
 * weight quantization and the W8A16 GEMV that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  This code is the independent statement of what
 * the library computes; it exists so that tests, the smoke check and the
 * benchmark's CPU baseline can compare against it.  No product code path may
 * include, link or call it, and it shares no code with the CUDA library.
 *
 * Formats and layouts (all row-major, K contiguous):
 *   w      bf16 [N,K]              (uint16_t bit patterns)
 *   codes  e4m3fn [N,K]            one byte per weight
 *   scales fp32 [ceil(N/128), ceil(K/128)]        128x128 block scales
 *   e8m0   uint8 [N, ceil(K/32)]   MX power-of-two scale exponents (bias 127)
 *   row scales fp32 [N]; tensor scale fp32 [1]
 *   x      bf16 [M,K], y bf16 [M,N]
 *
 * Sources: FreeToken PR #636 "opt-in fp8-block QAT for the lm_head"
 * (How it works, Changes, Validation); Atlas spark_model/weight_map/
 * quantize_fp8_bs.rs (quantize_to_fp8_blockscaled: [n,k] bf16 weight,
 * one byte per weight, one f32 per [128,128] tile, [n_blocks, k_blocks]
 * grid); FreeToken issue #624 "Load-time MXFP8 requantization" (Proposed
 * solution: e4m3 codes, one e8m0 scale per 32 elements, ceil-log2 of
 * amax/448); InfiniLM PR #586 (Summary: 128x128 block scales, W8A16);
 * FreeToken PR #389 "load-time per-tensor FP8 dense projections" (What
 * this adds: one fp32 scale per weight; Why: the per-row W8A16 route).
 *
 * Build: plain C11, no -ffast-math, -ffp-contract=off, so that every float
 * operation below is one IEEE-754 binary32 or binary64 operation.
 */
#ifndef FP8BS_ORACLE_H
#define FP8BS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* e4m3fn code -> value (NaN for 0x7F / 0xFF). */
double oracle_e4m3_decode(uint8_t code);
/* nearest e4m3fn code, ties to even, saturating to +-448; sign kept for zero. */
uint8_t oracle_e4m3_encode(double v);
/* element-wise oracle_e4m3_encode over binary32 inputs. */
void oracle_e4m3_encode_f32_array(const float *v, int64_t n, uint8_t *out);

double oracle_bf16_to_double(uint16_t bits);
/* round a double to the nearest bf16 (ties to even; overflow -> inf). */
uint16_t oracle_double_to_bf16(double v);

/* 128x128 block quantization: amax over the real elements of each tile,
 * s = amax/448 in fp32 (s = 1 for an all-zero tile), q = e4m3(w/s) with the
 * quotient formed in fp32. */
void oracle_block_quantize(const uint16_t *w, int64_t n, int64_t k,
                           uint8_t *codes, float *scales);
/* the same for a single tile (bn, bk); writes only that tile's codes and
 * its one scale into the full-size arrays. */
void oracle_block_quantize_tile(const uint16_t *w, int64_t n, int64_t k,
                                int64_t bn, int64_t bk,
                                uint8_t *codes, float *scales);

/* MXFP8: per row, per group of 32 consecutive K elements (the last group
 * may be short): e = smallest integer with 448*2^e >= amax, E = e+127
 * clamped to [0,254] (E = 127 for amax = 0), q = e4m3(w * 2^(127-E)). */
void oracle_mx_quantize(const uint16_t *w, int64_t n, int64_t k,
                        uint8_t *codes, uint8_t *e8m0);
void oracle_mx_quantize_rows(const uint16_t *w, int64_t n, int64_t k,
                             const int64_t *rows, int64_t nrows,
                             uint8_t *codes, uint8_t *e8m0);

/* y64[mi, j] = sum_k x[mi,k] * dec(q[rows[j],k]) * s(rows[j],k), in fp64.
 * Output layout [m, nrows].  rows == NULL means all n rows in order. */
void oracle_block_gemv(const uint16_t *x, int64_t m, const uint8_t *codes,
                       const float *scales, int64_t n, int64_t k,
                       const int64_t *rows, int64_t nrows, double *y64);
void oracle_mx_gemv(const uint16_t *x, int64_t m, const uint8_t *codes,
                    const uint8_t *e8m0, int64_t n, int64_t k,
                    const int64_t *rows, int64_t nrows, double *y64);

/* Per-row FP8: one fp32 scale per output row, s_r = amax_r/448 in fp32
 * (s = 1 for an all-zero row), q = e4m3(w/s_r) with the quotient in fp32.
 * scales has n entries; the _rows form writes only the listed rows (NULL:
 * all n rows in order). */
void oracle_row_quantize(const uint16_t *w, int64_t n, int64_t k,
                         uint8_t *codes, float *scales);
void oracle_row_quantize_rows(const uint16_t *w, int64_t n, int64_t k,
                              const int64_t *rows, int64_t nrows,
                              uint8_t *codes, float *scales);
/* Per-tensor FP8: the same with one scale over all n*k elements.  The _rows
 * form still takes the amax over the whole tensor but encodes only the
 * listed rows. */
void oracle_tensor_quantize(const uint16_t *w, int64_t n, int64_t k,
                            uint8_t *codes, float *scale);
void oracle_tensor_quantize_rows(const uint16_t *w, int64_t n, int64_t k,
                                 const int64_t *rows, int64_t nrows,
                                 uint8_t *codes, float *scale);
/* y64[mi, j] = sum_k x[mi,k] * dec(q[rows[j],k]) * scales[rows[j]*stride]
 * in fp64; stride 1 for per-row scales, 0 for a per-tensor scale. */
void oracle_row_gemv(const uint16_t *x, int64_t m, const uint8_t *codes,
                     const float *scales, int64_t scale_stride, int64_t n,
                     int64_t k, const int64_t *rows, int64_t nrows,
                     double *y64);

/* W8A8: x quantized per tensor (oracle_tensor_quantize of x gives xcodes,
 * sx), weight per tensor (wcodes, sw).  y64[mi, j] = sx * sw *
 * sum_k dec(qx[mi,k]) * dec(qw[rows[j],k]) in fp64; rows == NULL: all. */
void oracle_w8a8_gemv(const uint8_t *xcodes, int64_t m, float sx,
                      const uint8_t *wcodes, float sw, int64_t n, int64_t k,
                      const int64_t *rows, int64_t nrows, double *y64);

/* Grouped MoE: y64[t, j, r] = block GEMV of x[t] with expert ids[t*topk+j]
 * (codes [E, n, k], scales [E, ceil(n/128), ceil(k/128)]); out-of-range
 * ids give 0.  Layout [m, topk, nrows]. */
void oracle_moe_gemv(const uint16_t *x, int64_t m, const int32_t *ids,
                     int64_t topk, const uint8_t *codes, const float *scales,
                     int64_t num_experts, int64_t n, int64_t k,
                     const int64_t *rows, int64_t nrows, double *y64);

/* FP8 KV cache, paged: cache [num_blocks, page_size, kv_heads, head_dim]
 * e4m3.  Append: cache[slots[t]] = e4m3(x[t] / scale) (binary32 quotient). */
void oracle_kv_append(const uint16_t *x, int64_t num_tokens, int64_t kv_heads,
                      int64_t head_dim, const int32_t *slots, float scale,
                      uint8_t *cache);
/* Decode attention in fp64 (softmax over seq_lens[b] tokens, GQA group =
 * q_heads / kv_heads); o64 [batch, q_heads, head_dim]. */
void oracle_kv_attention(const uint16_t *q, int64_t batch, int64_t q_heads,
                         int64_t kv_heads, int64_t head_dim,
                         const uint8_t *k_cache, const uint8_t *v_cache,
                         float k_scale, float v_scale, const int32_t *block_table,
                         int64_t max_blocks, const int32_t *seq_lens,
                         int64_t page_size, double sm_scale, double *o64);

#ifdef __cplusplus
}
#endif
#endif
