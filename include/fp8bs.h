/*
 * fp8bs.h -- C ABI of libfp8bs: block-scaled FP8 (E4M3), MXFP8 and per-row /
 * per-tensor FP8 weight quantization, the W8A16 GEMV / skinny GEMM /
 * prefill GEMM that consumes it, the W8A8 route (dynamic per-tensor
 * activation quantization + e4m3 x e4m3 GEMM), the grouped MoE GEMV and an
 * FP8 E4M3 paged KV cache with split-KV decode attention, for NVIDIA GB300
 * (sm_103a).
 *
 * Common conventions
 * ------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller; the
 *    library never allocates, frees or keeps a pointer after the call
 *    returns ("The BF16 source is the caller's to free -- this does not take
 *    ownership", Atlas spark_model/weight_map/quantize_fp8_bs.rs).
 *  - Matrices are row-major with the last index contiguous:
 *      weight w   bf16  [n, k]   (n = output features, k = input features)
 *      codes      e4m3  [n, k]   one byte per weight
 *      scales     fp32  [ceil(n/128), ceil(k/128)]   one per 128x128 tile
 *      e8m0       uint8 [n, ceil(k/32)]              one per 32 k of a row
 *      row scales fp32  [n] (per row) or [1] (per tensor)
 *      x          bf16  [m, k]
 *      y          bf16  [m, n]
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    only enqueues work on `stream` and returns: no host synchronisation, no
 *    allocation, and the kernel choice depends on shapes only, never on
 *    values, so a sequence of calls can be captured into a CUDA graph.
 *  - Arguments are validated before anything is enqueued; on a negative
 *    status nothing was launched.  Launch failures report FP8BS_ERR_CUDA.
 *  - Inputs must be finite (no NaN or Inf); results for non-finite inputs
 *    are unspecified.
 *  - Results are deterministic: for a given shape the reduction order is
 *    fixed.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_NULL = -1,    /* a required pointer is NULL                     */
    FP8BS_ERR_SHAPE = -2,   /* n, k or m out of range                         */
    FP8BS_ERR_BLOCK = -3,   /* block size other than 128                      */
    FP8BS_ERR_ALIGN = -4,   /* pointer not aligned to its element size        */
    FP8BS_ERR_CUDA = -5,    /* a CUDA runtime/driver call or launch failed    */
    FP8BS_ERR_DEVICE = -6,  /* a kernel gave up a bounded wait (see below)    */
    FP8BS_ERR_PATH = -7     /* the requested kernel path cannot take the call */
} fp8bs_status;

/* Kernel paths for the *_ex entry points. */
typedef enum {
    FP8BS_PATH_AUTO = 0,     /* choose by shape (what fp8bs_gemv does)         */
    FP8BS_PATH_DECODE = 1,   /* TMA-staged skinny kernel, m <= 32 per launch
                                (larger m runs in chunks of 32 rows)          */
    FP8BS_PATH_PREFILL = 2,  /* tcgen05 tensor-core kernel (block / row / tensor
                                scales, MXFP8)                               */
    FP8BS_PATH_GENERIC = 3   /* plain-load kernel for any shape / alignment    */
} fp8bs_path;

/*
 * fp8bs_quantize -- load-time requantization of a bf16 [n, k] weight to FP8
 * E4M3 codes with one fp32 scale per 128x128 tile.
 *
 * Defined by: Atlas spark_model/weight_map/quantize_fp8_bs.rs
 * (quantize_to_fp8_blockscaled: [n, k] bf16 in, one byte per weight, one f32
 * per [128,128] tile laid out [n_blocks, k_blocks], n > 0 && k > 0 required,
 * launch grid [k_blocks, n_blocks]); FreeToken PR #636 "opt-in fp8-block QAT
 * for the lm_head" (How it works: quantize to fp8 with a 128-block scale
 * after load); FreeToken issue #624 (amax/448).
 *
 * For each tile (bn, bk), over the tile's real elements only (edge tiles may
 * be partial): amax = max|w|, s = amax / 448 as an IEEE fp32 division, s = 1
 * when amax = 0; codes[r, c] = e4m3(w[r, c] / s) with the quotient an IEEE
 * fp32 division, rounded to nearest-even and saturated to +-448.
 *
 *   w_bf16      device, n*k bf16, 2-byte aligned
 *   n, k        > 0 (else FP8BS_ERR_SHAPE)
 *   block       must be 128, the tile edge the consumers hard-code
 *               (else FP8BS_ERR_BLOCK)
 *   codes_u8    device, n*k bytes, written
 *   scales_f32  device, ceil(n/128)*ceil(k/128) floats, 4-byte aligned
 *   stream      cudaStream_t
 * Any alignment is accepted; 16-byte-aligned w with k % 8 == 0 takes the
 * vectorised kernel, everything else a scalar kernel with identical results.
 */
int fp8bs_quantize(const void *w_bf16, int64_t n, int64_t k, int block,
                   uint8_t *codes_u8, float *scales_f32, void *stream);

/*
 * fp8bs_gemv -- decode-time W8A16 block-FP8 linear:
 *   y[i, j] = bf16_rn( sum_kb s[j/128, kb] * sum_{c in kb} x[i, c] * dec(q[j, c]) )
 * with fp32 accumulation.  dec(q) is exact in bf16; the scale multiplies the
 * fp32 partial sum of each 128-wide K block (it is never folded into a
 * rounded bf16 weight).
 *
 * Defined by: InfiniLM PR #586 (Summary: 128x128 block-FP8 W8A16 weights run
 * without materialising bf16 weights; decode routing by M); FreeToken PR #389
 * (the decode GEMV micro-benchmark over M = 1/8/16, and testing the op
 * against a linear on the dequantized weight); FreeToken PR #636 (the fp8
 * lm_head served by the block-FP8 GEMV).
 *
 *   x_bf16   device, m*k bf16, 2-byte aligned
 *   m        >= 0; m == 0 is a no-op returning FP8BS_OK
 *   codes    device, n*k bytes from fp8bs_quantize
 *   scales   device, fp32 [ceil(n/128), ceil(k/128)], 4-byte aligned
 *   n, k     > 0
 *   y_bf16   device, m*n bf16, written (must not overlap the inputs)
 * Shape-only dispatch (FP8BS_PATH_AUTO): m <= 32 -> decode kernel; larger m
 * -> tcgen05 prefill kernel; k % 16 != 0 or unaligned (non-16-byte) x/codes
 * -> generic kernel.
 */
int fp8bs_gemv(const void *x_bf16, int64_t m, const uint8_t *codes,
               const float *scales, int64_t n, int64_t k, void *y_bf16,
               void *stream);

/* fp8bs_gemv with an explicit kernel path (fp8bs_path).  A path that cannot
 * take the call (e.g. DECODE with k % 16 != 0) returns FP8BS_ERR_PATH. */
int fp8bs_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes,
                  const float *scales, int64_t n, int64_t k, void *y_bf16,
                  int path, void *stream);

/*
 * fp8bs_gemv_ws -- fp8bs_gemv with caller-provided device scratch, for the
 * decode path (m <= 32, k % 16 == 0, 16-byte aligned x and codes): a first
 * kernel writes an f16 copy of x with one power-of-two factor per (row,
 * 128-column K block) -- the largest |x| of the block moved into
 * [2^14, 2^15), every x within 2^-31 of it converting exactly -- into the
 * workspace, and the GEMV reads it in place of x: e4m3 codes then enter the
 * tensor cores as f16 (one conversion per code pair) at every m, where
 * fp8bs_gemv decodes to bf16 above m = 8.  The result obeys the same
 * definition and tolerance as fp8bs_gemv; the factor's inverse multiplies
 * each K block's fp32 partial together with the block scale.
 *
 * Defined by: InfiniLM PR #586 (Notes for Reviewers: 9 <= M <= 32 decode
 * batches on the tensor-core path) for the arithmetic, which is fp8bs_gemv's.
 *
 *   workspace        device, 16-byte aligned, >= fp8bs_gemv_ws_bytes(m, k)
 *                    bytes; its contents on entry do not matter, and it may
 *                    be reused once the call's work on `stream` is done
 *   other arguments  as fp8bs_gemv
 * Calls that do not take the decode path (m > 32: tensor-core prefill;
 * unaligned or k % 16 != 0: generic kernel) ignore the workspace.
 * FP8BS_ERR_NULL / FP8BS_ERR_ALIGN / FP8BS_ERR_SHAPE for a missing,
 * misaligned or too small workspace, before anything is launched.
 *
 * fp8bs_gemv_ws_bytes: bytes of workspace fp8bs_gemv_ws needs for m rows
 * of x with k columns (0 for m = 0), or FP8BS_ERR_SHAPE.  Host only.
 */
int64_t fp8bs_gemv_ws_bytes(int64_t m, int64_t k);
int fp8bs_gemv_ws(const void *x_bf16, int64_t m, const uint8_t *codes,
                  const float *scales, int64_t n, int64_t k, void *y_bf16,
                  void *workspace, int64_t workspace_bytes, void *stream);

/*
 * fp8bs_gemv_noalloc -- fp8bs_gemv_ws without a caller workspace, for
 * callers that cannot allocate device memory: a plugin whose host framework
 * owns all device memory through its own pool, a real-time loop that cannot
 * afford cudaMalloc / cudaFree (cudaFree synchronises the device), or a C
 * caller with nowhere to keep a buffer.  The scratch fp8bs_gemv_ws would
 * take from the caller (the f16 copy of x and its per-block factors) comes
 * from a fixed array of FP8BS_NOALLOC_SCRATCH_BYTES in the library's own
 * device memory; the call allocates and frees nothing.
 *
 * Defined by: no passage of the source pages has a counterpart; the
 * arithmetic and tolerance are fp8bs_gemv's (fp8bs_gemv_ws's).
 *
 *   arguments  as fp8bs_gemv (x, codes, scales, y are the caller's)
 *   returns    FP8BS_ERR_SHAPE, before anything is launched, when the
 *              decode path would need more scratch than the array holds:
 *              fp8bs_gemv_ws_bytes(m, k) > FP8BS_NOALLOC_SCRATCH_BYTES
 *              (2 MiB: m = 32 with k up to 32,256).  Calls that do not take
 *              the decode path (m > 32, unaligned, k % 16 != 0) need no
 *              scratch and run as fp8bs_gemv.
 * Every device that loads the library holds the array until the process
 * exits.  The first call on each device looks up the array's device address
 * once (cudaGetSymbolAddress, with that device current): make that first
 * call before any stream capture.  Every call shares the one array and
 * leaves its contents behind; each call writes all it reads, so nothing has
 * to be cleared, but calls that overlap on the GPU (different streams, no
 * ordering between them) race on it.  Calls on one stream are ordered.
 */
#define FP8BS_NOALLOC_SCRATCH_BYTES (2 * 1024 * 1024)
int fp8bs_gemv_noalloc(const void *x_bf16, int64_t m, const uint8_t *codes,
                       const float *scales, int64_t n, int64_t k, void *y_bf16,
                       void *stream);

/*
 * mxfp8_quantize -- load-time MXFP8 requantization: per row, per group of 32
 * consecutive k (the last group may be shorter), e = the smallest integer with
 * 448 * 2^e >= amax (i.e. 2^ceil(log2(amax/448))), E = clamp(e + 127, 0, 254)
 * (E = 127 when amax = 0), codes = e4m3(w * 2^(127 - E)) rounded to
 * nearest-even and saturated.
 *
 * Defined by: FreeToken issue #624 "Load-time MXFP8 requantization"
 * (Proposed solution: e4m3 codes with one e8m0 scale per 32 elements, ceil-log2
 * of amax/448, served by a W8A16 path).  This kernel streams bf16 straight to
 * codes; it needs no fp32 staging buffer.
 *
 *   w_bf16       device, n*k bf16, 2-byte aligned
 *   n, k         > 0
 *   codes_u8     device, n*k bytes, written
 *   scales_e8m0  device, n*ceil(k/32) bytes, written
 */
int mxfp8_quantize(const void *w_bf16, int64_t n, int64_t k,
                   uint8_t *codes_u8, uint8_t *scales_e8m0, void *stream);

/*
 * mxfp8_gemv -- W8A16 linear over MXFP8 weights:
 *   y[i, j] = bf16_rn( sum_g 2^(E[j,g]-127) * sum_{c in g} x[i, c] * dec(q[j, c]) )
 * Same argument rules and paths as fp8bs_gemv, with scales_e8m0
 * [n, ceil(k/32)].  Defined by: FreeToken issue #624 (the "mxfp8_linear
 * W8A16 path", which serves every batch size).
 * m > 32 runs on the tensor cores (PREFILL): each group's 2^(E-127) is
 * folded into the exact bf16 decode of its weights, which is exact for
 * every group with 3 <= E (amax >= 2^-116); groups with a smaller E have
 * their scaled weights rounded to bf16's subnormal grid (|error| <= 2^-134
 * per weight).
 */
int mxfp8_gemv(const void *x_bf16, int64_t m, const uint8_t *codes,
               const uint8_t *scales_e8m0, int64_t n, int64_t k, void *y_bf16,
               void *stream);

/* mxfp8_gemv with an explicit path (AUTO, DECODE, PREFILL or GENERIC). */
int mxfp8_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes,
                  const uint8_t *scales_e8m0, int64_t n, int64_t k,
                  void *y_bf16, int path, void *stream);

/*
 * fp8bs_gemv_batch / mxfp8_gemv_batch -- a sequence of W8A16 GEMVs with the
 * same m, e.g. the dense projections of every layer of a decode step:
 * the result is that of calling fp8bs_gemv (mxfp8_gemv) on ops[0],
 * ops[1], ..., ops[count-1] in that order on `stream`.
 *
 * Defined by: FreeToken PR #389 (Why: the decode micro-benchmark streams a
 * whole rotation of per-layer projection weights, 48 layers larger than L2,
 * at M = 1/8/16, and times the rotation, not one weight); InfiniLM PR #586
 * (Summary: block-FP8 W8A16 decode without bf16 weights) for the
 * arithmetic, which is fp8bs_gemv's (mxfp8_gemv's) exactly.
 *
 * Runs of consecutive ops that are independent (no op reads or writes the
 * bytes another op of the run writes) and fit the decode kernel (m <= 32,
 * k % 16 == 0, 16-byte aligned x and codes) go to one persistent launch of
 * up to 96 ops, which streams all their weights as one continuous sequence
 * of 128-row tiles instead of paying each GEMV's start-up and tail.  An op
 * that reads or writes an earlier op's output starts a new launch, so it
 * sees that output complete (stream order); ops that the decode kernel
 * cannot take run as their own fp8bs_gemv call in their place in the order.
 * A run too small to fill the GPU (fewer 128-row tiles than half its CTA
 * slots) runs as one launch per op.
 *
 *   ops      host array of count descriptors (read during the call only):
 *              x_bf16  device, m*k bf16      codes  device, n*k e4m3
 *              scales  device: fp32 [ceil(n/128), ceil(k/128)] (block) or
 *                      e8m0 uint8 [n, ceil(k/32)] (MXFP8)
 *              y_bf16  device, m*n bf16, written
 *              n, k    > 0
 *   count    >= 0 (0: no-op); m >= 0 (0: no-op), the same for every op
 * Every op is validated as fp8bs_gemv / mxfp8_gemv validates its arguments
 * before anything is enqueued; the first failure is returned and nothing
 * is launched.  The launches' parameters hold the ops (no device memory is
 * allocated or written besides y), so the call can be captured in a CUDA
 * graph.  _ex: path AUTO as above; DECODE runs every eligible run through the
 * batched kernel whatever its size (FP8BS_ERR_PATH if an op cannot take the
 * decode kernel); PREFILL / GENERIC run every op as fp8bs_gemv_ex
 * (mxfp8_gemv_ex) with that path.
 */
typedef struct fp8bs_gemv_op {
    const void *x_bf16;
    const uint8_t *codes;
    const void *scales;
    void *y_bf16;
    int64_t n, k;
} fp8bs_gemv_op;

int fp8bs_gemv_batch(const fp8bs_gemv_op *ops, int64_t count, int64_t m,
                     void *stream);
int fp8bs_gemv_batch_ex(const fp8bs_gemv_op *ops, int64_t count, int64_t m,
                        int path, void *stream);
int mxfp8_gemv_batch(const fp8bs_gemv_op *ops, int64_t count, int64_t m,
                     void *stream);
int mxfp8_gemv_batch_ex(const fp8bs_gemv_op *ops, int64_t count, int64_t m,
                        int path, void *stream);

/*
 * fp8row_quantize / fp8tensor_quantize -- load-time FP8 with one fp32 scale
 * per output row (scales_f32[n]) or one for the whole weight (scale_f32[1]).
 *
 * Defined by: FreeToken PR #389 "load-time per-tensor FP8 dense projections"
 * (What this adds: each weight quantized to e4m3 with one fp32 scale; Why:
 * the per-row W8A16 route in its decode table).  The scale rule is the tile
 * rule applied to a row / the tensor: amax over its elements, s = amax / 448
 * as an IEEE fp32 division, s = 1 when amax = 0, codes = e4m3(w / s) with an
 * IEEE fp32 quotient, nearest-even, saturated to +-448.
 *
 *   w_bf16      device, n*k bf16, 2-byte aligned
 *   n, k        > 0 (else FP8BS_ERR_SHAPE)
 *   codes_u8    device, n*k bytes, written
 *   scales_f32  device, n floats (per row) / 1 float (per tensor), 4-byte
 *               aligned, written.  The per-tensor form uses its one float as
 *               the amax accumulator before it writes s there, so no other
 *               work may read it until the call has completed on `stream`.
 * Asynchronous on `stream`; allocates nothing.
 */
int fp8row_quantize(const void *w_bf16, int64_t n, int64_t k,
                    uint8_t *codes_u8, float *scales_f32, void *stream);
int fp8tensor_quantize(const void *w_bf16, int64_t n, int64_t k,
                       uint8_t *codes_u8, float *scale_f32, void *stream);

/*
 * fp8row_gemv / fp8tensor_gemv -- W8A16 linear over per-row / per-tensor FP8:
 *   y[i, j] = bf16_rn( s_j * sum_c x[i, c] * dec(q[j, c]) )
 * with the sum in fp32 and s_j = scales[j] (per row) or scale[0] (per
 * tensor), applied once to the fp32 sum.  Same argument rules, paths and
 * errors as fp8bs_gemv, with the scale arrays of the quantizers above.
 * Defined by: FreeToken PR #389 (Why: the per-row W8A16 route of the decode
 * micro-benchmark over M = 1/8/16).
 */
int fp8row_gemv(const void *x_bf16, int64_t m, const uint8_t *codes,
                const float *scales, int64_t n, int64_t k, void *y_bf16,
                void *stream);
int fp8row_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes,
                   const float *scales, int64_t n, int64_t k, void *y_bf16,
                   int path, void *stream);
int fp8tensor_gemv(const void *x_bf16, int64_t m, const uint8_t *codes,
                   const float *scale, int64_t n, int64_t k, void *y_bf16,
                   void *stream);
int fp8tensor_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes,
                      const float *scale, int64_t n, int64_t k, void *y_bf16,
                      int path, void *stream);

/*
 * fp8bs_moe_gemv -- grouped block-FP8 W8A16 GEMV over routed experts:
 *   y[t, j, :] = x[t, :] . dequant(W[e])^T  with e = expert_ids[t, j],
 * each expert a block-FP8 weight [n, k] (fp8bs_quantize), the num_experts
 * weights stored back to back: codes [num_experts, n, k], scales
 * [num_experts, ceil(n/128), ceil(k/128)].  Every expert any token selected
 * is streamed once per call (whatever the number of its tokens); experts no
 * token selected are not read.  Same arithmetic and tolerance as fp8bs_gemv.
 *
 * Defined by: Atlas spark_model/weight_map/quantize_fp8_bs.rs (module
 * notes: the block-scaled quantizer exists for routed MoE experts; the
 * grouped MoE GEMM reads [N/128, K/128] fp32 block scales; decode reads the
 * top-12 of 256 experts per token).
 *
 *   x_bf16       device, m*k bf16, 16-byte aligned, k % 16 == 0
 *   expert_ids   device, m*topk int32; ids of one token must be distinct
 *                (a token listing an expert twice gets only its lowest such
 *                slot written and sets the device error word); an id
 *                outside [0, num_experts) selects nothing and sets the
 *                device error word (fp8bs_check_device_error)
 *   topk         1..num_experts;  num_experts 1..1024, num_experts*n < 2^31
 *   y_bf16       device, m*topk*n bf16, written for every valid id
 * The ids are read on the device (no host synchronisation); m > 32 runs in
 * chunks of 32 tokens.  FP8BS_ERR_PATH if k % 16 != 0 or x / codes are not
 * 16-byte aligned.
 */
int fp8bs_moe_gemv(const void *x_bf16, int64_t m, const int32_t *expert_ids,
                   int64_t topk, const uint8_t *codes, const float *scales,
                   int64_t num_experts, int64_t n, int64_t k, void *y_bf16,
                   void *stream);

/*
 * fp8bs_moe_gemv_ws -- fp8bs_moe_gemv with caller-provided device scratch,
 * for batches of m > 32 tokens: four small kernels group the (token, slot)
 * pairs by expert in the workspace (counts, prefix sums, the pairs expert by
 * expert, and a copy of each pair's x row in that order), then each selected
 * expert's weight is multiplied with exactly the x rows routed to it and
 * each output row written to its (token, slot).  With at most 32 pairs per
 * expert on average (m * topk <= 32 * num_experts) the decode kernel streams
 * each expert once per tile of up to 32 of its pairs, on an f16 copy of the
 * x rows with one power-of-two factor per (row, 128-column K block), as
 * fp8bs_gemv_ws prepares x (every x within 2^-31 of its block's largest
 * |x| converts exactly; the codes enter the tensor cores as f16); otherwise one grouped
 * GEMM on the 5th-generation tensor cores (the weight decoded to bf16 in
 * shared memory) runs tiles of up to 128 pairs of one expert (a deeper
 * pipeline) while the experts average at most 128 pairs, else of up to
 * 256.  Every
 * selected expert's weight is read once per tile of its pairs;
 * fp8bs_moe_gemv instead runs the decode kernel per 32 tokens, reading
 * every selected expert once per 32 tokens.
 * Same definition, arguments and tolerance as fp8bs_moe_gemv; m <= 32
 * takes fp8bs_moe_gemv's decode path and ignores the workspace.  In the
 * grouped path a token that lists an expert twice has both slots computed.
 *
 * Defined by: Atlas spark_model/weight_map/quantize_fp8_bs.rs (module
 * notes: the grouped MoE GEMM over block-FP8 routed experts with
 * [N/128, K/128] fp32 scales).
 *
 *   workspace        device, 256-byte aligned, >= fp8bs_moe_gemv_ws_bytes(m,
 *                    topk, num_experts, k) bytes (0 for m <= 32; about
 *                    2 * m * topk * k for the x copy, plus the factors);
 *                    contents on entry do not matter
 *   other arguments  as fp8bs_moe_gemv (m * topk < 2^31)
 * FP8BS_ERR_NULL / FP8BS_ERR_ALIGN / FP8BS_ERR_SHAPE for a missing,
 * misaligned or too small workspace, before anything is launched.
 */
int64_t fp8bs_moe_gemv_ws_bytes(int64_t m, int64_t topk, int64_t num_experts,
                                int64_t k);
int fp8bs_moe_gemv_ws(const void *x_bf16, int64_t m, const int32_t *expert_ids,
                      int64_t topk, const uint8_t *codes, const float *scales,
                      int64_t num_experts, int64_t n, int64_t k, void *y_bf16,
                      void *workspace, int64_t workspace_bytes, void *stream);

/*
 * FP8 E4M3 KV cache for paged decode attention.
 *
 * Defined by: InfiniLM PR #586 (Summary: an F8 cache with per-layer fp32
 * k_scale / v_scale for paged attention; Benchmark: split-KV decode
 * attention over the FP8 cache, "halves cache capacity and decode attention
 * read bandwidth").
 *
 * Cache layout: [num_blocks, page_size, num_kv_heads, head_dim] e4m3, token
 * i of sequence b in block block_table[b * max_blocks_per_seq +
 * i / page_size] at offset i % page_size.  head_dim must be 128, page_size a
 * multiple of 16, num_q_heads a multiple of num_kv_heads with at most 8
 * query heads per kv head.
 *
 * fp8kv_append: cache[slot_mapping[t]] = e4m3(x[t] / scale) for the new
 * tokens x [num_tokens, num_kv_heads, head_dim] bf16 (IEEE fp32 quotient,
 * nearest-even, saturating); slot = block * page_size + offset;
 * num_slots = num_blocks * page_size.  A slot outside [0, num_slots) is
 * skipped and sets the device error word.  x 16-byte aligned.
 */
int fp8kv_append(const void *x_bf16, int64_t num_tokens, int64_t num_kv_heads,
                 int64_t head_dim, const int32_t *slot_mapping,
                 const float *scale, uint8_t *cache, int64_t num_slots,
                 void *stream);

/*
 * fp8kv_decode_attention: one query token per sequence,
 *   o[b, h, :] = sum_l p_l * dec(V[l, g]) * v_scale,
 *   p = softmax_l( sm_scale * q[b, h, :] . dec(K[l, g]) * k_scale ),
 * g = h / (num_q_heads / num_kv_heads), over the seq_lens[b] tokens of
 * sequence b (0 tokens: o = 0).  K and V decode exactly; scores, the
 * softmax and the sums are fp32 (the weights enter the V sum as f16); one
 * bf16 rounding at the end.  The KV range of a sequence is split over a
 * thread-block cluster and merged on chip (no workspace).
 *
 *   q_bf16       device, [batch, num_q_heads, 128] bf16, 16-byte aligned
 *   k_cache, v_cache   device, e4m3 caches as above, 16-byte aligned
 *   k_scale, v_scale   device, 1 float each
 *   block_table  device, [batch, max_blocks_per_seq] int32
 *   seq_lens     device, [batch] int32, each <= max_blocks_per_seq * page_size
 *                (a larger or negative length is clamped and sets the device
 *                error word, as does a block id outside [0, num_blocks))
 *   max_seq_len  host upper bound of seq_lens (sizes the split), <=
 *                max_blocks_per_seq * page_size
 *   out_bf16     device, [batch, num_q_heads, 128] bf16, written
 */
int fp8kv_decode_attention(const void *q_bf16, const uint8_t *k_cache,
                           const uint8_t *v_cache, const float *k_scale,
                           const float *v_scale, const int32_t *block_table,
                           int64_t max_blocks_per_seq, const int32_t *seq_lens,
                           int64_t batch, int64_t num_q_heads,
                           int64_t num_kv_heads, int64_t head_dim,
                           int64_t page_size, int64_t num_blocks,
                           int64_t max_seq_len, float sm_scale, void *out_bf16,
                           void *stream);

/*
 * fp8act_quantize -- dynamic per-tensor activation quantization for the
 * W8A8 route: the per-tensor rule applied to x [m, k] (amax over all m*k
 * elements, s = amax / 448 in fp32, s = 1 if all zero, codes = e4m3(x / s)
 * with an IEEE fp32 quotient).  Up to 65536 elements run as one single-CTA
 * launch (amax and cast fused; the per-call cost dominates at decode sizes),
 * larger tensors as the grid-wide fp8tensor_quantize, bit for bit the same.
 *
 * Defined by: FreeToken PR #389 (What this adds: a dynamic per-tensor
 * activation scale, an amax pass then the cast; the follow-up commit: a
 * block-parallel partial amax plus a reduce and cast for large inputs).
 *
 *   x_bf16     device, m*k bf16
 *   codes_u8   device, m*k bytes, written
 *   scale_f32  device, 1 float, written (used as the amax accumulator by
 *              the grid-wide form, see fp8tensor_quantize)
 */
int fp8act_quantize(const void *x_bf16, int64_t m, int64_t k,
                    uint8_t *codes_u8, float *scale_f32, void *stream);

/*
 * w8a8_gemm -- W8A8 linear:
 *   y[i, j] = bf16_rn( sx * sw * sum_c dec(qx[i, c]) * dec(qw[j, c]) )
 * with e4m3 x e4m3 products (exact) summed in fp32 on the tensor cores.
 *
 * Defined by: FreeToken PR #389 (What this adds / Why: the per-tensor W8A8
 * GEMM of the projections, raw scaled-mm row of its decode table).
 *
 *   x_codes   device, m*k e4m3 (fp8act_quantize), 16-byte aligned for the
 *             TMA paths
 *   x_scale   device, 1 float
 *   w_codes   device, n*k e4m3 (fp8tensor_quantize), w_scale device, 1 float
 *   y_bf16    device, m*n bf16, written
 * Paths: m <= 32 -> DECODE (mma.sync e4m3, m > 32 in chunks of 32 rows);
 * larger m -> PREFILL (tcgen05 kind::f8f6f4); k % 16 != 0 or unaligned
 * codes -> GENERIC.  Errors as fp8bs_gemv.
 */
int w8a8_gemm(const uint8_t *x_codes, int64_t m, const float *x_scale,
              const uint8_t *w_codes, const float *w_scale, int64_t n,
              int64_t k, void *y_bf16, void *stream);
int w8a8_gemm_ex(const uint8_t *x_codes, int64_t m, const float *x_scale,
                 const uint8_t *w_codes, const float *w_scale, int64_t n,
                 int64_t k, void *y_bf16, int path, void *stream);

/* Path FP8BS_PATH_AUTO would take for these shapes and pointers
 * (host-only, launches nothing).  `mx` selects the MXFP8 GEMV; the block,
 * per-row and per-tensor GEMVs share the same paths (mx = 0). */
int fp8bs_select_path(int64_t m, int64_t n, int64_t k, const void *x_bf16,
                      const void *codes, int mx);

/* Human-readable text for a status code (static storage).
 * Defined by: no passage of the source pages (library infrastructure). */
const char *fp8bs_strerror(int status);

/*
 * Debug query: every wait inside the pipelined kernels is bounded; a kernel
 * that gives up sets a device-side error word instead of hanging.  This
 * synchronises `stream`, copies the word to *word_out (may be NULL), clears
 * it, and returns FP8BS_ERR_DEVICE if it was non-zero, else FP8BS_OK (or
 * FP8BS_ERR_CUDA if the synchronisation itself failed).
 *
 * Defined by: no passage of the source pages (library infrastructure: the
 * bounded waits' failure report).  Beyond a status, the call hands back the
 * word itself (word_out) so that a caller can tell a wait expiry
 * (bits 0-3) from a bad index argument (bit 4).
 */
int fp8bs_check_device_error(void *stream, uint32_t *word_out);

/*
 * Debug: exercise the give-up path of the bounded waits without a fault.
 * Launches one thread on `stream` that waits, with the same bounded wait the
 * pipelined kernels use, on a barrier nothing completes; after the bound
 * (about 2 s) it sets the FULL_WAIT bit (1) of the device error word and
 * returns, leaving the context usable.  Reads and writes no caller memory.
 * Returns FP8BS_OK once launched (FP8BS_ERR_CUDA if the launch failed);
 * fp8bs_check_device_error then reports FP8BS_ERR_DEVICE.
 *
 * Defined by: no passage of the source pages; this is the library's own
 * test hook for its failure detection.
 */
int fp8bs_debug_wait_expiry(void *stream);

/*
 * Debug: the e4m3 encode step that every quantizer here applies to its
 * fp32 quotients (round to nearest even, saturating to +-448, the sign kept
 * on zero results), run on consecutive binary32 bit patterns:
 * codes_u8[i] = e4m3(the float whose bits are first_bits + i), 0 <= i < count.
 *
 *   first_bits  first binary32 bit pattern
 *   count       > 0, a multiple of 4, first_bits + count <= 2^32
 *   codes_u8    device, count bytes, 4-byte aligned (written)
 *
 * Codes for NaN or Inf patterns are unspecified.  Asynchronous on `stream`.
 * Returns FP8BS_ERR_NULL, FP8BS_ERR_SHAPE or FP8BS_ERR_ALIGN before any
 * launch, FP8BS_ERR_CUDA if the launch failed.
 *
 * Defined by: the rounding of the block quantizer's codes (Atlas
 * spark_model/weight_map/quantize_fp8_bs.rs, one e4m3 byte per weight;
 * FreeToken PR #636, How it works: fp8 with a 128-block scale).  A test
 * hook so that the encode step can be compared with an independent encoder
 * over every finite binary32 value.
 */
int fp8bs_debug_encode_f32(uint32_t first_bits, int64_t count, uint8_t *codes_u8, void *stream);

/* ABI version (major * 100 + minor). */
int fp8bs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP8BS_H */
