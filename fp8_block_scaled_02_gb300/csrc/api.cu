// api.cu -- the C ABI (include/fp8bs.h): argument validation and shape-only
// dispatch to the kernels.  Nothing here allocates, synchronises (except the
// explicit debug query) or branches on tensor values.
#include "fp8bs.h"
#include "internal.h"

namespace {

using namespace fp8bs;

constexpr int64_t kDecodeMaxM = 32;   // rows of x per decode launch
constexpr int64_t kMaxDim = 1ll << 31;  // n, k and m must fit int32 for the kernels
// Grouped MoE: the largest average of pairs per expert that runs the GEMM on
// 128-pair tiles (beyond it, 256-pair tiles).  Measured on [2048, 4096]
// experts, top-12, same box: 48 pairs per expert 396 vs 450 us, 96: 229 vs
// 264 and 819 vs 954, 192: 787 vs 632, 384: 708 vs 608 (128 vs 256 pairs).
constexpr int64_t kMoeNarrowAvg = 128;

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8BS_OK : FP8BS_ERR_CUDA; }

// The TMA-staged kernels need 16-byte aligned x and codes with k % 16 == 0
// (TMA row pitch and base address rules).
inline bool tma_ok(int64_t k, const void *x, const void *codes) {
    return (k % 16) == 0 && aligned(x, 16) && aligned(codes, 16);
}

int select_path(int64_t m, int64_t k, const void *x, const void *codes, bool mx) {
    (void)mx;  // MXFP8 takes the same paths (its prefill folds the group scales into the decode)
    if (!tma_ok(k, x, codes)) return FP8BS_PATH_GENERIC;
    if (m <= kDecodeMaxM) return FP8BS_PATH_DECODE;
    return FP8BS_PATH_PREFILL;
}

int check_gemv_args(const void *x, int64_t m, const uint8_t *codes, const void *scales, int64_t n,
                    int64_t k, void *y, int path) {
    if (m < 0 || n <= 0 || k <= 0 || m >= kMaxDim || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (path < FP8BS_PATH_AUTO || path > FP8BS_PATH_GENERIC) return FP8BS_ERR_PATH;
    if (m == 0) return FP8BS_OK;
    if (!x || !codes || !scales || !y) return FP8BS_ERR_NULL;
    if (!aligned(x, 2) || !aligned(y, 2)) return FP8BS_ERR_ALIGN;
    return FP8BS_OK;
}

int run_decode_chunks(const DecodeArgs &a, cudaStream_t st) {
    for (int64_t m0 = 0; m0 < a.m; m0 += kDecodeMaxM) {
        DecodeArgs c = a;
        c.m = a.m - m0 < kDecodeMaxM ? a.m - m0 : kDecodeMaxM;
        c.x = static_cast<const char *>(a.x) + m0 * a.k * 2;
        c.y = static_cast<char *>(a.y) + m0 * a.n * 2;
        const cudaError_t e = launch_decode(c, st);
        if (e != cudaSuccess) return FP8BS_ERR_CUDA;
    }
    return FP8BS_OK;
}

int gemv_dispatch(const DecodeArgs &a, int path, cudaStream_t st) {
    const bool tma = tma_ok(a.k, a.x, a.codes);
    if (path == FP8BS_PATH_AUTO) path = select_path(a.m, a.k, a.x, a.codes, a.kind == kScaleMx);
    switch (path) {
        case FP8BS_PATH_GENERIC:
            return cuda_status(launch_generic_gemv(a, st));
        case FP8BS_PATH_DECODE:
            if (!tma) return FP8BS_ERR_PATH;
            return run_decode_chunks(a, st);
        case FP8BS_PATH_PREFILL: {
            if (!tma) return FP8BS_ERR_PATH;
            const cudaError_t e = launch_prefill(a, st);
            if (e == cudaErrorNotSupported) return run_decode_chunks(a, st);
            return cuda_status(e);
        }
        default:
            return FP8BS_ERR_PATH;
    }
}

// ------------------------------------------------------------ batches
struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
inline Range range_of(const void *p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}
inline bool overlap(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

// What one op of a batch reads and writes.
struct OpSpan {
    Range x, codes, scales, y;
};
OpSpan span_of(const fp8bs_gemv_op &o, int64_t m, bool mx) {
    const int64_t sb = mx ? o.n * ((o.k + 31) / 32) : 4 * ((o.n + 127) / 128) * ((o.k + 127) / 128);
    return OpSpan{range_of(o.x_bf16, 2 * m * o.k), range_of(o.codes, o.n * o.k), range_of(o.scales, sb),
                  range_of(o.y_bf16, 2 * m * o.n)};
}
// b must wait for a if b writes what a reads or writes, or reads what a writes
bool depends(const OpSpan &b, const OpSpan &a) {
    return overlap(b.y, a.x) || overlap(b.y, a.codes) || overlap(b.y, a.scales) || overlap(b.y, a.y) ||
           overlap(b.x, a.y) || overlap(b.codes, a.y) || overlap(b.scales, a.y);
}

int gemv_batch_impl(const fp8bs_gemv_op *ops, int64_t count, int64_t m, bool mx, int path, cudaStream_t st) {
    if (count < 0 || count >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (path < FP8BS_PATH_AUTO || path > FP8BS_PATH_GENERIC) return FP8BS_ERR_PATH;
    if (count == 0) return FP8BS_OK;
    if (!ops) return FP8BS_ERR_NULL;
    // validate everything before anything is enqueued
    for (int64_t i = 0; i < count; ++i) {
        const fp8bs_gemv_op &o = ops[i];
        const int s = check_gemv_args(o.x_bf16, m, o.codes, o.scales, o.n, o.k, o.y_bf16, path);
        if (s != FP8BS_OK) return s;
        if (m == 0) continue;
        if (!mx && !aligned(o.scales, 4)) return FP8BS_ERR_ALIGN;
        const bool tma = tma_ok(o.k, o.x_bf16, o.codes);
        if ((path == FP8BS_PATH_DECODE || path == FP8BS_PATH_PREFILL) && !tma) return FP8BS_ERR_PATH;
    }
    if (m == 0) return FP8BS_OK;
    const ScaleKind kind = mx ? kScaleMx : kScaleBlock;
    const bool batchable_path = path == FP8BS_PATH_AUTO || path == FP8BS_PATH_DECODE;
    BatchItem run[kBatchMaxOps];
    OpSpan spans[kBatchMaxOps];
    int nrun = 0;
    auto flush = [&]() -> int {
        if (nrun == 0) return FP8BS_OK;
        const cudaError_t e = launch_decode_batch(run, nrun, m, kind, path == FP8BS_PATH_DECODE, st);
        nrun = 0;
        return cuda_status(e);
    };
    for (int64_t i = 0; i < count; ++i) {
        const fp8bs_gemv_op &o = ops[i];
        const bool eligible = batchable_path && m <= kDecodeMaxM && tma_ok(o.k, o.x_bf16, o.codes);
        if (!eligible) {
            int s = flush();
            if (s != FP8BS_OK) return s;
            const DecodeArgs a{o.x_bf16, o.codes, mx ? nullptr : static_cast<const float *>(o.scales),
                               mx ? static_cast<const uint8_t *>(o.scales) : nullptr, o.y_bf16, m, o.n, o.k, kind, 0};
            s = gemv_dispatch(a, path, st);
            if (s != FP8BS_OK) return s;
            continue;
        }
        const OpSpan sp = span_of(o, m, mx);
        bool dep = nrun == kBatchMaxOps;
        for (int j = 0; j < nrun && !dep; ++j) dep = depends(sp, spans[j]);
        if (dep) {
            const int s = flush();
            if (s != FP8BS_OK) return s;
        }
        run[nrun] = BatchItem{o.x_bf16, o.codes, o.scales, o.y_bf16, o.n, o.k};
        spans[nrun] = sp;
        ++nrun;
    }
    return flush();
}

int run_w8a8_decode_chunks(const W8A8Args &a, cudaStream_t st) {
    for (int64_t m0 = 0; m0 < a.m; m0 += kDecodeMaxM) {
        W8A8Args c = a;
        c.m = a.m - m0 < kDecodeMaxM ? a.m - m0 : kDecodeMaxM;
        c.xq = a.xq + m0 * a.k;
        c.y = static_cast<char *>(a.y) + m0 * a.n * 2;
        if (launch_w8a8_decode(c, st) != cudaSuccess) return FP8BS_ERR_CUDA;
    }
    return FP8BS_OK;
}

}  // namespace

extern "C" {

int fp8bs_version(void) { return 106; }

const char *fp8bs_strerror(int status) {
    switch (status) {
        case FP8BS_OK: return "ok";
        case FP8BS_ERR_NULL: return "a required pointer is NULL";
        case FP8BS_ERR_SHAPE: return "shape out of range (need n > 0, k > 0, m >= 0, all < 2^31)";
        case FP8BS_ERR_BLOCK: return "unsupported block size (only 128 is supported)";
        case FP8BS_ERR_ALIGN: return "pointer not aligned to its element size";
        case FP8BS_ERR_CUDA: return "CUDA call or kernel launch failed";
        case FP8BS_ERR_DEVICE: return "a kernel gave up a bounded wait (device error word set)";
        case FP8BS_ERR_PATH: return "the requested kernel path cannot take this call";
        default: return "unknown status";
    }
}

int fp8bs_quantize(const void *w_bf16, int64_t n, int64_t k, int block, uint8_t *codes_u8, float *scales_f32,
                   void *stream) {
    if (n <= 0 || k <= 0 || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (block != 128) return FP8BS_ERR_BLOCK;
    if (!w_bf16 || !codes_u8 || !scales_f32) return FP8BS_ERR_NULL;
    if (!aligned(w_bf16, 2) || !aligned(scales_f32, 4)) return FP8BS_ERR_ALIGN;
    const bool vec = (k % 8) == 0 && aligned(w_bf16, 16) && aligned(codes_u8, 8);
    return cuda_status(
        launch_block_quantize(w_bf16, n, k, codes_u8, scales_f32, vec, static_cast<cudaStream_t>(stream)));
}

int mxfp8_quantize(const void *w_bf16, int64_t n, int64_t k, uint8_t *codes_u8, uint8_t *scales_e8m0,
                   void *stream) {
    if (n <= 0 || k <= 0 || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (!w_bf16 || !codes_u8 || !scales_e8m0) return FP8BS_ERR_NULL;
    if (!aligned(w_bf16, 2)) return FP8BS_ERR_ALIGN;
    const bool vec = (k % 8) == 0 && aligned(w_bf16, 16) && aligned(codes_u8, 8);
    return cuda_status(
        launch_mx_quantize(w_bf16, n, k, codes_u8, scales_e8m0, vec, static_cast<cudaStream_t>(stream)));
}

int fp8bs_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales, int64_t n,
                  int64_t k, void *y_bf16, int path, void *stream) {
    int st = check_gemv_args(x_bf16, m, codes, scales, n, k, y_bf16, path);
    if (st != FP8BS_OK || m == 0) return st;
    if (!aligned(scales, 4)) return FP8BS_ERR_ALIGN;
    DecodeArgs a{x_bf16, codes, scales, nullptr, y_bf16, m, n, k, kScaleBlock, 0};
    return gemv_dispatch(a, path, static_cast<cudaStream_t>(stream));
}

int fp8bs_gemv(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales, int64_t n, int64_t k,
               void *y_bf16, void *stream) {
    return fp8bs_gemv_ex(x_bf16, m, codes, scales, n, k, y_bf16, FP8BS_PATH_AUTO, stream);
}

int64_t fp8bs_gemv_ws_bytes(int64_t m, int64_t k) {
    if (m < 0 || k <= 0 || m >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    return m == 0 ? 0 : xprep_bytes(m < kDecodeMaxM ? m : kDecodeMaxM, k);
}

int fp8bs_gemv_ws(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales, int64_t n, int64_t k,
                  void *y_bf16, void *workspace, int64_t workspace_bytes, void *stream) {
    int st = check_gemv_args(x_bf16, m, codes, scales, n, k, y_bf16, FP8BS_PATH_AUTO);
    if (st != FP8BS_OK || m == 0) return st;
    if (!aligned(scales, 4)) return FP8BS_ERR_ALIGN;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    DecodeArgs a{x_bf16, codes, scales, nullptr, y_bf16, m, n, k, kScaleBlock, 0};
    // only the decode path (m <= 32, TMA-eligible) uses the workspace
    if (select_path(m, k, x_bf16, codes, false) != FP8BS_PATH_DECODE) return gemv_dispatch(a, FP8BS_PATH_AUTO, s);
    if (!workspace) return FP8BS_ERR_NULL;
    if (!aligned(workspace, 16)) return FP8BS_ERR_ALIGN;
    if (workspace_bytes < xprep_bytes(m, k)) return FP8BS_ERR_SHAPE;
    return cuda_status(launch_decode_xprep(a, workspace, s));
}

int mxfp8_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes, const uint8_t *scales_e8m0, int64_t n,
                  int64_t k, void *y_bf16, int path, void *stream) {
    int st = check_gemv_args(x_bf16, m, codes, scales_e8m0, n, k, y_bf16, path);
    if (st != FP8BS_OK || m == 0) return st;
    DecodeArgs a{x_bf16, codes, nullptr, scales_e8m0, y_bf16, m, n, k, kScaleMx, 0};
    return gemv_dispatch(a, path, static_cast<cudaStream_t>(stream));
}

int mxfp8_gemv(const void *x_bf16, int64_t m, const uint8_t *codes, const uint8_t *scales_e8m0, int64_t n,
               int64_t k, void *y_bf16, void *stream) {
    return mxfp8_gemv_ex(x_bf16, m, codes, scales_e8m0, n, k, y_bf16, FP8BS_PATH_AUTO, stream);
}

int fp8bs_gemv_batch_ex(const fp8bs_gemv_op *ops, int64_t count, int64_t m, int path, void *stream) {
    return gemv_batch_impl(ops, count, m, false, path, static_cast<cudaStream_t>(stream));
}

int fp8bs_gemv_batch(const fp8bs_gemv_op *ops, int64_t count, int64_t m, void *stream) {
    return gemv_batch_impl(ops, count, m, false, FP8BS_PATH_AUTO, static_cast<cudaStream_t>(stream));
}

int mxfp8_gemv_batch_ex(const fp8bs_gemv_op *ops, int64_t count, int64_t m, int path, void *stream) {
    return gemv_batch_impl(ops, count, m, true, path, static_cast<cudaStream_t>(stream));
}

int mxfp8_gemv_batch(const fp8bs_gemv_op *ops, int64_t count, int64_t m, void *stream) {
    return gemv_batch_impl(ops, count, m, true, FP8BS_PATH_AUTO, static_cast<cudaStream_t>(stream));
}

static int rowwise_quantize(const void *w_bf16, int64_t n, int64_t k, uint8_t *codes_u8, float *scales_f32,
                            bool per_tensor, void *stream) {
    if (n <= 0 || k <= 0 || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (!w_bf16 || !codes_u8 || !scales_f32) return FP8BS_ERR_NULL;
    if (!aligned(w_bf16, 2) || !aligned(scales_f32, 4)) return FP8BS_ERR_ALIGN;
    const bool vec = (k % 8) == 0 && aligned(w_bf16, 16) && aligned(codes_u8, 8);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(per_tensor ? launch_tensor_quantize(w_bf16, n, k, codes_u8, scales_f32, vec, st)
                                  : launch_row_quantize(w_bf16, n, k, codes_u8, scales_f32, vec, st));
}

int fp8row_quantize(const void *w_bf16, int64_t n, int64_t k, uint8_t *codes_u8, float *scales_f32, void *stream) {
    return rowwise_quantize(w_bf16, n, k, codes_u8, scales_f32, false, stream);
}

int fp8tensor_quantize(const void *w_bf16, int64_t n, int64_t k, uint8_t *codes_u8, float *scale_f32,
                       void *stream) {
    return rowwise_quantize(w_bf16, n, k, codes_u8, scale_f32, true, stream);
}

static int rowwise_gemv(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales, int64_t n,
                        int64_t k, void *y_bf16, int row_stride, int path, void *stream) {
    int st = check_gemv_args(x_bf16, m, codes, scales, n, k, y_bf16, path);
    if (st != FP8BS_OK || m == 0) return st;
    if (!aligned(scales, 4)) return FP8BS_ERR_ALIGN;
    DecodeArgs a{x_bf16, codes, scales, nullptr, y_bf16, m, n, k, kScaleRow, row_stride};
    return gemv_dispatch(a, path, static_cast<cudaStream_t>(stream));
}

int fp8row_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales, int64_t n, int64_t k,
                   void *y_bf16, int path, void *stream) {
    return rowwise_gemv(x_bf16, m, codes, scales, n, k, y_bf16, 1, path, stream);
}

int fp8row_gemv(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales, int64_t n, int64_t k,
                void *y_bf16, void *stream) {
    return rowwise_gemv(x_bf16, m, codes, scales, n, k, y_bf16, 1, FP8BS_PATH_AUTO, stream);
}

int fp8tensor_gemv_ex(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scale, int64_t n,
                      int64_t k, void *y_bf16, int path, void *stream) {
    return rowwise_gemv(x_bf16, m, codes, scale, n, k, y_bf16, 0, path, stream);
}

int fp8tensor_gemv(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scale, int64_t n, int64_t k,
                   void *y_bf16, void *stream) {
    return rowwise_gemv(x_bf16, m, codes, scale, n, k, y_bf16, 0, FP8BS_PATH_AUTO, stream);
}

static int moe_check(const void *x_bf16, int64_t m, const int32_t *expert_ids, int64_t topk, const uint8_t *codes,
                     const float *scales, int64_t num_experts, int64_t n, int64_t k, void *y_bf16) {
    if (m < 0 || n <= 0 || k <= 0 || m >= kMaxDim || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (topk < 1 || num_experts < 1 || num_experts > 1024 || topk > num_experts) return FP8BS_ERR_SHAPE;
    if (num_experts * n >= kMaxDim || m * topk >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (m == 0) return FP8BS_OK;
    if (!x_bf16 || !expert_ids || !codes || !scales || !y_bf16) return FP8BS_ERR_NULL;
    if (!aligned(x_bf16, 2) || !aligned(y_bf16, 2) || !aligned(scales, 4) || !aligned(expert_ids, 4))
        return FP8BS_ERR_ALIGN;
    if (!tma_ok(k, x_bf16, codes)) return FP8BS_ERR_PATH;
    return FP8BS_OK;
}

static int moe_decode_chunks(const void *x_bf16, int64_t m, const int32_t *expert_ids, int64_t topk,
                             const uint8_t *codes, const float *scales, int64_t num_experts, int64_t n, int64_t k,
                             void *y_bf16, cudaStream_t st) {
    for (int64_t m0 = 0; m0 < m; m0 += kDecodeMaxM) {
        const int64_t mc = m - m0 < kDecodeMaxM ? m - m0 : kDecodeMaxM;
        DecodeArgs a{static_cast<const char *>(x_bf16) + m0 * k * 2, codes, scales, nullptr,
                     static_cast<char *>(y_bf16) + m0 * topk * n * 2, mc, n, k, kScaleBlock, 0};
        const MoeArgs g{expert_ids + m0 * topk, topk, num_experts};
        if (launch_moe_decode(a, g, st) != cudaSuccess) return FP8BS_ERR_CUDA;
    }
    return FP8BS_OK;
}

int fp8bs_moe_gemv(const void *x_bf16, int64_t m, const int32_t *expert_ids, int64_t topk, const uint8_t *codes,
                   const float *scales, int64_t num_experts, int64_t n, int64_t k, void *y_bf16, void *stream) {
    const int s = moe_check(x_bf16, m, expert_ids, topk, codes, scales, num_experts, n, k, y_bf16);
    if (s != FP8BS_OK || m == 0) return s;
    return moe_decode_chunks(x_bf16, m, expert_ids, topk, codes, scales, num_experts, n, k, y_bf16,
                             static_cast<cudaStream_t>(stream));
}

int64_t fp8bs_moe_gemv_ws_bytes(int64_t m, int64_t topk, int64_t num_experts, int64_t k) {
    if (m < 0 || topk < 1 || num_experts < 1 || num_experts > 1024 || m >= kMaxDim || m * topk >= kMaxDim ||
        k <= 0 || k >= kMaxDim)
        return FP8BS_ERR_SHAPE;
    return m <= kDecodeMaxM ? 0 : moe_route_bytes(m * topk, num_experts, k);
}

int fp8bs_moe_gemv_ws(const void *x_bf16, int64_t m, const int32_t *expert_ids, int64_t topk, const uint8_t *codes,
                      const float *scales, int64_t num_experts, int64_t n, int64_t k, void *y_bf16, void *workspace,
                      int64_t workspace_bytes, void *stream) {
    const int s = moe_check(x_bf16, m, expert_ids, topk, codes, scales, num_experts, n, k, y_bf16);
    if (s != FP8BS_OK || m == 0) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (m <= kDecodeMaxM)
        return moe_decode_chunks(x_bf16, m, expert_ids, topk, codes, scales, num_experts, n, k, y_bf16, st);
    if (!workspace) return FP8BS_ERR_NULL;
    if (!aligned(workspace, 256)) return FP8BS_ERR_ALIGN;
    if (workspace_bytes < moe_route_bytes(m * topk, num_experts, k)) return FP8BS_ERR_SHAPE;
    MoeRoute r = moe_route_views(workspace, m * topk, num_experts, k);
    // GEMM tiles of 128 pairs (a deeper pipeline) while the experts average
    // at most kMoeNarrowAvg pairs, else of 256
    r.gemm_tile = m * topk <= kMoeNarrowAvg * num_experts ? kMoeGemmTileNarrow : kMoeGemmTileWide;
    // few pairs per expert on average: stream each selected expert once per
    // tile of 32 of its pairs at GEMV speed (x copied as f16 operands); more:
    // the tensor-core GEMM (x copied as bf16)
    const bool decode_tiles = m * topk <= kMoeDecodeTile * num_experts;
    cudaError_t e = launch_moe_route(x_bf16, k, expert_ids, m * topk, static_cast<int>(topk),
                                     static_cast<int>(num_experts), r, decode_tiles, st);
    if (e != cudaSuccess) return FP8BS_ERR_CUDA;
    const DecodeArgs a{x_bf16, codes, scales, nullptr, y_bf16, m, n, k, kScaleBlock, 0};
    const MoeArgs g{expert_ids, topk, num_experts};
    if (decode_tiles) return cuda_status(launch_moe_grouped(a, g, r, st));
    e = launch_prefill_moe(a, g, r, st);
    if (e == cudaErrorNotSupported)
        return moe_decode_chunks(x_bf16, m, expert_ids, topk, codes, scales, num_experts, n, k, y_bf16, st);
    return cuda_status(e);
}

int fp8kv_append(const void *x_bf16, int64_t num_tokens, int64_t num_kv_heads, int64_t head_dim,
                 const int32_t *slot_mapping, const float *scale, uint8_t *cache, int64_t num_slots, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || num_slots <= 0 || num_tokens >= kMaxDim || num_kv_heads >= 4096)
        return FP8BS_ERR_SHAPE;
    if (head_dim != 128) return FP8BS_ERR_SHAPE;
    if (num_slots * num_kv_heads * head_dim >= (int64_t{1} << 40)) return FP8BS_ERR_SHAPE;
    if (num_tokens == 0) return FP8BS_OK;
    if (!x_bf16 || !slot_mapping || !scale || !cache) return FP8BS_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(cache, 8) || !aligned(slot_mapping, 4) || !aligned(scale, 4))
        return FP8BS_ERR_ALIGN;
    return cuda_status(launch_kv_append(x_bf16, num_tokens, num_kv_heads, slot_mapping, scale, cache, num_slots,
                                        static_cast<cudaStream_t>(stream)));
}

int fp8kv_decode_attention(const void *q_bf16, const uint8_t *k_cache, const uint8_t *v_cache, const float *k_scale,
                           const float *v_scale, const int32_t *block_table, int64_t max_blocks_per_seq,
                           const int32_t *seq_lens, int64_t batch, int64_t num_q_heads, int64_t num_kv_heads,
                           int64_t head_dim, int64_t page_size, int64_t num_blocks, int64_t max_seq_len, float sm_scale,
                           void *out_bf16, void *stream) {
    if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return FP8BS_ERR_SHAPE;
    if (head_dim != 128 || num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 8) return FP8BS_ERR_SHAPE;
    if (page_size < 16 || page_size % 16 != 0 || page_size > 4096) return FP8BS_ERR_SHAPE;
    if (num_blocks * page_size >= kMaxDim || batch * num_kv_heads >= kMaxDim || max_blocks_per_seq >= kMaxDim)
        return FP8BS_ERR_SHAPE;
    if (max_seq_len < 0 || max_seq_len > max_blocks_per_seq * page_size) return FP8BS_ERR_SHAPE;
    if (!(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f) return FP8BS_ERR_SHAPE;
    if (batch == 0) return FP8BS_OK;
    if (!q_bf16 || !k_cache || !v_cache || !k_scale || !v_scale || !block_table || !seq_lens || !out_bf16)
        return FP8BS_ERR_NULL;
    if (!aligned(q_bf16, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out_bf16, 2) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return FP8BS_ERR_ALIGN;
    KvAttnArgs a{q_bf16, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out_bf16,
                 batch, num_q_heads, num_kv_heads, page_size, num_blocks, max_blocks_per_seq, max_seq_len, sm_scale};
    return cuda_status(launch_kv_attention(a, static_cast<cudaStream_t>(stream)));
}

int fp8act_quantize(const void *x_bf16, int64_t m, int64_t k, uint8_t *codes_u8, float *scale_f32, void *stream) {
    if (m <= 0 || k <= 0 || m >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (!x_bf16 || !codes_u8 || !scale_f32) return FP8BS_ERR_NULL;
    if (!aligned(x_bf16, 2) || !aligned(scale_f32, 4)) return FP8BS_ERR_ALIGN;
    const bool vec = (k % 8) == 0 && aligned(x_bf16, 16) && aligned(codes_u8, 8);
    return cuda_status(launch_act_quantize(x_bf16, m, k, codes_u8, scale_f32, vec, static_cast<cudaStream_t>(stream)));
}

int w8a8_gemm_ex(const uint8_t *x_codes, int64_t m, const float *x_scale, const uint8_t *w_codes,
                 const float *w_scale, int64_t n, int64_t k, void *y_bf16, int path, void *stream) {
    if (m < 0 || n <= 0 || k <= 0 || m >= kMaxDim || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (path < FP8BS_PATH_AUTO || path > FP8BS_PATH_GENERIC) return FP8BS_ERR_PATH;
    if (m == 0) return FP8BS_OK;
    if (!x_codes || !x_scale || !w_codes || !w_scale || !y_bf16) return FP8BS_ERR_NULL;
    if (!aligned(x_scale, 4) || !aligned(w_scale, 4) || !aligned(y_bf16, 2)) return FP8BS_ERR_ALIGN;
    const bool tma = tma_ok(k, x_codes, w_codes);
    if (path == FP8BS_PATH_AUTO) path = !tma ? FP8BS_PATH_GENERIC : (m <= kDecodeMaxM ? FP8BS_PATH_DECODE : FP8BS_PATH_PREFILL);
    const W8A8Args a{x_codes, x_scale, w_codes, w_scale, y_bf16, m, n, k};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (path) {
        case FP8BS_PATH_GENERIC: return cuda_status(launch_w8a8_generic(a, st));
        case FP8BS_PATH_DECODE: return tma ? run_w8a8_decode_chunks(a, st) : FP8BS_ERR_PATH;
        case FP8BS_PATH_PREFILL: return tma ? cuda_status(launch_w8a8_prefill(a, st)) : FP8BS_ERR_PATH;
        default: return FP8BS_ERR_PATH;
    }
}

int w8a8_gemm(const uint8_t *x_codes, int64_t m, const float *x_scale, const uint8_t *w_codes, const float *w_scale,
              int64_t n, int64_t k, void *y_bf16, void *stream) {
    return w8a8_gemm_ex(x_codes, m, x_scale, w_codes, w_scale, n, k, y_bf16, FP8BS_PATH_AUTO, stream);
}

int fp8bs_select_path(int64_t m, int64_t n, int64_t k, const void *x_bf16, const void *codes, int mx) {
    (void)n;
    if (m <= 0 || k <= 0) return FP8BS_ERR_SHAPE;
    return select_path(m, k, x_bf16, codes, mx != 0);
}

int fp8bs_debug_wait_expiry(void *stream) {
    return cuda_status(launch_wait_expiry_probe(static_cast<cudaStream_t>(stream)));
}

int fp8bs_debug_encode_f32(uint32_t first_bits, int64_t count, uint8_t *codes_u8, void *stream) {
    if (!codes_u8) return FP8BS_ERR_NULL;
    if (count <= 0 || count % 4 != 0 || static_cast<uint64_t>(first_bits) + static_cast<uint64_t>(count) > (1ull << 32))
        return FP8BS_ERR_SHAPE;
    if (!aligned(codes_u8, 4)) return FP8BS_ERR_ALIGN;
    return cuda_status(launch_encode_probe(first_bits, count, codes_u8, static_cast<cudaStream_t>(stream)));
}

int fp8bs_check_device_error(void *stream, uint32_t *word_out) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8BS_ERR_CUDA;
    const uint32_t w = take_decode_error() | take_prefill_error() | take_w8a8_error() | take_kv_error() |
                       take_moe_error();
    if (word_out) *word_out = w;
    return w ? FP8BS_ERR_DEVICE : FP8BS_OK;
}

}  // extern "C"
