// internal.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8bs {

// quantize.cu
cudaError_t launch_block_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                                  float *scales, bool vector_ok, cudaStream_t stream);
cudaError_t launch_mx_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                               uint8_t *e8m0, bool vector_ok, cudaStream_t stream);
// one fp32 scale per row (scales[n]) or per tensor (scales[1]); the
// per-tensor form zeroes scales[0] and accumulates the amax there first.
cudaError_t launch_row_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                                float *scales, bool vector_ok, cudaStream_t stream);
cudaError_t launch_tensor_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                                   float *scale, bool vector_ok, cudaStream_t stream);
// dynamic per-tensor activation quantization (the per-tensor rule); up to
// kActSmall elements in one single-CTA launch, larger tensors grid-wide
constexpr int64_t kActSmall = 65536;
cudaError_t launch_act_quantize(const void *x, int64_t m, int64_t k, uint8_t *codes, float *scale,
                                bool vector_ok, cudaStream_t stream);

// How the weight's scales are laid out.
enum ScaleKind : int {
    kScaleBlock = 0,  // fp32 [ceil(n/128), ceil(k/128)], one per 128x128 tile
    kScaleMx = 1,     // e8m0 [n, ceil(k/32)], one per 32 consecutive k of a row
    kScaleRow = 2,    // fp32 scales[r * row_stride]: per row (stride 1) or per tensor (stride 0)
};

// decode.cu -- TMA-staged skinny GEMM, m <= 32 per launch.
struct DecodeArgs {
    const void *x;           // bf16 [m, k] (row offset already applied)
    const uint8_t *codes;    // e4m3 [n, k]
    const float *scales;     // block or row scales (kScaleBlock / kScaleRow), else nullptr
    const uint8_t *e8m0;     // MX exponents [n, ceil(k/32)] (kScaleMx), else nullptr
    void *y;                 // bf16 [m, n] (row offset already applied)
    int64_t m, n, k;
    ScaleKind kind;
    int row_stride;          // kScaleRow: 1 per row, 0 per tensor
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
// Block-scaled decode (m <= 32) with x prepared once per call: an f16 copy
// of x with one power-of-two factor per (row, 128-column K block) is written
// to the caller's workspace by a first kernel and read by every CTA of the
// decode kernel in place of bf16 x (f16 weight decode at every m, no
// converter warp).  Workspace: xprep_bytes(m, k) bytes, 16-byte aligned.
int64_t xprep_bytes(int64_t m, int64_t k);
cudaError_t launch_decode_xprep(const DecodeArgs &a, void *workspace, cudaStream_t stream);
// Grouped MoE: a.codes / a.scales hold num_experts block-FP8 weights of
// [a.n, a.k] back to back; ids [a.m, topk]; a.y is [a.m, topk, a.n].
struct MoeArgs {
    const int32_t *ids;
    int64_t topk, num_experts;
};
cudaError_t launch_moe_decode(const DecodeArgs &a, const MoeArgs &g, cudaStream_t stream);
// A batch of GEMVs with one m <= 32, every op TMA-eligible (k % 16 == 0,
// 16-byte aligned x and codes) and none reading or writing another's output:
// one persistent launch streams all their weights (decode.cu).  count <=
// kBatchMaxOps.  Unless `force`, a batch too small to fill the GPU's CTA
// slots runs as one launch per op instead.
constexpr int kBatchMaxOps = 96;
struct BatchItem {
    const void *x;           // bf16 [m, k] (f16, prepared, when xinv is set)
    const uint8_t *codes;    // e4m3 [n, k]
    const void *scales;      // fp32 block scales (kScaleBlock) or e8m0 exponents (kScaleMx)
    void *y;                 // bf16 [m, n]
    int64_t n, k;
    const float *xinv = nullptr;  // prepared x: inverse factors [ceil(k/128)][32]
};
cudaError_t launch_decode_batch(const BatchItem *ops, int count, int64_t m, ScaleKind kind, bool force,
                                cudaStream_t stream);
uint32_t take_decode_error();  // reads and clears the decode kernels' error word
// one thread waits on a barrier nothing completes until the bounded wait
// gives up (about 2 s), then sets the decode error word
cudaError_t launch_wait_expiry_probe(cudaStream_t stream);
cudaError_t launch_encode_probe(uint32_t first, int64_t count, uint8_t *codes, cudaStream_t stream);

// moe.cu -- the routing of the grouped MoE GEMM: the (token, slot) pairs of
// ids [pairs] grouped by expert and their x rows copied in that order, built
// on the device in a caller workspace of moe_route_bytes(pairs, E, k) bytes.
// Pairs per expert tile of the grouped decode path (the decode kernel's x rows).
constexpr int kMoeDecodeTile = 32;
// Pairs per tile of the tensor-core grouped GEMM (prefill.cu, MOE form):
// 128 (deeper pipeline) while the experts average few enough pairs, else 256.
constexpr int kMoeGemmTileNarrow = 128, kMoeGemmTileWide = 256;
struct MoeRoute {
    int32_t *counts;    // [E] pairs per expert
    int32_t *cursor;    // [E] scatter cursors
    int32_t *tok_off;   // [E + 1] first pair of each expert in perm
    int32_t *tile_off;  // [E + 1] first GEMM tile (gemm_tile pairs) of each expert
    int32_t *tile_off_dec;  // [E + 1] first kMoeDecodeTile-pair tile of each expert (decode path)
    int4 *tile_info;        // [GEMM tile bound] {expert, first pair, pairs, 0} of each GEMM tile
    int4 *tile_info_dec;    // [decode tile bound] the same for the kMoeDecodeTile-pair tiles
    int32_t *perm;      // [pairs] t * topk + j, expert by expert
    float *xinv;        // decode tiles: [tile bound][kblocks][32] f16 inverse factors, slot order
    void *xs;           // [pairs, k]: x[perm[q] / topk] in perm's order; bf16 for the
                        // tensor-core GEMM, f16 rescaled per (row, K block) for decode tiles
    int gemm_tile;      // pairs per GEMM tile of this routing (kMoeGemmTileNarrow / Wide)
};
// Upper bound on the kMoeDecodeTile-pair tiles of `pairs` routed pairs:
// one partial tile per expert at most, besides the full ones.
inline int64_t moe_decode_tile_bound(int64_t pairs, int64_t num_experts) {
    return (pairs + kMoeDecodeTile - 1) / kMoeDecodeTile + (num_experts < pairs ? num_experts : pairs);
}
// ... and on the `tile`-pair tiles of the tensor-core grouped GEMM.
inline int64_t moe_gemm_tile_bound(int64_t pairs, int64_t num_experts, int tile) {
    return (pairs + tile - 1) / tile + (num_experts < pairs ? num_experts : pairs);
}
int64_t moe_route_bytes(int64_t pairs, int64_t num_experts, int64_t k);
MoeRoute moe_route_views(void *workspace, int64_t pairs, int64_t num_experts, int64_t k);
// decode_tiles: write xs as f16 with the per-(row, K block) inverse factors
// of each decode tile in xinv (the decode kernel's operands); else bf16.
// The GEMM tiles are of r.gemm_tile pairs.
cudaError_t launch_moe_route(const void *x, int64_t k, const int32_t *ids, int64_t pairs, int topk,
                             int num_experts, const MoeRoute &r, bool decode_tiles, cudaStream_t stream);
uint32_t take_moe_error();
// decode.cu: the grouped MoE GEMV by the routing's kMoeDecodeTile-pair expert
// tiles (f16 x rows from r.xs, routed with decode_tiles set).
cudaError_t launch_moe_grouped(const DecodeArgs &a, const MoeArgs &g, const MoeRoute &r, cudaStream_t stream);

// generic.cu -- plain-load kernels for any shape / alignment.
cudaError_t launch_generic_gemv(const DecodeArgs &a, cudaStream_t stream);

// prefill.cu -- tcgen05 block-FP8 / row-scaled / MXFP8 GEMM for larger m.
cudaError_t launch_prefill(const DecodeArgs &a, cudaStream_t stream);
// Grouped MoE GEMM over the routed experts (block scales): a.x [m, k] the
// tokens, a.codes / a.scales the stacked experts ([E * n, k], [E, ceil(n/128),
// ceil(k/128)]), a.y [m, topk, n]; the routing built by launch_moe_route.
cudaError_t launch_prefill_moe(const DecodeArgs &a, const MoeArgs &g, const MoeRoute &r, cudaStream_t stream);
uint32_t take_prefill_error();

// w8a8.cu -- e4m3 activations x e4m3 weight, both scaled per tensor.
struct W8A8Args {
    const uint8_t *xq;       // e4m3 [m, k] (row offset already applied)
    const float *sx;         // activation scale [1]
    const uint8_t *wq;       // e4m3 [n, k]
    const float *sw;         // weight scale [1]
    void *y;                 // bf16 [m, n] (row offset already applied)
    int64_t m, n, k;
};
cudaError_t launch_w8a8_decode(const W8A8Args &a, cudaStream_t stream);   // m <= 32
cudaError_t launch_w8a8_prefill(const W8A8Args &a, cudaStream_t stream);  // tcgen05
cudaError_t launch_w8a8_generic(const W8A8Args &a, cudaStream_t stream);  // any shape / alignment
uint32_t take_w8a8_error();

// tensormap.cu -- cuTensorMapEncodeTiled through the runtime's driver entry
// point (no link against libcuda).
bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// 3-D variant: dims innermost first, strides of dims 1 and 2 in bytes.
bool encode_tensor_map_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, const uint64_t (&dims)[3],
                          const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle);

// kvattn.cu -- FP8 E4M3 paged KV cache: append and split-KV decode attention.
struct KvAttnArgs {
    const void *q;               // bf16 [batch, q_heads, 128]
    const uint8_t *k_cache;      // e4m3 [num_blocks, page_size, kv_heads, 128]
    const uint8_t *v_cache;
    const float *k_scale;        // [1]
    const float *v_scale;        // [1]
    const int32_t *block_table;  // [batch, max_blocks]
    const int32_t *seq_lens;     // [batch]
    void *out;                   // bf16 [batch, q_heads, 128]
    int64_t batch, q_heads, kv_heads, page_size, num_blocks, max_blocks, max_seq_len;
    float sm_scale;
};
cudaError_t launch_kv_attention(const KvAttnArgs &a, cudaStream_t stream);
cudaError_t launch_kv_append(const void *x, int64_t num_tokens, int64_t kv_heads, const int32_t *slots,
                             const float *scale, uint8_t *cache, int64_t num_slots, cudaStream_t stream);
uint32_t take_kv_error();

// Multiprocessor count of the current device (cached per device).
int device_sm_count();

// Split-K cluster size for `tiles` clusters of one launch: the largest
// s <= max_split (<= 16; above 8 the kernel must allow non-portable cluster
// sizes) whose clusters of s CTAs (kernel `kern`, `threads` threads,
// `smem` dynamic shared memory, cluster dims (1, s, 1)) can all be resident
// at once, so the launch runs as a single wave -- a cluster size that does
// not pack onto the GPCs can halve the clusters that fit.  The per-device
// answers of cudaOccupancyMaxActiveClusters are cached in `fit`, one per
// kernel instantiation.  Returns 1 (no cluster) if none fits.
struct ClusterFit {
    int max_clusters[64][17] = {};  // 0: not asked yet; -1: the query failed
};
int pick_split(ClusterFit &fit, const void *kern, int threads, int smem, int tiles, int max_split);

}  // namespace fp8bs
