// moe.cu -- routing for the grouped MoE GEMM on the tensor cores (large m).
//
// The grouped GEMM (prefill.cu, prefill_kernel<kScaleBlock, MOE = true>)
// multiplies each selected expert's weight with the x rows of exactly the
// tokens routed to it.  It needs the (token, slot) pairs grouped by expert,
// which these kernels build on the device from the routing ids, with no host
// synchronisation, in the caller's workspace:
//   counts[e]    pairs routed to expert e
//   tok_off[e]   exclusive prefix sum of counts (tok_off[E] = valid pairs)
//   tile_off[e]  exclusive prefix sum of ceil(counts / gemm_tile): the
//                first of expert e's GEMM tiles (tile_off[E] = tiles in all)
//   tile_off_dec[e]  the same for tiles of kMoeDecodeTile pairs (the
//                decode path for few pairs per expert)
//   tile_info[t], tile_info_dec[t]  tile t of either kind as {expert,
//                first pair, pairs, 0}, so that a CTA finds its tile with
//                one load instead of a search over the offsets
//   perm[...]    pair indices p = t * topk + j, expert by expert
//                (tok_off[e] .. tok_off[e + 1]); within an expert in no
//                particular order -- every pair's output is computed on its
//                own, so the order changes no result.
//   xs[q, :]     x[perm[q] / topk, :]: the x rows in the same order, so that
//                each expert's rows are contiguous and the GEMM loads them
//                as ordinary TMA tiles.  For the decode tiles the copy is
//                written as f16, rescaled per (row, 128-column K block) by a
//                power of two, with the inverse factors of each tile in xinv
//                (the operands of the decode kernel's f16 MMAs).
// An id outside [0, E) routes nowhere and sets the error bit ERRBIT_INDEX.
#include "common.cuh"
#include "internal.h"

namespace fp8bs {

__device__ uint32_t g_moe_err;

namespace {

constexpr int kScanThreads = 1024;  // one block scans up to 1024 experts

__global__ void moe_count_kernel(const int32_t *__restrict__ ids, int64_t pairs, int num_experts,
                                 int32_t *__restrict__ counts) {
    pdl_launch_dependents();
    pdl_wait();  // the ids may come from the router, the previous kernel
    for (int64_t p = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; p < pairs;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int e = __ldg(ids + p);
        if (e >= 0 && e < num_experts)
            atomicAdd(counts + e, 1);
        else
            atomicOr(&g_moe_err, ERRBIT_INDEX);
    }
}

// Tiles of `size` pairs from the block's inclusive scans (s_tok: pairs,
// s_t: tiles of each expert): record t = {expert, first pair, pairs, 0},
// the expert found by a search in shared memory.
__device__ __forceinline__ void write_tiles(const int32_t *s_tok, const int32_t *s_t, int num_experts, int size,
                                            int4 *__restrict__ info) {
    const int ntiles = s_t[num_experts - 1];
    for (int t = threadIdx.x; t < ntiles; t += kScanThreads) {
        int lo = 0, hi = num_experts - 1;  // first e whose tiles end past t
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_t[mid] > t) hi = mid; else lo = mid + 1;
        }
        const int32_t first_pair = lo ? s_tok[lo - 1] : 0;
        const int32_t cnt = s_tok[lo] - first_pair;
        const int32_t i = t - (s_t[lo] - (cnt + size - 1) / size);  // tile index within the expert
        info[t] = make_int4(lo, first_pair + size * i, min(size, cnt - size * i), 0);
    }
}

// Exclusive prefix sums of counts and of their tile counts (gemm_tile pairs
// and kMoeDecodeTile pairs), the tile records of both kinds; the scatter
// cursors start at zero.
__global__ void __launch_bounds__(kScanThreads) moe_scan_kernel(const int32_t *__restrict__ counts,
                                                                int num_experts, int gemm_tile,
                                                                int32_t *__restrict__ tok_off,
                                                                int32_t *__restrict__ tile_off,
                                                                int32_t *__restrict__ tile_off_dec,
                                                                int4 *__restrict__ tile_info,
                                                                int4 *__restrict__ tile_info_dec,
                                                                int32_t *__restrict__ cursor) {
    __shared__ int32_t s_tok[kScanThreads], s_tile[kScanThreads], s_dec[kScanThreads];
    pdl_launch_dependents();
    pdl_wait();
    const int e = threadIdx.x;
    const int32_t c = e < num_experts ? counts[e] : 0;
    s_tok[e] = c;
    s_tile[e] = (c + gemm_tile - 1) / gemm_tile;
    s_dec[e] = (c + kMoeDecodeTile - 1) / kMoeDecodeTile;
    __syncthreads();
    // Hillis-Steele inclusive scan over the block
    for (int o = 1; o < kScanThreads; o <<= 1) {
        const int32_t a = e >= o ? s_tok[e - o] : 0, b = e >= o ? s_tile[e - o] : 0,
                      d = e >= o ? s_dec[e - o] : 0;
        __syncthreads();
        s_tok[e] += a;
        s_tile[e] += b;
        s_dec[e] += d;
        __syncthreads();
    }
    if (e < num_experts) {
        tok_off[e + 1] = s_tok[e];
        tile_off[e + 1] = s_tile[e];
        tile_off_dec[e + 1] = s_dec[e];
        cursor[e] = 0;
    }
    if (e == 0) {
        tok_off[0] = 0;
        tile_off[0] = 0;
        tile_off_dec[0] = 0;
    }
    write_tiles(s_tok, s_tile, num_experts, gemm_tile, tile_info);
    write_tiles(s_tok, s_dec, num_experts, kMoeDecodeTile, tile_info_dec);
}

// xs[q, :] = x[perm[q] / topk, :] for the routed pairs q < tok_off[E]; one
// warp per row, 16-byte copies (k % 16 == 0 on this path).
__global__ void moe_gather_kernel(const uint4 *__restrict__ x, int64_t pairs, int topk, int k,
                                  const int32_t *__restrict__ tok_off, int num_experts,
                                  const int32_t *__restrict__ perm, uint4 *__restrict__ xs) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t q = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (q >= pairs || q >= tok_off[num_experts]) return;
    const int64_t t = perm[q] / topk;
    const int chunks = k / 8;  // 16-byte chunks of a bf16 row
    const uint4 *src = x + t * chunks;
    uint4 *dst = xs + q * chunks;
    for (int c = lane; c < chunks; c += 32) dst[c] = __ldg(src + c);
}

// The decode-tile form of the gather.  Decode tile `tile` of expert e holds
// pairs p0 .. p0 + cnt - 1 (p0 = tok_off[e] + kMoeDecodeTile * (tile -
// tile_off_dec[e])); its row r < cnt becomes xs[p0 + r, :] =
// x[perm[p0 + r] / topk, :] * 2^s per 128-column K block kb, s =
// f16_rescale_exp(the largest |x| of that row and block), stored as f16, and
// xinv[(tile * kblocks + kb) * 32 + xinv_slot(r)] = 2^-s.  Rows r >= cnt
// (the next expert's pairs, whose outputs this tile never stores) read as
// zero here and get factor 1.  Block (tile, chunk of kGatherKb K blocks);
// warp w takes rows w, w + 8, w + 16, w + 24, all its loads in flight
// before the first reduction.  k % 4 == 0 (a lane's 4 columns are all in or
// all out).
constexpr int kGatherKb = 4;
__global__ void __launch_bounds__(256) moe_gather_f16_kernel(const uint2 *__restrict__ x, int topk, int k,
                                                             int kblocks, const int32_t *__restrict__ tile_off_dec,
                                                             const int4 *__restrict__ tile_info_dec,
                                                             int num_experts, const int32_t *__restrict__ perm,
                                                             uint2 *__restrict__ xs, float *__restrict__ xinv) {
    static_assert(kMoeDecodeTile == 32, "a block covers the 32 rows of one decode tile");
    pdl_launch_dependents();
    pdl_wait();
    const int tile = static_cast<int>(blockIdx.x);
    const int ntiles = tile_off_dec[num_experts];
    const int4 ti = tile_info_dec[tile];  // in bounds (the grid's bound); used only if tile < ntiles
    if (tile >= ntiles) return;
    const int p0 = ti.y, cnt = ti.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kbase = static_cast<int>(blockIdx.y) * kGatherKb;
    const int q4 = k >> 2;  // 4-value (8-byte) groups per row
    int64_t src[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = warp + 8 * i;
        src[i] = r < cnt ? static_cast<int64_t>(perm[p0 + r] / topk) : -1;
    }
    uint2 v[4][kGatherKb];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < kGatherKb; ++j) {
            const int c = (kbase + j) * 32 + lane;
            v[i][j] = (src[i] >= 0 && c < q4) ? __ldg(x + src[i] * q4 + c) : make_uint2(0u, 0u);
        }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < kGatherKb; ++j) {
            const int r = warp + 8 * i, kb = kbase + j;
            if (kb >= kblocks) continue;  // uniform across the block
            const uint32_t mx = max_u16x2(v[i][j].x & 0x7FFF7FFFu, v[i][j].y & 0x7FFF7FFFu);
            uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);  // |max| as bf16 bits
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, o));
            const int e = f16_rescale_exp(m16);
            const float mult = pow2_int(e);
            const int c = kb * 32 + lane;
            if (r < cnt && c < q4) {
                uint2 o;
                o.x = f32x2_to_f16x2(bf16lo_to_f32(v[i][j].x) * mult, bf16hi_to_f32(v[i][j].x) * mult);
                o.y = f32x2_to_f16x2(bf16lo_to_f32(v[i][j].y) * mult, bf16hi_to_f32(v[i][j].y) * mult);
                xs[static_cast<int64_t>(p0 + r) * q4 + c] = o;
            }
            if (lane == 0) xinv[(static_cast<int64_t>(tile) * kblocks + kb) * 32 + xinv_slot(r)] = pow2_int(-e);
        }
}

__global__ void moe_scatter_kernel(const int32_t *__restrict__ ids, int64_t pairs, int num_experts,
                                   const int32_t *__restrict__ tok_off, int32_t *__restrict__ cursor,
                                   int32_t *__restrict__ perm) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t p = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; p < pairs;
         p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int e = __ldg(ids + p);
        if (e < 0 || e >= num_experts) continue;
        perm[tok_off[e] + atomicAdd(cursor + e, 1)] = static_cast<int32_t>(p);
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

inline int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace

int64_t moe_route_bytes(int64_t pairs, int64_t num_experts, int64_t k) {
    const int64_t kblocks = (k + 127) / 128;
    const int64_t dec = moe_decode_tile_bound(pairs, num_experts);
    return 2 * align256(4 * num_experts) + 3 * align256(4 * (num_experts + 1)) +
           align256(16 * moe_gemm_tile_bound(pairs, num_experts, kMoeGemmTileNarrow)) + align256(16 * dec) +
           align256(4 * pairs) +
           align256(4 * dec * kblocks * 32) + align256(2 * pairs * k);
}

MoeRoute moe_route_views(void *workspace, int64_t pairs, int64_t num_experts, int64_t k) {
    char *p = static_cast<char *>(workspace);
    MoeRoute r;
    r.counts = reinterpret_cast<int32_t *>(p);
    p += align256(4 * num_experts);
    r.cursor = reinterpret_cast<int32_t *>(p);
    p += align256(4 * num_experts);
    r.tok_off = reinterpret_cast<int32_t *>(p);
    p += align256(4 * (num_experts + 1));
    r.tile_off = reinterpret_cast<int32_t *>(p);
    p += align256(4 * (num_experts + 1));
    r.tile_off_dec = reinterpret_cast<int32_t *>(p);
    p += align256(4 * (num_experts + 1));
    r.tile_info = reinterpret_cast<int4 *>(p);
    p += align256(16 * moe_gemm_tile_bound(pairs, num_experts, kMoeGemmTileNarrow));
    r.tile_info_dec = reinterpret_cast<int4 *>(p);
    p += align256(16 * moe_decode_tile_bound(pairs, num_experts));
    r.perm = reinterpret_cast<int32_t *>(p);
    p += align256(4 * pairs);
    r.xinv = reinterpret_cast<float *>(p);
    p += align256(4 * moe_decode_tile_bound(pairs, num_experts) * ((k + 127) / 128) * 32);
    r.xs = p;
    r.gemm_tile = kMoeGemmTileWide;
    return r;
}

cudaError_t launch_moe_route(const void *x, int64_t k, const int32_t *ids, int64_t pairs, int topk,
                             int num_experts, const MoeRoute &r, bool decode_tiles, cudaStream_t stream) {
    if (num_experts < 1 || num_experts > kScanThreads || pairs < 1) return cudaErrorInvalidValue;
    if (r.gemm_tile != kMoeGemmTileNarrow && r.gemm_tile != kMoeGemmTileWide) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(r.counts, 0, 4 * static_cast<size_t>(num_experts), stream);
    const unsigned blocks = static_cast<unsigned>((pairs + 255) / 256 < 1024 ? (pairs + 255) / 256 : 1024);
    if (e == cudaSuccess)
        e = launch_pdl(moe_count_kernel, dim3(blocks), dim3(256), stream, ids, pairs, num_experts, r.counts);
    if (e == cudaSuccess)
        e = launch_pdl(moe_scan_kernel, dim3(1), dim3(kScanThreads), stream, static_cast<const int32_t *>(r.counts),
                       num_experts, r.gemm_tile, r.tok_off, r.tile_off, r.tile_off_dec, r.tile_info, r.tile_info_dec,
                       r.cursor);
    if (e == cudaSuccess)
        e = launch_pdl(moe_scatter_kernel, dim3(blocks), dim3(256), stream, ids, pairs, num_experts,
                       static_cast<const int32_t *>(r.tok_off), r.cursor, r.perm);
    if (e == cudaSuccess && decode_tiles) {
        const int64_t tbound = moe_decode_tile_bound(pairs, num_experts);
        const int kblocks = static_cast<int>((k + 127) / 128);
        if (tbound > 0x7FFFFFFF || k % 4 != 0 || (kblocks + kGatherKb - 1) / kGatherKb > 65535)
            return cudaErrorInvalidValue;
        return launch_pdl(moe_gather_f16_kernel,
                          dim3(static_cast<unsigned>(tbound), static_cast<unsigned>((kblocks + kGatherKb - 1) / kGatherKb)),
                          dim3(256), stream, static_cast<const uint2 *>(x), topk, static_cast<int>(k), kblocks,
                          static_cast<const int32_t *>(r.tile_off_dec), static_cast<const int4 *>(r.tile_info_dec),
                          num_experts, static_cast<const int32_t *>(r.perm), static_cast<uint2 *>(r.xs), r.xinv);
    }
    if (e == cudaSuccess)
        e = launch_pdl(moe_gather_kernel, dim3(static_cast<unsigned>((pairs + 7) / 8)), dim3(256), stream,
                       static_cast<const uint4 *>(x), pairs, topk, static_cast<int>(k),
                       static_cast<const int32_t *>(r.tok_off), num_experts, static_cast<const int32_t *>(r.perm),
                       static_cast<uint4 *>(r.xs));
    return e;
}

uint32_t take_moe_error() {
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_moe_err, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_moe_err, &zero, sizeof zero);
    return v;
}

}  // namespace fp8bs
