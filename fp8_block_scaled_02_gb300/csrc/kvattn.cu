// kvattn.cu -- FP8 E4M3 paged KV cache (InfiniLM PR #586: an F8 cache with
// per-layer fp32 k_scale / v_scale for paged attention, split-KV decode).
//
//  * kv_append_kernel: new keys or values [tokens, kv_heads, 128] bf16 ->
//    e4m3(x / scale) (IEEE fp32 quotient, nearest-even, saturating) at flat
//    token slots of the cache [num_blocks, page_size, kv_heads, 128].
//  * kv_attn_kernel: decode attention o = softmax(sm_scale q.K^T) V for one
//    query token per sequence, K and V dequantized exactly (e4m3 -> f16) and
//    scaled once: k_scale folds into the score scale, v_scale into the
//    final normalisation.  One CTA per (sequence, kv head, KV split); the
//    query heads of the GQA group (<= 8) ride on the MMA's n axis, so each
//    K/V byte is read once for the whole group.  Each of 4 warps streams its
//    own 16-token chunks (3-D TMA of one page slice of one kv head, 128-byte
//    swizzle) through a 4-stage ring and runs, per chunk:
//      - S^T[16 tokens x 8 heads] = K (cvt.rn.f16x2.e4m3x2, exact) x q^T with
//        f16 mma.sync m16n8k16 (q carried in f16 after an exact power-of-two
//        rescale per head, undone in the score scale);
//      - an online softmax per head in fp32 (exp2, running max and sum);
//      - O^T[128 dims x 8 heads] += V^T x P^T: V converted to f16 in a
//        per-warp buffer and read transposed with ldmatrix.trans, P^T
//        (f16) assembled from the S^T fragments with four shuffles.
//    The 4 warps merge through shared memory; KV splits of one (sequence,
//    kv head) form a thread-block cluster and merge through DSMEM in rank
//    order (log-sum-exp rescaling), with no global workspace.
#include "common.cuh"
#include "internal.h"

#include <mutex>

namespace fp8bs {

namespace {

__device__ uint32_t g_kv_err;

constexpr int kD = 128;                      // head_dim
constexpr int kChunk = 16;                   // tokens per MMA tile / TMA box
constexpr int kGroup = 8;                    // query heads per kv head (MMA n)
constexpr int kMaxSplit = 16;                // cluster size (non-portable above 8)
constexpr int kTileBytes = kChunk * kD;      // 2 KB: one chunk of K or V
constexpr int kStageBytes = 2 * kTileBytes;  // K + V
constexpr int kVStride = kD * 2 + 16;        // f16 V row in the transpose buffer, padded
constexpr int kVScratch = kChunk * kVStride;
constexpr int kMergeFloats = 2 * kGroup + kD * kGroup;  // m[8], l[8], O[128][8]
// split merge receive buffer: [source rank][m[8], l[8], this rank's share of
// O]; splits * (16 + ceil(1024 / splits)) <= 16 * 16 + 1024 + 15 floats
constexpr int kRecvFloats = kMaxSplit * 2 * kGroup + kD * kGroup + kMaxSplit;
// W consumer warps per CTA, S chunks in flight per warp.  4 x 5 (two CTAs
// per SM) measured fastest on every decode shape; 8 x 5, 8 x 3, 4 x 8, 4 x 10
// (one CTA per SM) and 2 x 5 were all slower.
template <int W, int S>
struct KvCfg {
    static constexpr int kSmemBytes =
        1024 + W * S * kStageBytes + W * kVScratch + (kMergeFloats + kRecvFloats) * 4 + W * S * 8;
    static constexpr int kResident = kSmemBytes <= 113 * 1024 ? 2 : 1;  // CTAs per SM
    // a warp's merge record (after its loop) reuses its own, then idle, stages
    static_assert(kMergeFloats * 4 <= S * kStageBytes, "merge record fits a warp's stages");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <int W, int S>
__global__ void __launch_bounds__(W * 32, KvCfg<W, S>::kResident) kv_attn_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16 *__restrict__ q, const float *__restrict__ k_scale_p, const float *__restrict__ v_scale_p,
    const int32_t *__restrict__ table, const int32_t *__restrict__ seq_lens, __nv_bfloat16 *__restrict__ out,
    int kv_heads, int group, int page_size, int num_blocks, int max_blocks, int max_len, int splits,
    float sm_scale) {
    constexpr int kWarps = W, kStages = S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;                                         // [warp][stage][K | V]
    uint8_t *vscr = stages + kWarps * kStages * kStageBytes;        // [warp][16][kVStride]
    float *res = reinterpret_cast<float *>(vscr + kWarps * kVScratch);  // this CTA's m, l, O
    float *recv = res + kMergeFloats;                                   // split merge inputs
    uint64_t *full = reinterpret_cast<uint64_t *>(recv + kRecvFloats);  // [warp][stage]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int b = blockIdx.x / kv_heads, kvh = blockIdx.x % kv_heads;
    const int split = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWarps * kStages; ++i) mbar_init(&full[i], 1);
        fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    __syncthreads();
    pdl_wait();  // q, the cache and the tables may come from the previous kernel

    // The splits and warps partition the chunks of the longest sequence
    // (max_len, known on the host), so the block ids of a warp's chunks can
    // be read in the same round trip as the sequence length; chunks past
    // this sequence's length are then neither loaded nor computed.
    // Lane j holds the block id of the warp's chunk (window + j).
    const int max_chunks = (max_len + kChunk - 1) / kChunk;
    const int c0 = static_cast<int>((static_cast<int64_t>(split) * max_chunks) / splits);
    const int c1 = static_cast<int>((static_cast<int64_t>(split + 1) * max_chunks) / splits);
    const int my_max = c0 + warp < c1 ? (c1 - c0 - warp + kWarps - 1) / kWarps : 0;  // chunks c0 + warp + kWarps i
    const int32_t *trow = table + static_cast<int64_t>(b) * max_blocks;
    auto load_window = [&](int w0) -> int {
        const int i = w0 + lane;
        return i < my_max ? __ldg(trow + (c0 + warp + kWarps * i) * kChunk / page_size) : 0;
    };
    int len = __ldg(seq_lens + b);
    int win = 0;
    int myblk = load_window(0);
    const float k_scale = __ldg(k_scale_p), v_scale = __ldg(v_scale_p);
    const int cap = max_blocks * page_size;
    if (len < 0 || len > cap) {
        if (threadIdx.x == 0) atomicOr(&g_kv_err, ERRBIT_INDEX);
        len = len < 0 ? 0 : cap;
    }
    const int nchunks = (len + kChunk - 1) / kChunk;
    // this warp's chunks below the sequence length
    const int my_n = c0 + warp < min(c1, nchunks) ? (min(c1, nchunks) - c0 - warp + kWarps - 1) / kWarps : 0;

    // ---- q of head g of the group as f16 B fragments, exact power-of-two
    // rescale per head (maximum into [2^14, 2^15)).  Thread t holds dims
    // 32 sl + 8t .. +7 of each 32-wide slice sl (the k order the K fragments
    // use); heads beyond the group are zero.
    const int hq0 = kvh * group;
    const bool hvalid = g < group;
    const __nv_bfloat16 *qrow = q + (static_cast<int64_t>(b) * kv_heads * group + hq0 + (hvalid ? g : 0)) * kD;
    uint4 qv[4];
#pragma unroll
    for (int sl = 0; sl < 4; ++sl)
        qv[sl] = hvalid ? *reinterpret_cast<const uint4 *>(qrow + 32 * sl + 8 * t) : make_uint4(0, 0, 0, 0);
    uint32_t mx = 0;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
        mx = max_u16x2(mx, qv[sl].x & 0x7FFF7FFFu);
        mx = max_u16x2(mx, qv[sl].y & 0x7FFF7FFFu);
        mx = max_u16x2(mx, qv[sl].z & 0x7FFF7FFFu);
        mx = max_u16x2(mx, qv[sl].w & 0x7FFF7FFFu);
    }
    uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);
    m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, 1));
    m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, 2));
    int e = 0;
    if (m16 != 0) {
        const int field = static_cast<int>(m16 >> 7);
        e = min(126, max(-126, 14 - (field ? field - 127 : -133)));
    }
    const float mult = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    uint32_t bq[4][4];
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
        bq[sl][0] = f32x2_to_f16x2(bf16lo_to_f32(qv[sl].x) * mult, bf16hi_to_f32(qv[sl].x) * mult);
        bq[sl][1] = f32x2_to_f16x2(bf16lo_to_f32(qv[sl].y) * mult, bf16hi_to_f32(qv[sl].y) * mult);
        bq[sl][2] = f32x2_to_f16x2(bf16lo_to_f32(qv[sl].z) * mult, bf16hi_to_f32(qv[sl].z) * mult);
        bq[sl][3] = f32x2_to_f16x2(bf16lo_to_f32(qv[sl].w) * mult, bf16hi_to_f32(qv[sl].w) * mult);
    }
    // score scale (log2 domain) of this thread's C columns: heads 2t, 2t+1
    const float base = sm_scale * k_scale * kLog2e;
    const float sc0 = base * __shfl_sync(0xffffffffu, inv, 8 * t);
    const float sc1 = base * __shfl_sync(0xffffffffu, inv, 8 * t + 4);

    // ---- stream this warp's chunks
    uint64_t *wfull = full + warp * kStages;
    uint8_t *wst = stages + warp * kStages * kStageBytes;
    auto issue = [&](int i) {  // whole warp: TMA of K and V for the warp's i-th chunk (lane 0 issues)
        if ((i & ~31) != win) {
            win = i & ~31;
            myblk = load_window(win);
        }
        int blk = __shfl_sync(0xffffffffu, myblk, i & 31);
        if (lane == 0) {
            const int tok = (c0 + warp + kWarps * i) * kChunk;
            if (blk < 0 || blk >= num_blocks) {
                atomicOr(&g_kv_err, ERRBIT_INDEX);
                blk = 0;
            }
            const int row = blk * page_size + tok % page_size;
            uint64_t *bar = &wfull[i % kStages];
            uint8_t *st = wst + (i % kStages) * kStageBytes;
            mbar_arrive_expect_tx(bar, kStageBytes);
            tma_load_3d(st, &tm_k, bar, 0, kvh, row);
            tma_load_3d(st + kTileBytes, &tm_v, bar, 0, kvh, row);
        }
    };
    for (int i = 0; i < my_n && i < kStages; ++i) issue(i);

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[i][j] = 0.0f;
    uint8_t *myscr = vscr + warp * kVScratch;
    const int ra = 2 * g, rb = ra + 1;  // this thread's K rows (tokens) in the chunk
    const int coff = (t & 1) * 8;
    bool failed = false;
    int issued = my_n < kStages ? my_n : kStages;
    int consumed = 0;
    for (int i = 0; i < my_n; ++i, consumed = i) {
        const int s = i % kStages;
        const bool ready = mbar_wait_bounded(&wfull[s], (i / kStages) & 1);
        if (!__all_sync(0xffffffffu, ready)) {
            if (lane == 0) atomicOr(&g_kv_err, ERRBIT_FULL_WAIT);
            failed = true;
            break;
        }
        const uint8_t *kt = wst + s * kStageBytes;
        const uint8_t *vt = kt + kTileBytes;

        // S^T = K q^T: c0 (token 2g, head 2t), c1 (2g, 2t+1), c2 (2g+1, 2t), c3 (2g+1, 2t+1);
        // two accumulators (even / odd slices) halve the dependent MMA chain
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const int cchunk = 2 * sl + (t >> 1);
            const uint2 qa = *reinterpret_cast<const uint2 *>(kt + ra * 128 + ((cchunk ^ (ra & 7)) << 4) + coff);
            const uint2 qb = *reinterpret_cast<const uint2 *>(kt + rb * 128 + ((cchunk ^ (rb & 7)) << 4) + coff);
            uint32_t a00, a02, a01, a03, a10, a12, a11, a13;
            e4m3x4_to_f16x2x2(qa.x, a00, a02);
            e4m3x4_to_f16x2x2(qb.x, a01, a03);
            e4m3x4_to_f16x2x2(qa.y, a10, a12);
            e4m3x4_to_f16x2x2(qb.y, a11, a13);
            if (sl & 1) {
                mma_f16_16816(c2, a00, a01, a02, a03, bq[sl][0], bq[sl][1]);
                mma_f16_16816(c2, a10, a11, a12, a13, bq[sl][2], bq[sl][3]);
            } else {
                mma_f16_16816(c, a00, a01, a02, a03, bq[sl][0], bq[sl][1]);
                mma_f16_16816(c, a10, a11, a12, a13, bq[sl][2], bq[sl][3]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] += c2[j];
        const int tok0 = (c0 + warp + kWarps * i) * kChunk;
        const bool va = tok0 + ra < len, vb = tok0 + rb < len;
        const float s0 = va ? c[0] * sc0 : -INFINITY, s1 = va ? c[1] * sc1 : -INFINITY;
        const float s2 = vb ? c[2] * sc0 : -INFINITY, s3 = vb ? c[3] * sc1 : -INFINITY;
        // online softmax per head (2t: s0, s2; 2t+1: s1, s3) over the chunk's tokens
        float mt0 = fmaxf(s0, s2), mt1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, off));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, off));
        }
        const float mn0 = fmaxf(m_run[0], mt0), mn1 = fmaxf(m_run[1], mt1);
        const bool any0 = mn0 != -INFINITY, any1 = mn1 != -INFINITY;
        const float al0 = any0 ? exp2f(m_run[0] - mn0) : 1.0f;
        const float al1 = any1 ? exp2f(m_run[1] - mn1) : 1.0f;
        const float p0 = any0 ? exp2f(s0 - mn0) : 0.0f, p2 = any0 ? exp2f(s2 - mn0) : 0.0f;
        const float p1 = any1 ? exp2f(s1 - mn1) : 0.0f, p3 = any1 ? exp2f(s3 - mn1) : 0.0f;
        l_run[0] = l_run[0] * al0 + (p0 + p2);
        l_run[1] = l_run[1] * al1 + (p1 + p3);
        m_run[0] = mn0;
        m_run[1] = mn1;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
            o[d][0] *= al0;
            o[d][1] *= al1;
            o[d][2] *= al0;
            o[d][3] *= al1;
        }
        // P^T as the B operand (k = tokens, n = head g): b0 tokens 2t, 2t+1,
        // b1 tokens 2t+8, 2t+9 -- held by lanes (t, g/2) and (t+4, g/2)
        const uint32_t pk0 = f32x2_to_f16x2(p0, p2), pk1 = f32x2_to_f16x2(p1, p3);
        const int src0 = t * 4 + (g >> 1), src1 = (t + 4) * 4 + (g >> 1);
        const uint32_t x0 = __shfl_sync(0xffffffffu, pk0, src0), x1 = __shfl_sync(0xffffffffu, pk1, src0);
        const uint32_t y0 = __shfl_sync(0xffffffffu, pk0, src1), y1 = __shfl_sync(0xffffffffu, pk1, src1);
        const uint32_t pb0 = (g & 1) ? x1 : x0, pb1 = (g & 1) ? y1 : y0;

        // V chunk -> f16 [16 tokens][128 dims] (exact), then O^T += V^T P^T;
        // rows past the sequence end are zeroed (their p is 0, but unused
        // cache slots may hold any byte, NaN codes included)
        {
            const int row = lane >> 1;
            const bool live = tok0 + row < len;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int chunk = (lane & 1) * 4 + cc;
                const uint4 w = live ? *reinterpret_cast<const uint4 *>(vt + row * 128 + ((chunk ^ (row & 7)) << 4))
                                     : make_uint4(0, 0, 0, 0);
                uint4 lo, hi;
                e4m3x4_to_f16x2x2(w.x, lo.x, lo.y);
                e4m3x4_to_f16x2x2(w.y, lo.z, lo.w);
                e4m3x4_to_f16x2x2(w.z, hi.x, hi.y);
                e4m3x4_to_f16x2x2(w.w, hi.z, hi.w);
                uint8_t *dst = myscr + row * kVStride + chunk * 32;
                *reinterpret_cast<uint4 *>(dst) = lo;
                *reinterpret_cast<uint4 *>(dst + 16) = hi;
            }
        }
        __syncwarp();
        const uint32_t lbase =
            smem_u32(myscr) + ((lane & 7) + ((lane >> 4) << 3)) * kVStride + (((lane >> 3) & 1) << 3) * 2;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, lbase + d * 32);
            mma_f16_16816(o[d], a[0], a[1], a[2], a[3], pb0, pb1);
        }
        __syncwarp();  // stage and buffer reads are done: the stage may be refilled
        if (issued < my_n) issue(issued);
        ++issued;
    }
    // never leave with copies in flight (only after a failed wait): wait for
    // the chunks issued but not consumed, oldest first
    if (failed && lane == 0)
        for (int i = consumed; i < my_n && i < issued; ++i)
            (void)mbar_wait_bounded(&wfull[i % kStages], (i / kStages) & 1);

    // ---- per-warp totals: l summed over the chunk rows (lanes differing in g)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], off);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], off);
    }
    float *mw = reinterpret_cast<float *>(wst);  // m[8], l[8], O[d][8] in the warp's own idle stages
    if (g == 0) {
        mw[2 * t] = failed ? -INFINITY : m_run[0];
        mw[2 * t + 1] = failed ? -INFINITY : m_run[1];
        mw[kGroup + 2 * t] = failed ? 0.0f : l_run[0];
        mw[kGroup + 2 * t + 1] = failed ? 0.0f : l_run[1];
    }
    float *ow = mw + 2 * kGroup;
#pragma unroll
    for (int d = 0; d < 8; ++d) {
        const int d0 = 16 * d + g;
        ow[d0 * kGroup + 2 * t] = failed ? 0.0f : o[d][0];
        ow[d0 * kGroup + 2 * t + 1] = failed ? 0.0f : o[d][1];
        ow[(d0 + 8) * kGroup + 2 * t] = failed ? 0.0f : o[d][2];
        ow[(d0 + 8) * kGroup + 2 * t + 1] = failed ? 0.0f : o[d][3];
    }
    __syncthreads();

    // ---- merge the 4 warps: thread = one dim, all 8 heads
    auto rec = [&](int w) { return reinterpret_cast<const float *>(stages + w * kStages * kStageBytes); };
    if (threadIdx.x < kD) {
        const int d = threadIdx.x;
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, rec(w)[h]);
            float L = 0.0f, O = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float mw_h = rec(w)[h];
                    const float f = mw_h == -INFINITY ? 0.0f : exp2f(mw_h - M);
                    L += f * rec(w)[kGroup + h];
                    O += f * rec(w)[2 * kGroup + d * kGroup + h];
                }
            }
            res[2 * kGroup + d * kGroup + h] = O;
            if (d == 0) {
                res[h] = M;
                res[kGroup + h] = L;
            }
        }
    }
    __syncthreads();
    pdl_launch_dependents();

    // ---- merge the KV splits (cluster ranks) and store
    __nv_bfloat16 *ob = out + (static_cast<int64_t>(b) * kv_heads * group + hq0) * kD;
    if (splits == 1) {
        const int d = threadIdx.x;
        if (d >= kD) return;
        for (int h = 0; h < group; ++h) {
            const float L = res[kGroup + h];
            const float v = L > 0.0f ? res[2 * kGroup + d * kGroup + h] / L * v_scale : 0.0f;
            ob[static_cast<int64_t>(h) * kD + d] = __float2bfloat16_rn(v);
        }
        return;
    }
    // Every CTA pushes m, l and the share of O that rank q finishes into q's
    // receive slot (DSMEM stores, slot = source rank); one release / acquire
    // cluster barrier makes them visible and each rank merges locally in rank
    // order.  Nothing reads another CTA's shared memory afterwards, so no
    // second barrier is needed before exit.
    const int rank = static_cast<int>(cluster_ctarank());
    const int per = (kD * group + splits - 1) / splits;  // (dim, head) outputs a rank finishes
    const int slot = 2 * kGroup + per;
    {
        const uint32_t recv_base = smem_u32(recv) + static_cast<uint32_t>(rank * slot * 4);
        for (int e = threadIdx.x; e < splits * slot; e += kWarps * 32) {
            const int q = e / slot;
            const int i = e - q * slot;
            float v;
            if (i < 2 * kGroup) {
                v = res[i];
            } else {
                const int e2 = q * per + (i - 2 * kGroup);
                if (e2 >= kD * group) continue;
                const int h = e2 / kD, d = e2 - h * kD;
                v = res[2 * kGroup + d * kGroup + h];
            }
            dsmem_st_f32(dsmem_map(recv_base + static_cast<uint32_t>(i * 4), static_cast<uint32_t>(q)), v);
        }
    }
    cluster_sync_all();
    for (int e2 = rank * per + threadIdx.x; e2 < min(kD * group, (rank + 1) * per); e2 += kWarps * 32) {
        const int h = e2 / kD, d = e2 - h * kD;
        const int i = 2 * kGroup + (e2 - rank * per);
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxSplit; ++r)
            if (r < splits) M = fmaxf(M, recv[r * slot + h]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int r = 0; r < kMaxSplit; ++r) {
                if (r >= splits) continue;
                const float mr = recv[r * slot + h];
                const float f = mr == -INFINITY ? 0.0f : exp2f(mr - M);
                L += f * recv[r * slot + kGroup + h];
                O += f * recv[r * slot + i];
            }
        }
        ob[static_cast<int64_t>(h) * kD + d] = __float2bfloat16_rn(L > 0.0f ? O / L * v_scale : 0.0f);
    }
}

// ------------------------------------------------------------- cache append
constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const __nv_bfloat16 *__restrict__ x,
                                                                   int64_t num_tokens, int row_elems,
                                                                   const int32_t *__restrict__ slots,
                                                                   const float *__restrict__ scale_p,
                                                                   uint8_t *__restrict__ cache, int64_t num_slots) {
    pdl_wait();
    const float s = __ldg(scale_p);
    const int per_row = row_elems / 8;
    const int64_t total = num_tokens * per_row;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * kAppendThreads + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * kAppendThreads) {
        const int64_t tkn = idx / per_row;
        const int c = static_cast<int>(idx - tkn * per_row);
        const int64_t slot = __ldg(slots + tkn);
        if (slot < 0 || slot >= num_slots) {
            if (c == 0) atomicOr(&g_kv_err, ERRBIT_INDEX);
            continue;
        }
        const uint4 v = ld_nc_v4(x + tkn * row_elems + 8 * c);
        *reinterpret_cast<uint2 *>(cache + slot * row_elems + 8 * c) = encode8_div(v, s);
    }
}

struct KvSetup {
    std::mutex mu;
    bool done[64] = {};
    cudaError_t err[64] = {};
    int max_split[64] = {};
    ClusterFit fit;
};

template <int W, int S>
cudaError_t launch_kv_t(const KvAttnArgs &a, const CUtensorMap &tm_k, const CUtensorMap &tm_v, cudaStream_t stream) {
    using C = KvCfg<W, S>;
    auto kern = kv_attn_kernel<W, S>;
    static KvSetup setup;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int max_split = 8;
    {
        std::lock_guard<std::mutex> lock(setup.mu);
        if (!setup.done[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
            // clusters of up to 16 CTAs where the device allows them
            setup.max_split[dev] =
                cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess ? kMaxSplit
                                                                                                             : 8;
            (void)cudaGetLastError();
            setup.err[dev] = e;
            setup.done[dev] = true;
        }
        if (setup.err[dev] != cudaSuccess) return setup.err[dev];
        max_split = setup.max_split[dev];
    }
    const int group = static_cast<int>(a.q_heads / a.kv_heads);
    const int64_t pairs = a.batch * a.kv_heads;
    // one wave of CTAs, each warp with at least two chunks
    const int64_t chunks = (a.max_seq_len + kChunk - 1) / kChunk;
    int64_t splits = (C::kResident * static_cast<int64_t>(device_sm_count())) / pairs;
    const int64_t by_len = chunks / (2 * W);
    if (splits > by_len) splits = by_len;
    if (splits > max_split) splits = max_split;
    // only a cluster size whose clusters all fit at once (one wave)
    if (splits > 1)
        splits = pick_split(setup.fit, reinterpret_cast<const void *>(kern), W * 32, C::kSmemBytes,
                            static_cast<int>(pairs), static_cast<int>(splits));
    if (splits < 1) splits = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pairs), static_cast<unsigned>(splits), 1);
    cfg.blockDim = dim3(W * 32, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = static_cast<unsigned>(splits);
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    auto launch = [&]() {
        return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, static_cast<const __nv_bfloat16 *>(a.q), a.k_scale,
                                  a.v_scale, a.block_table, a.seq_lens, static_cast<__nv_bfloat16 *>(a.out),
                                  static_cast<int>(a.kv_heads), group, static_cast<int>(a.page_size),
                                  static_cast<int>(a.num_blocks), static_cast<int>(a.max_blocks),
                                  static_cast<int>(a.max_seq_len), static_cast<int>(splits), a.sm_scale);
    };
    cudaError_t e = launch();
    if (e != cudaSuccess && splits > 8) {
        // a non-portable cluster the device cannot place: fall back to 8
        (void)cudaGetLastError();
        splits = 8;
        cfg.gridDim.y = 8;
        attrs[1].val.clusterDim.y = 8;
        {
            std::lock_guard<std::mutex> lock(setup.mu);
            setup.max_split[dev] = 8;
        }
        e = launch();
    }
    return e;
}

}  // namespace

cudaError_t launch_kv_attention(const KvAttnArgs &a, cudaStream_t stream) {
    CUtensorMap tm_k, tm_v;
    const uint64_t hkv = static_cast<uint64_t>(a.kv_heads);
    const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * static_cast<uint64_t>(a.page_size);
    const uint64_t dims[3] = {static_cast<uint64_t>(kD), hkv, rows};
    const uint64_t strides[2] = {static_cast<uint64_t>(kD), hkv * kD};
    const uint32_t box[3] = {static_cast<uint32_t>(kD), 1u, static_cast<uint32_t>(kChunk)};
    if (!encode_tensor_map_3d(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_3d(&tm_v, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v_cache, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    return launch_kv_t<4, 5>(a, tm_k, tm_v, stream);
}

cudaError_t launch_kv_append(const void *x, int64_t num_tokens, int64_t kv_heads, const int32_t *slots,
                             const float *scale, uint8_t *cache, int64_t num_slots, cudaStream_t stream) {
    const int row = static_cast<int>(kv_heads * kD);
    const int64_t total = num_tokens * (row / 8);
    int64_t blocks = (total + kAppendThreads - 1) / kAppendThreads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    kv_append_kernel<<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(x), num_tokens, row, slots, scale, cache, num_slots);
    return cudaGetLastError();
}

uint32_t take_kv_error() {
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_kv_err, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_kv_err, &zero, sizeof zero);
    return v;
}

}  // namespace fp8bs
