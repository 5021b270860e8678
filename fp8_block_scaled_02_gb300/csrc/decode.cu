// decode.cu -- W8A16 block-FP8 / MXFP8 / per-row FP8 GEMV and skinny GEMM
// for small m (decode batches, m <= 32 per launch):
// y[m, n] = x[m, k] . dequant(W)^T.
//
// Design (sm_103a):
//  * One CTA owns 128 weight rows (one row of 128x128 block scales) and a
//    contiguous range of 128-wide K blocks.  With enough row tiles the grid is
//    persistent (about two CTAs per SM) and each CTA's TMA ring streams across
//    row-tile boundaries; with too few, the K blocks are split over the CTAs
//    of a thread-block cluster (up to 8) and the partial sums are reduced in
//    rank order through distributed shared memory -- no global workspace and
//    no waits on other CTAs beyond the hardware cluster barrier.
//  * A TMA warp streams each K block's 128x128 code tile (16 KB) and the
//    matching x tile (2-D TMA, 128-byte swizzle) into a shared-memory ring.
//  * For m <= 8 a converter warp rewrites each staged x tile in place from
//    bf16 to f16 with an exact power-of-two rescale per (row of x, 128-column
//    K block; per 32-column slice for MXFP8): the maximum is moved into
//    [2^14, 2^15), so every value within 2^-31 of it converts exactly and
//    nothing overflows; the inverse power of two is kept for the promotion
//    step.  Wider x keeps bf16 operands and needs no converter.
//  * Eight consumer warps each own one 16-row tile of the weight across the
//    whole 128-wide K block (so row sums never cross warps) and run
//    mma.sync m16n8k16 with the weights as the 16-row A operand and x as the
//    8-wide B operand (m on the MMA's n axis, so m <= 32 needs at most four
//    n8 tiles).  Codes convert with cvt.rn.f16x2.e4m3x2 (f16 form) or decode
//    to bf16 with integer ops, both exact.  The MMAs of a 128-wide K block
//    accumulate from zero and the block's fp32 partial is multiplied by
//    (block scale x inverse x rescale) once before it joins the running sum,
//    so the scale is applied once per K block to an fp32 partial and is never
//    folded into a rounded weight.  For MXFP8 each 32-column slice is one
//    e8m0 group, promoted on its own, whose exponents each warp fetches for
//    its rows one K block ahead.  With one scale per row (or per tensor) the
//    K blocks accumulate unscaled (bf16 operands: straight in the MMA) and
//    the row's scale multiplies the fp32 sum once, just before the bf16
//    rounding.
//  * The logical k order inside each MMA is a fixed permutation of the
//    physical columns, applied identically to A and B, so every thread
//    fetches 8 contiguous code bytes and 16 contiguous x bytes per K block
//    with conflict-free shared-memory loads.
//  * Grouped MoE (MOE = true): grid.z enumerates "expert slots"; each CTA
//    reads the routing ids, takes the blockIdx.z-th smallest expert that any
//    token selected (or leaves at once if there are fewer), streams that
//    expert's weight rows, runs every token's x through them (the MMA cost
//    of the extra rows is nothing next to the weight stream at m <= 32) and
//    stores only the outputs of tokens routed to it.  Each selected expert's
//    weight is read once per call, whatever the number of its tokens.
//  * Programmatic dependent launch: every CTA lets the next kernel in the
//    stream be scheduled as soon as it has started, and may itself start
//    (barrier init, tensor-map prefetch, an L2 prefetch of its first
//    ring-depth of code tiles) while the previous kernel drains; it reads
//    global memory only after griddepcontrol.wait.  An L2 prefetch cannot
//    observe stale data, so it is safe even if the previous kernel writes the
//    weight; on a chain of small GEMVs it hides the first DRAM latency.
#include "common.cuh"
#include "internal.h"

#include <cstring>
#include <mutex>

namespace fp8bs {

namespace {

__device__ uint32_t g_decode_err;

constexpr int kKB = 128;             // K per stage (one scale block)
constexpr int kConsumerWarps = 8;    // one 16-row tile of the 128 weight rows each
constexpr int kWarpTma = kConsumerWarps;
constexpr int kWarpConv0 = kConsumerWarps + 1;
constexpr int kMaxSplit = 8;         // portable cluster size limit
constexpr int kMoeMaxExperts = 1024; // experts a grouped call may address (bitmap of 32 words)

// F16: operands are f16 (codes via cvt.rn.f16x2.e4m3x2, x rescaled to f16 by
// a converter warp); otherwise bf16 (codes decoded with integer ops, x used
// as staged).  The f16 form halves the decode work and wins while the
// consumers are bound by it (m <= 8); beyond that the single converter warp
// becomes the bottleneck and the bf16 form, which needs none, wins.
// XP: x arrives prepared (an f16 copy with one power-of-two factor per row
// and K block, written by xprep_kernel), so f16 operands need no converter.
template <int MT, bool MX, bool F16, bool XP = false>
struct Cfg {
    // weight rows per CTA: one block-scale row.  Each of the 8 consumer
    // warps owns one 16-row tile across the whole 128-wide K block, so row
    // sums never cross warps; with m > 16 the x fragments of a K block are
    // loaded by every warp, which costs shared-memory reads but no
    // cross-warp reduction and only MT x 4 accumulators per thread.
    static constexpr int kBN = 128;
    // ring depth.  Clock stamps on [12288, 4096] put each code tile's load
    // at ~4700 cycles from issue to landing against 1500-2500 cycles of MMAs
    // per K block at m = 9..32, so the ring's depth sets the K-block rate
    // there; for m > 8 the split-K buffers reuse the drained ring to make
    // room for a deeper one (this CTA's partials from MT = 2, the cluster's
    // pushes too at MT = 4, which costs one more cluster barrier).  m <= 8
    // keeps five stages (a sixth measured 1.6% slower on lm_head).
    static constexpr int kStages = MT == 1 ? 5 : (MT == 2 ? 5 : 4);
    static constexpr bool kRedInRing = MT >= 2;
    static constexpr bool kRecvInRing = MT >= 4;
    static constexpr bool kConv = F16 && !XP;           // converter warp present
    static constexpr int kConvWarps = kConv ? 1 : 0;
    static constexpr int kThreads = (kConsumerWarps + 1 + kConvWarps) * 32;
    static constexpr int kXRows = 8 * MT;               // x rows staged (zero-padded)
    static constexpr int kCodeBytes = kBN * kKB;        // 16 KB
    static constexpr int kXPanelBytes = kXRows * 128;   // 64 columns of each row
    static constexpr int kStageBytes = kCodeBytes + 2 * kXPanelBytes;
    static constexpr int kXInvFloats = 4 * kXRows;      // per stage: [slice][row]
    static constexpr int kAuxBytes = kXInvFloats * 4;
    static constexpr int kRedStride = kXRows + 1;       // padded fp32 row
    static constexpr int kRedBytes = kBN * kRedStride * 4;
    // split-K receive buffer: [source rank][row of this CTA's slice][m];
    // splits * ceil(kBN / splits) <= kBN + 7 rows (even, for alignment)
    static constexpr int kRecvFloats = (kBN + kMaxSplit) * kRedStride;
    static constexpr int kRecvBytes = kRecvFloats * 4;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStages * kAuxBytes +
                                      (kRedInRing ? 0 : kRedBytes) + (kRecvInRing ? 0 : kRecvBytes) +
                                      3 * kStages * 8;
    static constexpr int kMinBlocks = 2;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert(kAuxBytes % 8 == 0 && kRedBytes % 16 == 0 && kRecvBytes % 8 == 0,
                  "the split-K buffers and the barriers stay aligned");
    static_assert(kRedBytes + kRecvBytes <= kStages * kStageBytes, "the split-K buffers fit in the drained ring");
    static_assert(!kRecvInRing || kRedInRing, "the receive buffer follows the partials");
    static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
};

// The op table of a batched launch.  It travels in the kernel's parameter
// space (no device buffer to allocate or fill), so its size is bounded by the
// 32 KB parameter limit: kBatchMaxOps ops per launch.  The tensor maps keep
// their own arrays (128-byte aligned, no padding between them).
struct BatchOp {
    const float *scales;     // block or row scales, else nullptr
    const uint8_t *e8m0;     // MX exponents, else nullptr
    __nv_bfloat16 *y;        // bf16 [m, n]
    const float *xinv;       // prepared x: inverse factors [kblocks][32], else nullptr
    int n, kblocks, groups;
    int ntiles;              // 128-row tiles of this weight
    int unit0;               // index of its first tile in the batch's unit list
    int e8m0_vec, row_stride;
};
struct BatchParams {
    CUtensorMap tm_codes[kBatchMaxOps];  // e4m3 [n, k], 128x128 boxes, 128-byte swizzle
    CUtensorMap tm_x[kBatchMaxOps];      // bf16 [m, k], 64 x (8 * MT) boxes
    BatchOp ops[kBatchMaxOps];
    int count, units;
};
static_assert(sizeof(BatchParams) + 64 <= 32764, "the op table must fit the kernel parameter space");

__device__ __forceinline__ float pow2_e8m0(uint32_t E) {
    return E ? __uint_as_float(E << 23) : __uint_as_float(0x00400000u);
}

// Rewrite one (x row r, 32-column slice sl) of a staged x tile from bf16 to
// f16 in place with the exact power-of-two rescale described above.
// kBlock: one power of two for the row's whole 128-column K block (the four
// slices of a row sit in four adjacent lanes, whose maxima are combined with
// two shuffles; every lane of the warp must take part), so that the consumers
// can accumulate the K block before promoting it once.
template <int kXPanelBytes, int kXRows, bool kBlock>
__device__ __forceinline__ void convert_x_slice(uint8_t *xs, float *xinv, int r, int sl) {
    uint8_t *base = xs + (sl >> 1) * kXPanelBytes + r * 128;
    const int c0 = 4 * (sl & 1);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4 *>(base + (((c0 + i) ^ (r & 7)) << 4));
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mx = max_u16x2(mx, v[i].x & 0x7FFF7FFFu);
        mx = max_u16x2(mx, v[i].y & 0x7FFF7FFFu);
        mx = max_u16x2(mx, v[i].z & 0x7FFF7FFFu);
        mx = max_u16x2(mx, v[i].w & 0x7FFF7FFFu);
    }
    uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);        // |max| as bf16 bits
    if (kBlock) {
        m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, 1));
        m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, 2));
    }
    const int k = f16_rescale_exp(m16);                 // scale 2^k
    const float mult = pow2_int(k);
    const float inv = pow2_int(-k);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 o;
        o.x = f32x2_to_f16x2(bf16lo_to_f32(v[i].x) * mult, bf16hi_to_f32(v[i].x) * mult);
        o.y = f32x2_to_f16x2(bf16lo_to_f32(v[i].y) * mult, bf16hi_to_f32(v[i].y) * mult);
        o.z = f32x2_to_f16x2(bf16lo_to_f32(v[i].z) * mult, bf16hi_to_f32(v[i].z) * mult);
        o.w = f32x2_to_f16x2(bf16lo_to_f32(v[i].w) * mult, bf16hi_to_f32(v[i].w) * mult);
        *reinterpret_cast<uint4 *>(base + (((c0 + i) ^ (r & 7)) << 4)) = o;
    }
    xinv[sl * kXRows + xinv_slot(r)] = inv;
}

// The units a CTA works on.  A unit is one 128-row tile of one weight over a
// range of its 128-wide K blocks.
//  * One weight (BATCH = false): the CTA takes row tiles blockIdx.x,
//    blockIdx.x + gridDim.x, ... over the K range of its split.  With
//    splits == 1 the grid is persistent and the TMA ring streams across tile
//    boundaries, so the next tile's codes are already arriving while the
//    consumers store the previous tile; with splits > 1 each CTA owns one row
//    tile and the cluster reduces over K.
//  * A batch of weights (BATCH = true): the row tiles of all the ops, in op
//    order, form one list of units, each over the whole of its weight's K;
//    the CTA takes units blockIdx.x, blockIdx.x + gridDim.x, ...  The ring
//    streams across unit and op boundaries alike, so a sequence of GEMVs runs
//    as one continuous weight stream instead of one launch (with its start-up
//    and tail) per weight.
// Grouped MoE by expert tiles (MOE with tile_off set): the routing's tiles
// of up to kMoeDecodeTile (token, slot) pairs of one expert (moe.cu), whose
// x rows were copied in pair order; tile_off nullptr: route by ids.
struct MoeGroups {
    const int32_t *tile_off;  // [E + 1] first tile of each expert (tile_off[E]: the count)
    const int4 *tile_info;    // [tile bound] {expert, first pair, pairs, 0} of each tile
    const int32_t *perm;      // pair indices t * topk + j, expert by expert
};

// Per-op view of what the roles read: the tensor maps and the scale and
// output pointers and sizes of one weight.
struct OpRef {
    const CUtensorMap *tm_codes;
    const CUtensorMap *tm_x;
    const float *scales;     // block [ceil(n/128), kblocks] or row scales (scales[row * row_stride])
    const uint8_t *e8m0;     // MX exponents [n, groups]
    __nv_bfloat16 *y;        // [m, n]
    const float *xinv;       // prepared x (XP): inverse factors [kblocks][32]
    int n, kblocks, groups, e8m0_vec, row_stride;
};

// SC: how the weight is scaled (ScaleKind: 128x128 blocks, MX groups, rows)
// MOE: grouped expert GEMV (block scales); n is the rows of one expert, the
// codes / scales hold num_experts such weights back to back, ids [m, topk].
// With mg.tile_off set, blockIdx.z is an expert tile of the routing instead
// (x: the pair-order copy, its rows from the tile's first pair; output row i
// goes to y[pair_i * n + row], y: [tokens, topk, n]); with XP the copy is
// f16 and xinv_g holds each tile's inverse factors, [tile][kblocks][32]).
// BATCH: the ops come from `bp` (the single-weight arguments are unused).
template <int MT, int SC, bool F16, bool MOE, bool BATCH, bool XP = false>
__device__ __forceinline__ void decode_body(const BatchParams *bp, const float *__restrict__ xinv_g,
                                            const CUtensorMap *tm_codes,
                                            const CUtensorMap *tm_x, const float *__restrict__ scales,
                                            const uint8_t *__restrict__ e8m0, __nv_bfloat16 *__restrict__ y,
                                            int m, int n, int kblocks, int groups, int splits, int ntiles,
                                            int e8m0_vec, int row_stride, const int32_t *__restrict__ ids,
                                            int topk, int num_experts,
                                            MoeGroups mg = MoeGroups{nullptr, nullptr, nullptr}) {
    constexpr bool MX = SC == kScaleMx;
    constexpr bool ROW = SC == kScaleRow;  // no per-K-block scale; scales[row * row_stride] at the end
    // no per-slice factor (e8m0 groups): the MMAs accumulate a whole K block
    constexpr bool kWholeBlock = !MX;
    // ... and with bf16 operands and one scale per row, all of K
    constexpr bool kDirect = kWholeBlock && ROW && !F16;
    static_assert(!(MOE && BATCH), "a grouped MoE call is one launch of its own");
    // prepared x feeds the block-scaled f16 path (MOE: the routing's decode
    // tiles, whose factors are per tile)
    static_assert(!XP || (F16 && !MX), "prepared x feeds the block-scaled f16 path");
    using C = Cfg<MT, MX, F16, XP>;
    constexpr int kStages = C::kStages;
    constexpr int kBN = C::kBN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    float *aux = reinterpret_cast<float *>(smem + kStages * C::kStageBytes);
    // split-K (one unit per CTA): this CTA's partials and the cluster's
    // pushes, in the ring once every stage is consumed (see below) or after
    // the exponent area
    float *own = aux + kStages * C::kXInvFloats;
    float *red = C::kRedInRing ? reinterpret_cast<float *>(smem) : own;
    if (!C::kRedInRing) own += kBN * C::kRedStride;
    float *recv = C::kRecvInRing ? red + kBN * C::kRedStride : own;
    if (!C::kRecvInRing) own += C::kRecvFloats;
    uint64_t *full = reinterpret_cast<uint64_t *>(own);
    uint64_t *xready = full + kStages;
    uint64_t *empty = xready + kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // one weight: this CTA's K range (split-K); a batch: every unit runs all of K
    const int split = BATCH ? 0 : static_cast<int>(blockIdx.y);
    const int kb0 = BATCH ? 0 : static_cast<int>((static_cast<int64_t>(split) * kblocks) / splits);
    const int kb1 = BATCH ? 0 : static_cast<int>((static_cast<int64_t>(split + 1) * kblocks) / splits);
    const int tile0 = blockIdx.x, tstep = gridDim.x;
    const int nunits = BATCH ? bp->units : ntiles;
    const int my_units = tile0 < nunits ? (nunits - tile0 + tstep - 1) / tstep : 0;
    const int mm = min(m, C::kXRows);
    __shared__ uint32_t s_bits[kMoeMaxExperts / 32];  // MOE: experts any token selected
    __shared__ int s_expert;                          // MOE: this CTA's expert
    __shared__ signed char s_route[32];               // MOE: slot j of x row mi for it, -1 if none
    __shared__ int32_t s_pair[32];                    // MOE by tiles: pair of x row mi, -1 past the tile
    __shared__ int s_x_row0;                          // MOE by tiles: the tile's first pair

    // Unit i of this CTA: its op (BATCH: `op` is a cursor that only moves
    // forward, units are visited in increasing order), first weight row and
    // K blocks [kbb, kbb + nkb).
    auto locate = [&](int i, int &op, int &n0, int &kbb, int &nkb) {
        const int u = tile0 + i * tstep;
        if (BATCH) {
            while (u >= bp->ops[op].unit0 + bp->ops[op].ntiles) ++op;
            n0 = (u - bp->ops[op].unit0) * kBN;
            kbb = 0;
            nkb = bp->ops[op].kblocks;
        } else {
            n0 = u * kBN;
            kbb = kb0;
            nkb = kb1 - kb0;
        }
    };
    auto op_ref = [&](int op) -> OpRef {
        if (BATCH) {
            const BatchOp &o = bp->ops[op];
            return OpRef{&bp->tm_codes[op], &bp->tm_x[op], o.scales, o.e8m0, o.y, o.xinv, o.n, o.kblocks, o.groups,
                         o.e8m0_vec, o.row_stride};
        }
        return OpRef{tm_codes, tm_x, scales, e8m0, y, xinv_g, n, kblocks, groups, e8m0_vec, row_stride};
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&xready[s], C::kConv ? C::kConvWarps : 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbarrier_init();
    }
    if (warp == kWarpTma && lane == 0) {
        if (!BATCH) {
            prefetch_tensormap(tm_codes);
            prefetch_tensormap(tm_x);
        }
        // While the previous kernel drains, start this CTA's first ring-depth
        // of weight tiles on their way into L2 (more would delay the first
        // loads when there is nothing to overlap; MoE CTAs do not know their
        // expert yet).
        if (!MOE) {
            int left = kStages, op = 0, prev = -1;
            for (int i = 0; i < my_units && left > 0; ++i) {
                int n0, kbb, nkb;
                locate(i, op, n0, kbb, nkb);
                const OpRef o = op_ref(op);
                if (BATCH && op != prev) {
                    prefetch_tensormap(o.tm_codes);
                    prefetch_tensormap(o.tm_x);
                    prev = op;
                }
                for (int kb = 0; kb < nkb && left > 0; ++kb, --left)
                    tma_prefetch_l2_2d(o.tm_codes, (kbb + kb) * kKB, n0);
            }
        }
    }
    __syncthreads();
    // Nothing before this point reads what an earlier kernel writes, so the
    // next kernel in the stream may be scheduled now; it waits for this one
    // to complete before it reads any input.
    pdl_launch_dependents();
    pdl_wait();  // inputs may be produced by the previous kernel in the stream

    int expert = 0;
    int x_row0 = 0;  // MOE by tiles: the tile's first pair (row of the pair-order copy of x)
    const bool by_tiles = MOE && mg.tile_off != nullptr;
    if (MOE && XP && !by_tiles) {
        // prepared factors exist only per routing tile: nothing was issued yet
        if (threadIdx.x == 0) atomicOr(&g_decode_err, ERRBIT_INDEX);
        return;
    }
    if (by_tiles) {
        // blockIdx.z is an expert tile; every CTA of a cluster shares it, so
        // an idle cluster leaves whole, before anything is issued
        const int tile = static_cast<int>(blockIdx.z);
        // the tile count and the tile's record: two independent loads (the
        // record is in bounds, the grid's bound; used only if tile < count)
        int4 ti = make_int4(0, 0, 0, 0);
        if (threadIdx.x < 32) ti = __ldg(mg.tile_info + tile);
        if (tile >= __ldg(mg.tile_off + num_experts)) return;
        if (threadIdx.x < 32) {
            s_pair[threadIdx.x] = threadIdx.x < ti.z ? __ldg(mg.perm + ti.y + threadIdx.x) : -1;
            if (threadIdx.x == 0) {
                s_expert = ti.x;
                s_x_row0 = ti.y;
            }
        }
        __syncthreads();
        expert = s_expert;
        x_row0 = s_x_row0;
        if (XP) xinv_g += static_cast<int64_t>(tile) * kblocks * 32;  // this tile's factors
    } else if (MOE) {
        for (int i = threadIdx.x; i < kMoeMaxExperts / 32; i += blockDim.x) s_bits[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < m * topk; i += blockDim.x) {
            const int e = __ldg(ids + i);
            if (e >= 0 && e < num_experts)
                atomicOr(&s_bits[e >> 5], 1u << (e & 31));
            else
                atomicOr(&g_decode_err, ERRBIT_INDEX);
        }
        __syncthreads();
        if (warp == 0) {
            // slot blockIdx.z -> the blockIdx.z-th smallest selected expert
            const uint32_t word = s_bits[lane];
            const int cnt = __popc(word);
            int pre = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o) pre += v;
            }
            const int target = static_cast<int>(blockIdx.z);
            int found = -1;
            if (target >= pre - cnt && target < pre) {
                uint32_t w = word;
                for (int r = target - (pre - cnt); r > 0; --r) w &= w - 1;  // drop the r lowest set bits
                found = lane * 32 + __ffs(static_cast<int>(w)) - 1;
            }
            const unsigned holder = __ballot_sync(0xffffffffu, found >= 0);
            found = holder ? __shfl_sync(0xffffffffu, found, __ffs(static_cast<int>(holder)) - 1) : -1;
            if (lane == 0) s_expert = found;
        }
        __syncthreads();
        expert = s_expert;
        // fewer selected experts than slots: nothing was issued yet, and every
        // CTA of a cluster shares blockIdx.z, so the whole cluster leaves
        if (expert < 0) return;
        if (threadIdx.x < 32) {
            int r = -1, hits = 0;
            if (threadIdx.x < m)
                for (int j = topk - 1; j >= 0; --j)
                    if (__ldg(ids + threadIdx.x * topk + j) == expert) {
                        r = j;
                        ++hits;
                    }
            // a token that lists this expert twice breaks the distinct-ids
            // precondition: only the lowest slot would be written
            if (hits > 1) atomicOr(&g_decode_err, ERRBIT_INDEX);
            s_route[threadIdx.x] = static_cast<signed char>(r);
        }
        __syncthreads();
    }
    // flat index into y of output (x row mi, weight row nn) of a weight with
    // `nrows` rows, or -1 if not stored
    auto out_at = [&](int mi, int nn, int nrows) -> int64_t {
        if (!MOE) return static_cast<int64_t>(mi) * nrows + nn;
        if (by_tiles) {
            const int pr = mi < 32 ? s_pair[mi] : -1;
            return pr < 0 ? -1 : static_cast<int64_t>(pr) * nrows + nn;
        }
        const int j = s_route[mi];
        return j < 0 ? -1 : (static_cast<int64_t>(mi) * topk + j) * nrows + nn;
    };
    const int row_base = MOE ? expert * n : 0;  // expert's first row in the stacked codes
    const int64_t scale_off = MOE ? static_cast<int64_t>(expert) * ((n + 127) >> 7) * kblocks : 0;

    if (warp == kWarpTma) {
        // ------------------------------------------------------ TMA producer
        // The whole warp walks the ring (so it stays converged); lane 0
        // waits for a free stage and issues the TMA copies.
        const uint64_t stream_policy = policy_evict_first();
        int it = 0, op = 0;
        bool stop = false;
        for (int i = 0; i < my_units && !stop; ++i) {
            int n0, kbb, nkb;
            locate(i, op, n0, kbb, nkb);
            const OpRef o = op_ref(op);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = it % kStages;
                int good = 1;
                if (it >= kStages && lane == 0) good = mbar_wait_bounded(&empty[s], ((it / kStages) - 1) & 1);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    if (lane == 0) atomicOr(&g_decode_err, ERRBIT_EMPTY_WAIT);
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    const int kx = (kbb + kb) * kKB;
                    uint8_t *st = smem + s * C::kStageBytes;
                    mbar_arrive_expect_tx(&full[s], C::kStageBytes + (XP ? C::kXRows * 4 : 0));
                    tma_load_2d_hint(st, o.tm_codes, &full[s], kx, row_base + n0, stream_policy);
                    tma_load_2d(st + C::kCodeBytes, o.tm_x, &full[s], kx, x_row0);
                    tma_load_2d(st + C::kCodeBytes + C::kXPanelBytes, o.tm_x, &full[s], kx + 64, x_row0);
                    // prepared x: this K block's inverse factors, in the slot
                    // order the consumers read (xprep_kernel)
                    if (XP)
                        bulk_load_g2s(aux + s * C::kXInvFloats, o.xinv + (kbb + kb) * 32, C::kXRows * 4, &full[s]);
                }
                __syncwarp();
            }
        }
    } else if (C::kConv && warp >= kWarpConv0) {
        // ------------------------------------------------------ x converter
        const int clane = (warp - kWarpConv0) * 32 + lane;
        constexpr int kConvLanes = C::kConvWarps * 32;
        int it = 0, op = 0;
        bool stop = false;
        for (int i = 0; i < my_units && !stop; ++i) {
            int n0, kbb, nkb;
            locate(i, op, n0, kbb, nkb);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = it % kStages;
                const bool ready = mbar_wait_bounded(&full[s], (it / kStages) & 1);
                if (!__all_sync(0xffffffffu, ready)) {
                    // the consumers' own bounded waits on xready then give up too
                    if (lane == 0) atomicOr(&g_decode_err, ERRBIT_FULL_WAIT);
                    stop = true;
                    break;
                }
                uint8_t *xs = smem + s * C::kStageBytes + C::kCodeBytes;
                float *xinv = aux + s * C::kXInvFloats;
                static_assert(!C::kConv || MX || 4 * C::kXRows == kConvLanes,
                              "a per-block rescale needs one slice per lane");
                for (int u = clane; u < 4 * C::kXRows; u += kConvLanes)
                    convert_x_slice<C::kXPanelBytes, C::kXRows, !MX>(xs, xinv, u >> 2, u & 3);
                fence_proxy_async_smem();  // the TMA will overwrite these bytes later
                __syncwarp();
                if (lane == 0) mbar_arrive(&xready[s]);
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        const int g = lane >> 2, t = lane & 3;
        const int ra = warp * 16 + 2 * g, rb = ra + 1;  // this thread's two weight rows
        // x rows of this thread's B fragments: row 8j + pi(g) with
        // pi(g) = (g >> 1) | ((g & 1) << 2) (bank-conflict-free swizzle use)
        const int xrow_base = (g >> 1) | ((g & 1) << 2);
        const int coff = (t & 1) * 8;
        int it = 0, op = 0;
        bool failed = false;
        for (int ui = 0; ui < my_units && !failed; ++ui) {
            int n0, kbb, nkb;
            locate(ui, op, n0, kbb, nkb);
            const OpRef o = op_ref(op);
            // factor applied to a finished fp32 sum of weight row nn before rounding
            auto out_scale = [&](int nn) -> float {
                return ROW ? __ldg(o.scales + static_cast<int64_t>(nn) * o.row_stride) : 1.0f;
            };
            const float *srow = (MX || ROW) ? nullptr
                                            : o.scales + scale_off + static_cast<int64_t>(n0 >> 7) * o.kblocks + kbb;
            float acc[MT][4];
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;
            float s_next = (MX || ROW) ? 1.0f : __ldg(srow);
            // MX: lane l < 16 holds the e8m0 word (4 groups of this K block) of
            // weight row 16*warp + l, fetched two K blocks ahead
            auto load_e8m0_word = [&](int kbi) -> uint32_t {
                const int64_t row = static_cast<int64_t>(n0) + warp * 16 + lane;
                const int g0 = (kbb + kbi) * 4;
                uint32_t w = 0;
                if (lane < 16 && row < o.n) {
                    const uint8_t *p = o.e8m0 + row * o.groups + g0;
                    if (o.e8m0_vec) {
                        w = __ldg(reinterpret_cast<const uint32_t *>(p));
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (g0 + q < o.groups) w |= static_cast<uint32_t>(__ldg(p + q)) << (8 * q);
                    }
                }
                return w;
            };
            // MX: ask L2 for this warp's rows' exponents of the whole unit (each
            // row's run of 4 bytes per K block is contiguous), so the words
            // fetched two K blocks ahead below come from L2, not HBM
            if (MX && lane < 16) {
                const int64_t row = static_cast<int64_t>(n0) + warp * 16 + lane;
                const int g0 = kbb * 4;
                const int bytes = min(nkb * 4, o.groups - g0);
                if (row < o.n && bytes > 0) {
                    const uint8_t *p = o.e8m0 + row * o.groups + g0;
                    for (int off = 0; off < bytes; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p + bytes - 1));
                }
            }
            uint32_t e_next = MX ? load_e8m0_word(0) : 0u;
            uint32_t e_next2 = (MX && nkb > 1) ? load_e8m0_word(1) : 0u;
            for (int kbi = 0; kbi < nkb; ++kbi, ++it) {
                const int s = it % kStages;
                const float sblk = s_next;
                if (!MX && !ROW && kbi + 1 < nkb) s_next = __ldg(srow + kbi + 1);
                const uint32_t e_cur = e_next;
                if (MX) {
                    e_next = e_next2;
                    if (kbi + 2 < nkb) e_next2 = load_e8m0_word(kbi + 2);
                }
                const uint32_t ewa = MX ? __shfl_sync(0xffffffffu, e_cur, 2 * g) : 0u;
                const uint32_t ewb = MX ? __shfl_sync(0xffffffffu, e_cur, 2 * g + 1) : 0u;
                const uint32_t par = (it / kStages) & 1;
                const bool ready =
                    mbar_wait_bounded(&full[s], par) && (!C::kConv || mbar_wait_bounded(&xready[s], par));
                if (!__all_sync(0xffffffffu, ready)) {
                    if (lane == 0) atomicOr(&g_decode_err, ERRBIT_FULL_WAIT);
                    failed = true;
                    break;
                }
                const uint8_t *cs = smem + s * C::kStageBytes;
                const uint8_t *xbase = cs + C::kCodeBytes;
                const float *xinv = aux + s * C::kXInvFloats;
                // Without MX groups the promotion factor (block scale, times the
                // x rescale for f16 operands) is the same for the K block's four
                // slices: the MMAs accumulate the whole block and it is promoted
                // once.  bf16 with one scale per row needs no promotion at all.
                float cb[MT][4];
                if (kWholeBlock && !kDirect) {
#pragma unroll
                    for (int j = 0; j < MT; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) cb[j][q] = 0.0f;
                }
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    const uint8_t *xs = xbase + (sl >> 1) * C::kXPanelBytes;
                    const int xchunk = 4 * (sl & 1) + t;
                    uint32_t bx[MT][4];
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        const int xr = 8 * j + xrow_base;
                        const uint4 v =
                            *reinterpret_cast<const uint4 *>(xs + xr * 128 + ((xchunk ^ (xr & 7)) << 4));
                        bx[j][0] = v.x;
                        bx[j][1] = v.y;
                        bx[j][2] = v.z;
                        bx[j][3] = v.w;
                    }
                    const int cchunk = 2 * sl + (t >> 1);
                    const uint2 qa =
                        *reinterpret_cast<const uint2 *>(cs + ra * 128 + ((cchunk ^ (ra & 7)) << 4) + coff);
                    const uint2 qb =
                        *reinterpret_cast<const uint2 *>(cs + rb * 128 + ((cchunk ^ (rb & 7)) << 4) + coff);
                    uint32_t a00, a02, a01, a03, a10, a12, a11, a13;
                    if (F16) {
                        e4m3x4_to_f16x2x2(qa.x, a00, a02);
                        e4m3x4_to_f16x2x2(qb.x, a01, a03);
                        e4m3x4_to_f16x2x2(qa.y, a10, a12);
                        e4m3x4_to_f16x2x2(qb.y, a11, a13);
                    } else {
                        a00 = e4m3x2_to_bf16x2(qa.x, 0x9180u);
                        a02 = e4m3x2_to_bf16x2(qa.x, 0xB3A2u);
                        a01 = e4m3x2_to_bf16x2(qb.x, 0x9180u);
                        a03 = e4m3x2_to_bf16x2(qb.x, 0xB3A2u);
                        a10 = e4m3x2_to_bf16x2(qa.y, 0x9180u);
                        a12 = e4m3x2_to_bf16x2(qa.y, 0xB3A2u);
                        a11 = e4m3x2_to_bf16x2(qb.y, 0x9180u);
                        a13 = e4m3x2_to_bf16x2(qb.y, 0xB3A2u);
                    }
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        if constexpr (kWholeBlock) {
                            float(&d)[4] = kDirect ? acc[j] : cb[j];
                            if (F16) {
                                mma_f16_16816(d, a00, a01, a02, a03, bx[j][0], bx[j][1]);
                                mma_f16_16816(d, a10, a11, a12, a13, bx[j][2], bx[j][3]);
                            } else {
                                mma_bf16_16816(d, a00, a01, a02, a03, bx[j][0], bx[j][1]);
                                mma_bf16_16816(d, a10, a11, a12, a13, bx[j][2], bx[j][3]);
                            }
                        } else {
                            // MX: the slice is one e8m0 group of each row, and
                            // (f16) x carries its own per-slice rescale
                            float f0 = 1.0f, f1 = 1.0f;
                            if (F16) {
                                const float2 iv =
                                    *reinterpret_cast<const float2 *>(xinv + sl * C::kXRows + 8 * j + 2 * t);
                                f0 = iv.x;
                                f1 = iv.y;
                            }
                            const float sa = pow2_e8m0((ewa >> (8 * sl)) & 0xFFu);
                            const float sb = pow2_e8m0((ewb >> (8 * sl)) & 0xFFu);
                            float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            if (F16) {
                                mma_f16_16816(c, a00, a01, a02, a03, bx[j][0], bx[j][1]);
                                mma_f16_16816(c, a10, a11, a12, a13, bx[j][2], bx[j][3]);
                            } else {
                                mma_bf16_16816(c, a00, a01, a02, a03, bx[j][0], bx[j][1]);
                                mma_bf16_16816(c, a10, a11, a12, a13, bx[j][2], bx[j][3]);
                            }
                            acc[j][0] = fmaf(sa * f0, c[0], acc[j][0]);
                            acc[j][1] = fmaf(sa * f1, c[1], acc[j][1]);
                            acc[j][2] = fmaf(sb * f0, c[2], acc[j][2]);
                            acc[j][3] = fmaf(sb * f1, c[3], acc[j][3]);
                        }
                    }
                }
                if (kWholeBlock && !kDirect) {
                    // promotion factor of x rows 8j + t (f0) and 8j + t + 4 (f1)
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        float f0 = sblk, f1 = sblk;
                        if (F16) {
                            const float2 iv = *reinterpret_cast<const float2 *>(xinv + 8 * j + 2 * t);
                            f0 *= iv.x;
                            f1 *= iv.y;
                        }
                        acc[j][0] = fmaf(f0, cb[j][0], acc[j][0]);
                        acc[j][1] = fmaf(f1, cb[j][1], acc[j][1]);
                        acc[j][2] = fmaf(f0, cb[j][2], acc[j][2]);
                        acc[j][3] = fmaf(f1, cb[j][3], acc[j][3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // split-K: the partials go to `red`, which may overlay the ring:
            // every consumer warp has consumed every stage of its single
            // unit (and every TMA copy has landed) once all of them are here
            // -- failed warps included, so that none waits for a warp that left
            if (C::kRedInRing && splits > 1) asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            if (failed) break;
            // acc[j][q] is y[m = 8j + t + 4(q&1)][n_local = ra + (q>>1)]
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int mi = 8 * j + t + 4 * (q & 1);
                    const int nl = ra + (q >> 1);
                    if (splits == 1) {
                        const int64_t oi = (mi < m && n0 + nl < o.n) ? out_at(mi, n0 + nl, o.n) : -1;
                        if (oi >= 0)
                            o.y[oi] = __float2bfloat16_rn(ROW ? acc[j][q] * out_scale(n0 + nl) : acc[j][q]);
                    } else {
                        red[nl * C::kRedStride + mi] = acc[j][q];
                    }
                }
        }
    }
    if (BATCH || splits == 1) return;

    // Split-K: one row tile per CTA; reduce across the cluster in rank order.
    // CTA r finishes rows [r * rows_per, (r + 1) * rows_per) of the tile.
    // Every CTA pushes each row's partial straight into its finisher's
    // receive buffer (DSMEM stores, slot = source rank; where the buffer
    // overlays the owner's drained ring, a first cluster barrier waits for
    // every CTA's main loop), then a cluster barrier (release / acquire) makes all
    // of them visible; each CTA sums its slots locally in rank order and
    // leaves.  Nothing reads another CTA's shared memory, so no further
    // barrier is needed before exit.
    __syncthreads();  // local partials complete in red
    // pushes into a ring: wait until every CTA of the cluster is past its
    // main loop
    if (C::kRecvInRing) cluster_sync_all();
    const int n0 = tile0 * kBN;
    const int rank = static_cast<int>(cluster_ctarank());
    const int rows_per = (kBN + splits - 1) / splits;
    {
        const uint32_t recv_base = smem_u32(recv) + static_cast<uint32_t>(rank * rows_per * C::kRedStride * 4);
        for (int e = threadIdx.x; e < mm * kBN; e += C::kThreads) {
            const int nl = e / mm;
            const int mi = e - nl * mm;
            const int owner = nl / rows_per;
            const uint32_t off = static_cast<uint32_t>(((nl - owner * rows_per) * C::kRedStride + mi) * 4);
            dsmem_st_f32(dsmem_map(recv_base + off, static_cast<uint32_t>(owner)), red[nl * C::kRedStride + mi]);
        }
    }
    cluster_sync_all();
    const int r_begin = rank * rows_per;
    const int r_end = min(kBN, r_begin + rows_per);
    const int my_rows = max(0, r_end - r_begin);
    for (int e = threadIdx.x; e < mm * my_rows; e += C::kThreads) {
        const int mi = e / my_rows;
        const int rl = e - mi * my_rows;
        const int nn = n0 + r_begin + rl;
        const int64_t oi = nn < n ? out_at(mi, nn, n) : -1;
        if (oi < 0) continue;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
            if (q < splits) sum += recv[(q * rows_per + rl) * C::kRedStride + mi];
        y[oi] = __float2bfloat16_rn(ROW ? sum * __ldg(scales + static_cast<int64_t>(nn) * row_stride) : sum);
    }
}

template <int MT, int SC, bool F16, bool MOE = false, bool XP = false>
__global__ void __launch_bounds__(Cfg<MT, SC == kScaleMx, F16, XP>::kThreads,
                                  Cfg<MT, SC == kScaleMx, F16, XP>::kMinBlocks)
    decode_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_x,
                  const float *__restrict__ scales, const uint8_t *__restrict__ e8m0, __nv_bfloat16 *__restrict__ y,
                  int m, int n, int kblocks, int groups, int splits, int ntiles, int e8m0_vec, int row_stride,
                  const int32_t *__restrict__ ids, int topk, int num_experts, const float *__restrict__ xinv,
                  MoeGroups mg) {
    decode_body<MT, SC, F16, MOE, false, XP>(nullptr, xinv, &tm_codes, &tm_x, scales, e8m0, y, m, n, kblocks, groups,
                                             splits, ntiles, e8m0_vec, row_stride, ids, topk, num_experts, mg);
}

// A batch of independent GEMVs with the same m in one persistent launch
// (XP: every op's x prepared, BatchOp::xinv set).
template <int MT, int SC, bool F16, bool XP = false>
__global__ void __launch_bounds__(Cfg<MT, SC == kScaleMx, F16, XP>::kThreads,
                                  Cfg<MT, SC == kScaleMx, F16, XP>::kMinBlocks)
    gemv_batch_kernel(const __grid_constant__ BatchParams p, int m) {
    decode_body<MT, SC, F16, false, true, XP>(&p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, m, 0, 0, 0,
                                              1, 0, 0, 0, nullptr, 0, 0);
}

// ------------------------------------------------------------ x preparation
// One warp per (row r < mpad, 128-column K block kb) of x bf16 [m, k]:
// x16[r, kb*128 ..] = f16(x * 2^e), with the power of two 2^e that moves the
// block's largest |x| into [2^14, 2^15) -- the converter warp's rescale,
// done once per call instead of once per CTA -- and
// inv[kb * 32 + slot(r)] = 2^-e in the slot order the consumer warps read.
// Padding rows r in [m, mpad) get inv = 1 (their x rows load as zeros).
__device__ __forceinline__ void xprep_warp(const uint16_t *__restrict__ x, int m, int mpad, int k, int kblocks,
                                           uint16_t *__restrict__ x16, float *__restrict__ inv, int w, int lane) {
    const int r = w / kblocks, kb = w - r * kblocks;
    if (r >= mpad) return;
    const int c = kb * kKB + lane * 4;
    const bool in = r < m && c < k;  // k % 4 == 0: a lane's four values are all in or all out
    uint2 v = make_uint2(0u, 0u);
    if (in) v = *reinterpret_cast<const uint2 *>(x + static_cast<int64_t>(r) * k + c);
    const uint32_t mx = max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);  // |max| as bf16 bits
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, o));
    const int e = f16_rescale_exp(m16);
    const float mult = pow2_int(e);
    if (in) {
        uint2 o;
        o.x = f32x2_to_f16x2(bf16lo_to_f32(v.x) * mult, bf16hi_to_f32(v.x) * mult);
        o.y = f32x2_to_f16x2(bf16lo_to_f32(v.y) * mult, bf16hi_to_f32(v.y) * mult);
        *reinterpret_cast<uint2 *>(x16 + static_cast<int64_t>(r) * k + c) = o;
    }
    if (lane == 0)
        inv[kb * 32 + xinv_slot(r)] = r < m ? pow2_int(-e) : 1.0f;
}

__global__ void __launch_bounds__(256) xprep_kernel(const uint16_t *__restrict__ x, int m, int mpad, int k,
                                                    int kblocks, uint16_t *__restrict__ x16,
                                                    float *__restrict__ inv) {
    pdl_launch_dependents();  // the GEMV's prologue may start; it waits for this grid before reading
    pdl_wait();               // x may come from the previous kernel in the stream
    const int gw = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    xprep_warp(x, m, mpad, k, kblocks, x16, inv, gw, threadIdx.x & 31);
}

// Per-device, per-instantiation launch setup (shared-memory opt-in and the
// number of CTAs that fit on one SM), done once on first use.
struct Setup {
    std::mutex mu;
    bool done[64] = {};
    cudaError_t err[64] = {};
    int resident[64] = {};
    ClusterFit fit;
};

// Shared-memory opt-in and resident CTAs per SM of one kernel instantiation
// on the current device (done once per device).
cudaError_t setup_once(Setup &setup, const void *kern, int threads, int smem, int &resident) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(setup.mu);
    if (!setup.done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int blocks = 0;
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, threads, smem);
        setup.err[dev] = e;
        setup.resident[dev] = blocks > 0 ? blocks : 1;
        setup.done[dev] = true;
    }
    resident = setup.resident[dev];
    return setup.err[dev];
}

// XP: a.x is the prepared f16 copy of x and xinv its inverse factors
// (launch_decode_xprep).
template <int MT, int SC, bool F16, bool XP = false>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t stream, const float *xinv = nullptr) {
    using C = Cfg<MT, SC == kScaleMx, F16, XP>;
    constexpr int kBN = C::kBN;
    auto kern = decode_kernel<MT, SC, F16, false, XP>;
    static Setup setup;
    int resident = 1;
    {
        const cudaError_t e =
            setup_once(setup, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes, resident);
        if (e != cudaSuccess) return e;
    }

    CUtensorMap tm_codes, tm_x;
    const uint64_t n = static_cast<uint64_t>(a.n), k = static_cast<uint64_t>(a.k),
                   m = static_cast<uint64_t>(a.m);
    if (!encode_tensor_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, k, n, k, kKB, kBN,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&tm_x, XP ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x,
                              k, m, k * 2, 64, C::kXRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const int ntiles = static_cast<int>((a.n + kBN - 1) / kBN);
    const int groups = static_cast<int>((a.k + 31) / 32);
    const int capacity = device_sm_count() * resident;
    const int e8m0_vec = (groups % 4 == 0 && (reinterpret_cast<uintptr_t>(a.e8m0) & 3) == 0) ? 1 : 0;
    int splits = 1;
    if (ntiles < capacity) {
        // as many K splits as fill the SMs, but only a cluster size whose
        // clusters all fit at once (a second wave would cost more)
        int cap = capacity / ntiles;
        if (cap > kMaxSplit) cap = kMaxSplit;
        if (cap > kblocks) cap = kblocks;
        splits = pick_split(setup.fit, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes, ntiles, cap);
    }
    // splits == 1: persistent grid; splits > 1: one CTA per (row tile, split)
    const int gx = splits == 1 ? (ntiles < capacity ? ntiles : capacity) : ntiles;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(splits), 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, tm_codes, tm_x, a.scales, a.e8m0,
                              static_cast<__nv_bfloat16 *>(a.y), static_cast<int>(a.m),
                              static_cast<int>(a.n), kblocks, groups, splits, ntiles, e8m0_vec, a.row_stride,
                              static_cast<const int32_t *>(nullptr), 0, 0, xinv, MoeGroups{nullptr, nullptr, nullptr});
}

// A batch launch: one persistent grid over the row tiles of all the ops
// (XP: every op's x is its prepared f16 copy, with BatchItem::xinv set).
template <int MT, int SC, bool F16, bool XP = false>
cudaError_t launch_batch_t(const BatchItem *ops, int count, int64_t m, bool force, cudaStream_t stream) {
    using C = Cfg<MT, SC == kScaleMx, F16, XP>;
    constexpr int kBN = C::kBN;
    auto kern = gemv_batch_kernel<MT, SC, F16, XP>;
    static Setup setup;
    int resident = 1;
    {
        const cudaError_t e =
            setup_once(setup, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes, resident);
        if (e != cudaSuccess) return e;
    }
    int64_t units = 0;
    for (int i = 0; i < count; ++i) units += (ops[i].n + kBN - 1) / kBN;
    const int capacity = device_sm_count() * resident;
    // One op, or too few row tiles to keep the SMs streaming with whole-K
    // units: the single-weight launches (split-K clusters) do better.
    if (!force && (count == 1 || units * 2 < capacity)) {
        for (int i = 0; i < count; ++i) {
            DecodeArgs a{ops[i].x, ops[i].codes, SC == kScaleMx ? nullptr : static_cast<const float *>(ops[i].scales),
                         SC == kScaleMx ? static_cast<const uint8_t *>(ops[i].scales) : nullptr,
                         ops[i].y, m, ops[i].n, ops[i].k, static_cast<ScaleKind>(SC), 0};
            const cudaError_t e = launch_t<MT, SC, F16, XP>(a, stream, ops[i].xinv);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (units >= (int64_t{1} << 31)) return cudaErrorInvalidValue;

    BatchParams p;
    memset(&p, 0, sizeof p);
    int unit0 = 0;
    for (int i = 0; i < count; ++i) {
        const BatchItem &it = ops[i];
        BatchOp &o = p.ops[i];
        const uint64_t n = static_cast<uint64_t>(it.n), k = static_cast<uint64_t>(it.k);
        if (!encode_tensor_map_2d(&p.tm_codes[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, it.codes, k, n, k, kKB, kBN,
                                  CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tensor_map_2d(&p.tm_x[i], XP ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                  it.x, k, static_cast<uint64_t>(m), k * 2, 64, C::kXRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        o.xinv = it.xinv;
        o.scales = SC == kScaleMx ? nullptr : static_cast<const float *>(it.scales);
        o.e8m0 = SC == kScaleMx ? static_cast<const uint8_t *>(it.scales) : nullptr;
        o.y = static_cast<__nv_bfloat16 *>(it.y);
        o.n = static_cast<int>(it.n);
        o.kblocks = static_cast<int>((it.k + kKB - 1) / kKB);
        o.groups = static_cast<int>((it.k + 31) / 32);
        o.ntiles = static_cast<int>((it.n + kBN - 1) / kBN);
        o.unit0 = unit0;
        unit0 += o.ntiles;
        o.e8m0_vec = (o.groups % 4 == 0 && (reinterpret_cast<uintptr_t>(o.e8m0) & 3) == 0) ? 1 : 0;
        o.row_stride = 0;
    }
    p.count = count;
    p.units = unit0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(unit0 < capacity ? unit0 : capacity), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, static_cast<int>(m));
}

// Grouped MoE launch: grid (row tiles of one expert, K splits, expert slots).
template <int MT, bool F16>
cudaError_t launch_moe_t(const DecodeArgs &a, const MoeArgs &g, cudaStream_t stream) {
    using C = Cfg<MT, false, F16>;
    constexpr int kBN = C::kBN;
    auto kern = decode_kernel<MT, kScaleBlock, F16, true>;
    static Setup setup;
    int resident = 1;
    {
        const cudaError_t e =
            setup_once(setup, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes, resident);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm_codes, tm_x;
    const uint64_t rows = static_cast<uint64_t>(g.num_experts) * static_cast<uint64_t>(a.n);
    const uint64_t k = static_cast<uint64_t>(a.k), m = static_cast<uint64_t>(a.m);
    if (!encode_tensor_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, k, rows, k, kKB, kBN,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, k, m, k * 2, 64, C::kXRows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const int ntiles = static_cast<int>((a.n + kBN - 1) / kBN);
    const int64_t slots64 = a.m * g.topk < g.num_experts ? a.m * g.topk : g.num_experts;
    const int slots = static_cast<int>(slots64);
    // size the K split for the most tiles the call can have (every slot used)
    const int capacity = device_sm_count() * resident;
    int splits = 1;
    if (static_cast<int64_t>(ntiles) * slots < capacity) {
        int cap = capacity / (ntiles * slots);
        if (cap > kMaxSplit) cap = kMaxSplit;
        if (cap > kblocks) cap = kblocks;
        splits = pick_split(setup.fit, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes,
                            ntiles * slots, cap);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ntiles), static_cast<unsigned>(splits), static_cast<unsigned>(slots));
    cfg.blockDim = dim3(C::kThreads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, tm_codes, tm_x, a.scales, static_cast<const uint8_t *>(nullptr),
                              static_cast<__nv_bfloat16 *>(a.y), static_cast<int>(a.m), static_cast<int>(a.n),
                              kblocks, 0, splits, ntiles, 0, 0, g.ids, static_cast<int>(g.topk),
                              static_cast<int>(g.num_experts), static_cast<const float *>(nullptr),
                              MoeGroups{nullptr, nullptr, nullptr});
}


template <int SC>
cudaError_t launch_sc(const DecodeArgs &a, cudaStream_t stream) {
    // f16 operands (converter warp) for m <= 8, bf16 for wider x: beyond
    // eight rows one converter warp cannot keep up (lm_head M = 16: 129 us
    // with f16, 113 with bf16; MXFP8 M = 32: 62 us with f16, 46 with bf16)
    switch ((a.m + 7) / 8) {
        case 1: return launch_t<1, SC, true>(a, stream);
        case 2: return launch_t<2, SC, false>(a, stream);
        case 3: return launch_t<3, SC, false>(a, stream);
        case 4: return launch_t<4, SC, false>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int SC>
cudaError_t launch_batch_sc(const BatchItem *ops, int count, int64_t m, bool force, cudaStream_t stream) {
    switch ((m + 7) / 8) {
        case 1: return launch_batch_t<1, SC, true>(ops, count, m, force, stream);
        case 2: return launch_batch_t<2, SC, false>(ops, count, m, force, stream);
        case 3: return launch_batch_t<3, SC, false>(ops, count, m, force, stream);
        case 4: return launch_batch_t<4, SC, false>(ops, count, m, force, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_moe_decode(const DecodeArgs &a, const MoeArgs &g, cudaStream_t stream) {
    switch ((a.m + 7) / 8) {
        case 1: return launch_moe_t<1, true>(a, g, stream);
        case 2: return launch_moe_t<2, false>(a, g, stream);
        case 3: return launch_moe_t<3, false>(a, g, stream);
        case 4: return launch_moe_t<4, false>(a, g, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Grouped MoE by the routing's expert tiles (m > 32 with few pairs per
// expert): the same kernel at 32 x rows, grid (row tiles of one expert, K
// splits, expert tiles); each expert's weight streams once per tile of up to
// kMoeDecodeTile of its pairs, whose x rows the routing copied in pair order.
cudaError_t launch_moe_grouped(const DecodeArgs &a, const MoeArgs &g, const MoeRoute &r, cudaStream_t stream) {
    constexpr int MT = kMoeDecodeTile / 8;
    using C = Cfg<MT, false, true, true>;
    static_assert(C::kXRows == kMoeDecodeTile, "one expert tile is the kernel's staged x rows");
    constexpr int kBN = C::kBN;
    // f16 operands: the routing wrote the x copy rescaled, with each tile's
    // inverse factors (one cvt per code pair instead of a 4-op bf16 decode)
    auto kern = decode_kernel<MT, kScaleBlock, true, true, true>;
    static Setup setup;
    int resident = 1;
    {
        const cudaError_t e =
            setup_once(setup, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes, resident);
        if (e != cudaSuccess) return e;
    }
    const int64_t pairs = a.m * g.topk;
    const int64_t tbound = moe_decode_tile_bound(pairs, g.num_experts);
    if (tbound > 65535 || r.xinv == nullptr) return cudaErrorInvalidValue;
    CUtensorMap tm_codes, tm_x;
    const uint64_t rows = static_cast<uint64_t>(g.num_experts) * static_cast<uint64_t>(a.n);
    const uint64_t k = static_cast<uint64_t>(a.k);
    if (!encode_tensor_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, k, rows, k, kKB, kBN,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, r.xs, k, static_cast<uint64_t>(pairs), k * 2,
                              64, C::kXRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const int ntiles = static_cast<int>((a.n + kBN - 1) / kBN);
    // size the K split for the expert tiles the routing is expected to make
    // (one per selected expert and 32 pairs), not for the bound
    const int64_t expect64 = (pairs + kMoeDecodeTile - 1) / kMoeDecodeTile;
    const int expect = static_cast<int>(expect64 < g.num_experts ? g.num_experts : expect64);
    const int capacity = device_sm_count() * resident;
    int splits = 1;
    if (static_cast<int64_t>(ntiles) * expect < capacity) {
        int cap = capacity / (ntiles * expect);
        if (cap > kMaxSplit) cap = kMaxSplit;
        if (cap > kblocks) cap = kblocks;
        splits = pick_split(setup.fit, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes,
                            ntiles * expect, cap);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ntiles), static_cast<unsigned>(splits), static_cast<unsigned>(tbound));
    cfg.blockDim = dim3(C::kThreads, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, tm_codes, tm_x, a.scales, static_cast<const uint8_t *>(nullptr),
                              static_cast<__nv_bfloat16 *>(a.y), kMoeDecodeTile, static_cast<int>(a.n), kblocks, 0,
                              splits, ntiles, 0, 0, static_cast<const int32_t *>(nullptr), static_cast<int>(g.topk),
                              static_cast<int>(g.num_experts), static_cast<const float *>(r.xinv),
                              MoeGroups{r.tile_off_dec, r.tile_info_dec, r.perm});
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    switch (a.kind) {
        case kScaleBlock: return launch_sc<kScaleBlock>(a, stream);
        case kScaleMx: return launch_sc<kScaleMx>(a, stream);
        case kScaleRow: return launch_sc<kScaleRow>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_batch(const BatchItem *ops, int count, int64_t m, ScaleKind kind, bool force,
                                cudaStream_t stream) {
    if (count <= 0 || count > kBatchMaxOps || m <= 0 || m > 32) return cudaErrorInvalidValue;
    switch (kind) {
        case kScaleBlock: return launch_batch_sc<kScaleBlock>(ops, count, m, force, stream);
        case kScaleMx: return launch_batch_sc<kScaleMx>(ops, count, m, force, stream);
        default: return cudaErrorInvalidValue;
    }
}

int64_t xprep_bytes(int64_t m, int64_t k) {
    const int64_t x16 = (2 * m * k + 255) / 256 * 256;
    return x16 + 128 * ((k + kKB - 1) / kKB);
}

cudaError_t launch_decode_xprep(const DecodeArgs &a, void *workspace, cudaStream_t stream) {
    if (a.kind != kScaleBlock || a.m < 1 || a.m > 32) return cudaErrorInvalidValue;
    const int mt = static_cast<int>((a.m + 7) / 8);
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    uint16_t *x16 = static_cast<uint16_t *>(workspace);
    float *inv = reinterpret_cast<float *>(static_cast<char *>(workspace) + (2 * a.m * a.k + 255) / 256 * 256);
    const int mpad = 8 * mt;
    const int64_t warps = static_cast<int64_t>(mpad) * kblocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, xprep_kernel, static_cast<const uint16_t *>(a.x),
                                       static_cast<int>(a.m), mpad, static_cast<int>(a.k), kblocks, x16, inv);
    if (e != cudaSuccess) return e;
    DecodeArgs b = a;
    b.x = x16;
    switch (mt) {
        case 1: return launch_t<1, kScaleBlock, true, true>(b, stream, inv);
        case 2: return launch_t<2, kScaleBlock, true, true>(b, stream, inv);
        case 3: return launch_t<3, kScaleBlock, true, true>(b, stream, inv);
        default: return launch_t<4, kScaleBlock, true, true>(b, stream, inv);
    }
}

// One thread waits, with the same bounded wait every pipelined kernel uses,
// on an mbarrier whose phase nothing completes; when the bound expires it
// records ERRBIT_FULL_WAIT in the decode error word and returns.
__global__ void wait_expiry_kernel() {
    __shared__ uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    if (!mbar_wait_bounded(&bar, 0)) atomicOr(&g_decode_err, ERRBIT_FULL_WAIT);
}

cudaError_t launch_wait_expiry_probe(cudaStream_t stream) {
    wait_expiry_kernel<<<1, 1, 0, stream>>>();
    return cudaGetLastError();
}

uint32_t take_decode_error() {
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_err, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_decode_err, &zero, sizeof zero);
    return v;
}

}  // namespace fp8bs
