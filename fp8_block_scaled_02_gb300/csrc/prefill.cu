// prefill.cu -- block-FP8 / per-row FP8 W8A16 GEMM for prefill-shaped
// batches on the 5th-generation tensor cores (tcgen05),
// y[M, N] = x[M, K] . dequant(W)^T.
//
// Design (sm_103a, one CTA per 128 weight rows x 256 rows of x, 20 warps):
//  * Weights are the MMA's A operand.  A producer thread brings each K
//    block's 128 x 128 e4m3 codes with 2-D TMA (128-byte swizzle) into a
//    two-stage shared-memory ring, and for weights read from HBM asks L2
//    for the codes several K blocks further ahead.  Eight "decoder" warps
//    (each thread one weight row and one 64-wide K half) read their codes
//    from the ring, free the stage, convert them exactly to bf16 pairs in
//    registers and store them into a double-buffered shared-memory A slot
//    in the 128-byte-swizzled K-major layout the tensor core reads.  The
//    decoded weight never reaches HBM, and each decoded 128 x 128 block
//    feeds all 256 rows of x.  (Loading codes straight into the decoders'
//    registers, one K block ahead, left each decoder waiting a full memory
//    latency per K block: 16 KB in flight per SM.)
//  * x is the B operand: one producer thread brings each K block's 256 x
//    rows with 2-D TMA (128-byte swizzle, two 64-column panels) into a
//    two-stage 128 KB shared-memory ring.
//  * One thread issues tcgen05.mma.kind::f16 (bf16 x bf16 -> fp32, M=128,
//    N=256, K=16, 8 per K block, both operands from shared memory) into the
//    K block's own 256-column TMEM partial D_{kb & 1}, and one
//    tcgen05.commit per K block into a ring of "MMA done" barriers that
//    frees x stages and A slots alike.  Consecutive K blocks write different
//    partials, so the tensor core never waits on its own accumulator, and
//    the MMAs of K block kb + 1 overlap the promotion of K block kb.
//  * MXFP8 (one e8m0 exponent E per 32 K of a row): the decoders fold each
//    group's 2^(E-127) into the exact bf16 decode -- dec(q) * 2^(E-127) is
//    itself a bf16 value whenever 3 <= E <= 134 (at most four significant
//    bits, exponent in range), and above 134 after a second exact multiply
//    -- so the partials need no promotion and the epilogue sums them as they
//    are.  Only groups with E < 3 (amax below 2^-116) lose exactness: their
//    weights round to bf16's subnormal grid (|error| <= 2^-134 each).
//  * Eight epilogue warps (one per TMEM lane quarter and 128-column half)
//    read each partial with tcgen05.ld and add it, multiplied by the K
//    block's fp32 scale, into running totals held in their registers
//    ("promotion": the scale is applied once per 128-wide K block to an fp32
//    partial and never folded into a rounded bf16 weight).  With one scale
//    per weight row (or per tensor) the partials are summed unscaled and the
//    row's scale multiplies the fp32 total once, before the bf16 rounding.
//  * 128 totals per thread need more registers than an even split of the
//    register file gives 640 threads, so the warpgroups trade registers at
//    start (setmaxnreg): decoders and the control warpgroup give some up,
//    the epilogue warpgroups take them.
//  * Every wait is bounded; a kernel that gives up sets an error word,
//    drains what it issued and still frees its TMEM.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

#include <mutex>

namespace fp8bs {

namespace {

__device__ uint32_t g_prefill_err;

constexpr int kTileW = 128;                 // weight rows per CTA (= one scale row block, = MMA M)
constexpr int kKB = 128;                    // K per block
constexpr int kPanel = 128 * 128;           // one 64-column bf16 panel of 128 weight rows, 16 KB
constexpr int kASlots = 2;                  // decoded weight blocks in flight
constexpr int kASlot = 2 * kPanel;          // 32 KB
constexpr int kCStage = kTileW * kKB;      // one K block of e4m3 codes, 16 KB
constexpr int kRing = 8;  // MMA-completion barriers, one per K block; >= every look-back

// The geometry of a CTA with TX x rows (same 225 KB of shared memory in
// both forms).
//  TX = 256 (dense, and the grouped MoE with many pairs per expert): the
//  MMA's N up to 256, a two-stage x ring of 64 KB stages, a two-stage codes
//  ring; partials D_0, D_1 in TMEM columns [0, 256) and [256, 512).
//  TX = 128 (the grouped MoE with up to ~128 pairs per expert; its MMAs run
//  N = pairs rounded up to 16): the x stage is 32 KB and the space buys
//  depth, a four-stage x ring.  Each such CTA streams its own expert rows
//  from HBM, which no other CTA shares, with one CTA per SM: clock stamps of
//  the two-stage form showed each load landing 2600-4100 cycles after its
//  issue and a K block every ~2000 cycles, a ring's round trip.  Measured
//  against a three-stage x ring with four codes stages: 810 vs 820 us (256
//  experts, 96 pairs each); deeper codes rings or L2 prefetch gained
//  nothing.  Partials in columns [0, 128), [128, 256).
template <int TX>
struct Geo {
    static_assert(TX == 256 || TX == 128, "two geometries");
    static constexpr int kTileX = TX;                // x rows per CTA
    static constexpr int kHalfX = kTileX / 2;        // x rows (TMEM columns) per epilogue half
    static constexpr int kXPanel = kTileX * 128;     // one 64-column bf16 panel of the x rows
    static constexpr int kXStage = 2 * kXPanel;      // one K block of x
    static constexpr int kXStages = TX == 128 ? 4 : 2;
    static constexpr int kXBytes = kXStages * kXStage;
    static constexpr int kCStages = 2;                     // codes ring
    static constexpr int kCodesAhead = TX == 128 ? 6 : 4;  // L2 prefetch distance (K blocks past the load)
    static constexpr int kTmemCols = 2 * kTileX;     // partials D_0, D_1
    static constexpr int kSmemBytes = 1024 + kXBytes + kASlots * kASlot + kCStages * kCStage + 256;
    static_assert(kXStages <= kRing && kASlots <= kRing, "a wait must never reach back a full ring");
    static_assert(kSmemBytes + 4 * kTileX + 64 <= 227 * 1024, "shared memory per CTA (with the static arrays)");
    static_assert(kCodesAhead >= kCStages, "the L2 prefetch runs at or past the loads");
};

// 20 warps in 5 warpgroups (a warpgroup's warps all take the same register
// count):
//   warpgroups 0-1 (warps 0-7)  decoders: weight rows 32 (warp % 4) .. +31,
//                               K half warp / 4;
//   warpgroups 2-3 (warps 8-15) epilogue: TMEM lane quarter warp % 4, half
//                               (warp - 8) / 4, 128 fp32 totals per thread;
//   warpgroup 4   (warps 16-19) MMA issuer (+ TMEM), x producer, codes
//                               producer, one idle.
constexpr int kNumDec = 8;
constexpr int kNumEpi = 8;
constexpr int kWarpEpi0 = kNumDec;
constexpr int kWarpMma = kWarpEpi0 + kNumEpi;
constexpr int kWarpTma = kWarpMma + 1;
constexpr int kWarpCodes = kWarpMma + 2;
constexpr int kThreads = (kWarpMma + 4) * 32;
constexpr int kRegCtl = 40, kRegDec = 64, kRegEpi = 152;
// The split must fit in what the block is launched with (the launcher checks
// the compiled count against kRegLaunch before the first launch).
constexpr int kRegLaunch = 96;
static_assert(4 * 32 * kRegCtl + kNumDec * 32 * kRegDec + kNumEpi * 32 * kRegEpi <= kThreads * kRegLaunch,
              "register split exceeds the launch allocation");
static_assert(kThreads * kRegLaunch <= 65536, "launch allocation exceeds the register file");
static_assert(kRegCtl % 8 == 0 && kRegDec % 8 == 0 && kRegEpi % 8 == 0, "setmaxnreg counts are multiples of 8");
static_assert(kNumDec % 4 == 0 && kNumEpi % 4 == 0, "roles must fill whole warpgroups");

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_n(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(kTileW >> 4) << 24);
}
template <int N>
__host__ __device__ constexpr uint32_t idesc_f16() {
    return idesc_f16_n(N);
}

// MOE: x rows per TMA box.  A tile loads only the boxes that hold its pairs
// (an expert's tile often holds fewer than 128); stacked at 4 KB steps the
// boxes give the layout of one 128-row box.
constexpr int kMoeXBox = 32;

__device__ __forceinline__ void fail(uint32_t bit) { atomicOr(&g_prefill_err, bit); }

// Both operands from shared memory; the instruction descriptor in a register
// (MOE: N = the tile's pairs rounded up to 16).
__device__ __forceinline__ void tc_mma_ss_r(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(idesc)
        : "memory");
}

// Both operands from shared memory.
template <uint32_t kIdesc>
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(accumulate), "n"(kIdesc)
        : "memory");
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// The grouped MoE form: the routing (moe.cu) in device memory.
struct MoeTiles {
    const int32_t *tile_off;  // [E + 1] first GEMM tile of each expert
    const int4 *tile_info;    // [tile bound] {expert, first pair, pairs, 0} of each tile
    const int32_t *perm;      // pairs t * topk + j, expert by expert
    int topk, num_experts;
};

// SC: kScaleBlock (128x128 block scales, promoted per K block), kScaleRow
// (scales[row * row_stride] per weight row, stride 0: one per tensor,
// applied to the total) or kScaleMx (e8m0 [n, groups], folded into the
// decoded weights).
// MOE: grouped GEMM over routed experts (block scales).  blockIdx.y is a
// tile of up to TX (token, slot) pairs of one expert (CTAs past the last
// tile leave at once), blockIdx.x a 128-row tile of that expert's weight
// (codes [E * n, k], scales [E, ceil(n/128), kblocks]).  tm_x maps the x
// rows copied in pair order (moe.cu: xs [pairs, k]) in boxes of kMoeXBox
// rows, so a tile's rows are ordinary TMA boxes starting at its first pair;
// output row j goes to y[pair_j * n + row] (y: [tokens, topk, n]).  The
// tile's work follows its pair count: only the boxes holding its pairs are
// loaded, the MMAs run N = pairs rounded up to 16, and the epilogue reads
// only those TMEM columns.
template <int SC, bool MOE = false, int TX = 256>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                              const __grid_constant__ CUtensorMap tm_codes,
                                                              const float *__restrict__ scales,
                                                              const uint8_t *__restrict__ e8m0, int groups,
                                                              __nv_bfloat16 *__restrict__ y, int m, int n,
                                                              int k, int kblocks, int row_stride, int xfast,
                                                              int fast, int tile0, int ksplit, int pdl_mode,
                                                              MoeTiles moe) {
    constexpr bool ROW = SC == kScaleRow;
    constexpr bool MX = SC == kScaleMx;
    static_assert(!MOE || SC == kScaleBlock, "the grouped GEMM takes block scales");
    static_assert(MOE || TX == 256, "the dense form has 256 x rows per CTA");
    using G = Geo<TX>;
    constexpr int kTileX = G::kTileX, kHalfX = G::kHalfX, kXPanel = G::kXPanel, kXStage = G::kXStage,
                  kXStages = G::kXStages, kXBytes = G::kXBytes, kCStages = G::kCStages,
                  kCodesAhead = G::kCodesAhead, kTmemCols = G::kTmemCols;
    __shared__ int32_t s_pair[MOE ? kTileX : 1];  // MOE: this tile's pairs, -1 past its count
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *xring = smem;                              // [kXStages][2 panels][kTileX rows][128 B]
    uint8_t *aring = smem + kXBytes;                    // [kASlots][2 panels][128 rows][128 B]
    uint8_t *cring = aring + kASlots * kASlot;          // [kCStages][128 rows][128 B] codes
    uint64_t *bars = reinterpret_cast<uint64_t *>(cring + kCStages * kCStage);
    uint64_t *x_full = bars;                 // [kXStages]
    uint64_t *done = x_full + kXStages;      // [kRing] MMAs of K block kb finished
    uint64_t *a_full = done + kRing;         // [kASlots]
    uint64_t *d_empty = a_full + kASlots;    // [2] partial D_b read by every epilogue warp
    uint64_t *c_full = d_empty + 2;          // [kCStages] codes landed
    uint64_t *c_empty = c_full + kCStages;   // [kCStages] codes read by every decoder warp
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(c_empty + kCStages);
    int *s_fail = reinterpret_cast<int *>(c_empty + kCStages + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool deep_prefetch = MOE || xfast;
    // Tile order (dense: blockIdx.x is a linear index, tile t = tile0 +
    // blockIdx.x / ksplit, `fast` tiles along its fastest dimension).  xfast:
    // consecutive tiles walk the x tiles of one weight tile, so the CTAs
    // running at any one time share a few weight tiles and their code loads
    // hit L2 even when the weight does not fit there; otherwise they walk the
    // weight tiles of one x tile, which keeps a weight that fits in L2
    // together with one x tile there.  ksplit > 1 (the last, partial wave of
    // a call): the ksplit CTAs of a cluster share one tile, each taking a
    // contiguous range of its K blocks.  MOE: blockIdx.x = weight tile,
    // blockIdx.y = expert tile.
    int wtile, ksp = 0;
    int m0;  // MOE: the tile's first pair
    if (MOE) {
        wtile = blockIdx.x;
        m0 = blockIdx.y * kTileX;
    } else {
        const int t = tile0 + static_cast<int>(blockIdx.x) / ksplit;
        ksp = static_cast<int>(blockIdx.x) % ksplit;
        const int a = t % fast, b = t / fast;
        wtile = xfast ? b : a;
        m0 = (xfast ? a : b) * kTileX;
    }
    const int n0 = wtile * kTileW;
    // this CTA's K blocks [kb0, kb0 + nkb)
    const int kb0 = ksp * kblocks / ksplit;
    const int nkb = (ksp + 1) * kblocks / ksplit - kb0;

    int expert = 0;
    int live = kTileX;  // MOE: this tile's pairs
    int srow_moe = 0;   // MOE: this CTA's row of block scales
    if (MOE) {
        // this CTA's expert and pairs (the routing kernels ran before it in
        // the stream): the tile count and the tile's record, two independent
        // loads; every thread reads the same words, so the exit is uniform
        // and happens before anything is allocated
        const int tile = blockIdx.y;
        const int ntiles = __ldg(moe.tile_off + moe.num_experts);
        const int4 ti = __ldg(moe.tile_info + tile);  // in bounds (the grid's bound); used if tile < ntiles
        if (tile >= ntiles) return;
        expert = ti.x;
        m0 = ti.y;
        live = ti.z;
        srow_moe = expert * ((n + kTileW - 1) / kTileW) + wtile;
        for (int i = threadIdx.x; i < kTileX; i += blockDim.x) s_pair[i] = i < live ? __ldg(moe.perm + m0 + i) : -1;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kXStages; ++i) mbar_init(&x_full[i], 1);
        for (int i = 0; i < kRing; ++i) mbar_init(&done[i], 1);  // tcgen05.commit
        for (int i = 0; i < kASlots; ++i) mbar_init(&a_full[i], kNumDec);
        for (int i = 0; i < 2; ++i) mbar_init(&d_empty[i], kNumEpi);
        for (int i = 0; i < kCStages; ++i) {
            mbar_init(&c_full[i], 1);
            mbar_init(&c_empty[i], kNumDec);
        }
        *s_fail = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpTma && lane == 0) prefetch_tensormap(&tm_x);
    if (warp == kWarpCodes && lane == 0) prefetch_tensormap(&tm_codes);
    if (warp == kWarpMma) tc_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int wg = warp >> 2;
    // Programmatic dependent launch.  pdl_mode 0: wait for the previous
    // kernel, let the next one launch at the end.  1 (the full waves of a call
    // whose last wave runs split): wait, then let the split launch start at
    // once, so that its CTAs take SMs as this launch's last wave frees them.
    // 2 (that split launch): its tiles do not depend on the full waves and
    // its inputs were complete before they started, so it waits only at the
    // end, before it lets the next kernel go, so that the call is complete
    // when the next kernel's wait returns.
    if (pdl_mode != 2) pdl_wait();
    if (pdl_mode == 1) pdl_launch_dependents();

    // Each role's register count is set at the top of its own branch, so
    // that the compiler allocates the branch within it.
    if (wg == kWarpMma / 4) {
        setmaxnreg_dec<kRegCtl>();
        if (warp == kWarpMma) {
            // ------------------------------------------------------ MMA issuer
            int issued = 0;
            if (lane == 0) {
                for (int kb = 0; kb < nkb; ++kb) {
                    const int xs = kb % kXStages, as = kb % kASlots, b = kb & 1;
                    bool ok = mbar_wait_bounded(&x_full[xs], (kb / kXStages) & 1) &&
                              mbar_wait_bounded(&a_full[as], (kb / kASlots) & 1) &&
                              (kb < 2 || mbar_wait_bounded(&d_empty[b], ((kb - 2) >> 1) & 1));
                    if (!ok) {
                        fail(ERRBIT_MMA_WAIT);
                        *reinterpret_cast<volatile int *>(s_fail) = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sw128_desc(smem_u32(aring + as * kASlot));
                    const uint64_t bdesc = sw128_desc(smem_u32(xring + xs * kXStage));
                    const uint32_t d_tmem = tmem + kTileX * b;
    #pragma unroll
                    for (int kk = 0; kk < kKB / 16; ++kk) {
                        const uint64_t aoff = static_cast<uint64_t>((kk >> 2) * (kPanel >> 4) + (kk & 3) * 2);
                        const uint64_t boff = static_cast<uint64_t>((kk >> 2) * (kXPanel >> 4) + (kk & 3) * 2);
                        if (MOE)
                            tc_mma_ss_r(d_tmem, adesc + aoff, bdesc + boff, idesc_f16_n((live + 15) & ~15),
                                        kk > 0 ? 1u : 0u);
                        else
                            tc_mma_ss<idesc_f16<kTileX>()>(d_tmem, adesc + aoff, bdesc + boff, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&done[kb % kRing]);
                    issued = kb + 1;
                }
                // drain: wait for the last committed block before TMEM can be freed
                if (issued > 0 && !mbar_wait_bounded(&done[(issued - 1) % kRing], ((issued - 1) / kRing) & 1))
                    fail(ERRBIT_MMA_WAIT);
            }
            __syncwarp();
        } else if (warp == kWarpTma) {
            // ------------------------------------------------------ x producer
            if (lane == 0) {
                int issued = 0;
                for (int kb = 0; kb < nkb; ++kb) {
                    const int xs = kb % kXStages;
                    const int kx = (kb0 + kb) * kKB;  // K coordinate
                    if (kb >= kXStages &&
                        !mbar_wait_bounded(&done[(kb - kXStages) % kRing], ((kb - kXStages) / kRing) & 1)) {
                        fail(ERRBIT_EMPTY_WAIT);
                        break;
                    }
                    if (*reinterpret_cast<volatile int *>(s_fail)) break;
                    uint8_t *st = xring + xs * kXStage;
                    if (MOE) {
                        // the boxes holding the tile's pairs (rows past the
                        // pairs feed only MMA columns that are never stored)
                        const int boxes = (live + kMoeXBox - 1) / kMoeXBox;
                        mbar_arrive_expect_tx(&x_full[xs], boxes * 2 * kMoeXBox * 128);
                        for (int bx = 0; bx < boxes; ++bx) {
                            tma_load_2d(st + bx * kMoeXBox * 128, &tm_x, &x_full[xs], kx, m0 + bx * kMoeXBox);
                            tma_load_2d(st + kXPanel + bx * kMoeXBox * 128, &tm_x, &x_full[xs], kx + 64,
                                        m0 + bx * kMoeXBox);
                        }
                    } else {
                        mbar_arrive_expect_tx(&x_full[xs], kXStage);
                        tma_load_2d(st, &tm_x, &x_full[xs], kx, m0);
                        tma_load_2d(st + kXPanel, &tm_x, &x_full[xs], kx + 64, m0);
                    }
                    issued = kb + 1;
                }
                // never leave with copies in flight
                for (int u = issued - kXStages < 0 ? 0 : issued - kXStages; u < issued; ++u)
                    if (!mbar_wait_bounded(&x_full[u % kXStages], (u / kXStages) & 1)) fail(ERRBIT_FULL_WAIT);
            }
            __syncwarp();
        } else if (warp == kWarpCodes) {
            // ------------------------------------------------------ codes producer
            if (lane == 0) {
                // MOE: the expert's rows start at expert * n of the stacked
                // codes (rows of a ragged last tile past n belong to the next
                // expert or lie outside the map: they only feed TMEM lanes
                // whose outputs are never stored)
                const int crow0 = (MOE ? expert * n : 0) + n0;
                int issued = 0;
                for (int kb = 0; kb < nkb; ++kb) {
                    const int cs = kb % kCStages;
                    if (kb >= kCStages &&
                        !mbar_wait_bounded(&c_empty[cs], ((kb - kCStages) / kCStages) & 1)) {
                        fail(ERRBIT_EMPTY_WAIT);
                        break;
                    }
                    if (*reinterpret_cast<volatile int *>(s_fail)) break;
                    if (deep_prefetch) {
                        // a weight read from HBM (too large for L2, or an
                        // expert read once per tile of its pairs): keep L2
                        // fetching kCodesAhead K blocks past the loads
                        if (kb == 0)
                            for (int p = kCStages; p < kCodesAhead && p < nkb; ++p)
                                tma_prefetch_l2_2d(&tm_codes, (kb0 + p) * kKB, crow0);
                        if (kb + kCodesAhead < nkb)
                            tma_prefetch_l2_2d(&tm_codes, (kb0 + kb + kCodesAhead) * kKB, crow0);
                    }
                    mbar_arrive_expect_tx(&c_full[cs], kCStage);
                    tma_load_2d(cring + cs * kCStage, &tm_codes, &c_full[cs], (kb0 + kb) * kKB, crow0);
                    issued = kb + 1;
                }
                for (int u = issued - kCStages < 0 ? 0 : issued - kCStages; u < issued; ++u)
                    if (!mbar_wait_bounded(&c_full[u % kCStages], (u / kCStages) & 1)) fail(ERRBIT_FULL_WAIT);
            }
            __syncwarp();
        }
    } else if (wg < kWarpEpi0 / 4) {
        setmaxnreg_dec<kRegDec>();
        // ------------------------------------------------------ decoders
        // thread = one weight row r; this warp converts the K half kh of
        // every K block from the codes ring
        const int r = (warp & 3) * 32 + lane;
        const int kh = warp >> 2;
        const int row = n0 + r;
        const bool row_ok = row < n;
        // MX: the row's exponents of the two 32-column groups of this K half
        // (E = 127, scale 1, past the row's groups: those codes are zero),
        // loaded four K blocks ahead into a register queue
        const uint8_t *ep = MX ? e8m0 + static_cast<int64_t>(row_ok ? row : 0) * groups + 2 * kh : nullptr;
        auto load_e = [&](int kbl) -> uint32_t {  // this CTA's K block kbl
            uint32_t e = 0x7F7Fu;
            if (MX && row_ok && kbl < nkb) {
                const int kb = kb0 + kbl;
                const int g = kb * 4 + 2 * kh;
                if (g < groups) e = (e & 0xFF00u) | __ldg(ep + kb * 4);
                if (g + 1 < groups) e = (e & 0x00FFu) | (static_cast<uint32_t>(__ldg(ep + kb * 4 + 1)) << 8);
            }
            return e;
        };
        uint32_t eq0 = load_e(0), eq1 = load_e(1), eq2 = load_e(2), eq3 = load_e(3);
        for (int kb = 0; kb < nkb; ++kb) {
            const int as = kb % kASlots, cs = kb % kCStages;
            // this K block's codes: 16 bytes at a time from the swizzled
            // rows (chunk c of row r sits at chunk c ^ (r & 7)), then the
            // stage goes back to the producer
            bool ok = mbar_wait_bounded(&c_full[cs], (kb / kCStages) & 1);
            if (!__all_sync(0xffffffffu, ok) || *reinterpret_cast<volatile int *>(s_fail)) {
                if (lane == 0) fail(ERRBIT_FULL_WAIT);
                break;
            }
            uint4 c0[4];
            const uint8_t *crow = cring + cs * kCStage + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                c0[j] = *reinterpret_cast<const uint4 *>(crow + (((4 * kh + j) ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(&c_empty[cs]);
            const uint32_t e0 = eq0;
            if (MX) {
                eq0 = eq1;
                eq1 = eq2;
                eq2 = eq3;
                eq3 = load_e(kb + 4);
            }
            // slot `as` was last read by the MMAs of K block kb - kASlots
            const int prev = kb - kASlots;
            ok = kb < kASlots || mbar_wait_bounded(&done[prev % kRing], (prev / kRing) & 1);
            if (!__all_sync(0xffffffffu, ok) || *reinterpret_cast<volatile int *>(s_fail)) {
                if (lane == 0) fail(ERRBIT_EMPTY_WAIT);
                break;
            }
            uint8_t *arow = aring + as * kASlot + kh * kPanel + r * 128;
            // decode multiplier per group: 2^120 restores the plain decode;
            // MX folds 2^(E-127) in: one multiply by 2^(E-7) when that is a
            // normal bf16 and the result exact (3 <= E <= 134), else 2^120
            // and a second multiply by 2^(E-127)
            uint32_t m1[2] = {0x7B807B80u, 0x7B807B80u}, m2[2] = {0u, 0u};
            bool two[2] = {false, false};
            if (MX) {
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    const uint32_t E = (e0 >> (8 * gi)) & 0xFFu;
                    if (E - 3u <= 131u) {
                        const uint32_t f = (E + 120u) << 7;
                        m1[gi] = f | (f << 16);
                    } else {
                        const uint32_t f = E ? E << 7 : 0x0040u;  // 2^(E-127); E = 0: subnormal 2^-127
                        m2[gi] = f | (f << 16);
                        two[gi] = true;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 c = c0[j];
                const int gi = j >> 1;  // 16 codes of one 32-column group
                uint4 lo, hi;
                lo.x = e4m3x2_to_bf16x2_mul(c.x, 0x9180u, m1[gi]);
                lo.y = e4m3x2_to_bf16x2_mul(c.x, 0xB3A2u, m1[gi]);
                lo.z = e4m3x2_to_bf16x2_mul(c.y, 0x9180u, m1[gi]);
                lo.w = e4m3x2_to_bf16x2_mul(c.y, 0xB3A2u, m1[gi]);
                hi.x = e4m3x2_to_bf16x2_mul(c.z, 0x9180u, m1[gi]);
                hi.y = e4m3x2_to_bf16x2_mul(c.z, 0xB3A2u, m1[gi]);
                hi.z = e4m3x2_to_bf16x2_mul(c.w, 0x9180u, m1[gi]);
                hi.w = e4m3x2_to_bf16x2_mul(c.w, 0xB3A2u, m1[gi]);
                if (MX && two[gi]) {
                    lo.x = mul_bf16x2(lo.x, m2[gi]);
                    lo.y = mul_bf16x2(lo.y, m2[gi]);
                    lo.z = mul_bf16x2(lo.z, m2[gi]);
                    lo.w = mul_bf16x2(lo.w, m2[gi]);
                    hi.x = mul_bf16x2(hi.x, m2[gi]);
                    hi.y = mul_bf16x2(hi.y, m2[gi]);
                    hi.z = mul_bf16x2(hi.z, m2[gi]);
                    hi.w = mul_bf16x2(hi.w, m2[gi]);
                }
                *reinterpret_cast<uint4 *>(arow + (((2 * j) ^ (r & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(arow + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
            }
            fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[as]);
        }
    } else {
        setmaxnreg_inc<kRegEpi>();
        // ------------------------------------------------------ epilogue
        // thread = one weight row (TMEM lane of quarter q); this warp owns
        // the 128 columns (rows of x) of half h of every partial D_b and
        // keeps their running totals in registers
        const int q = warp & 3;
        const int h = (warp - kWarpEpi0) >> 2;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * kHalfX;
        const int row = n0 + q * 32 + lane;
        const float *srow = (ROW || MX) ? nullptr : scales + static_cast<int64_t>(MOE ? srow_moe : wtile) * kblocks;
        const int live_cols = MOE ? live - h * kHalfX : kHalfX;  // MOE: TMEM columns the MMAs wrote
        float tot[kHalfX];
#pragma unroll
        for (int j = 0; j < kHalfX; ++j) tot[j] = 0.0f;
        bool ok = true;
        // K block scale, loaded one block ahead (1 with one scale per row:
        // the partials add unscaled).  A deeper queue spills the 128 totals.
        auto load_s = [&](int kb) -> float { return (ROW || MX || kb >= nkb) ? 1.0f : __ldg(srow + kb0 + kb); };
        float s_next = load_s(0);
        for (int kb = 0; kb < nkb; ++kb) {
            const float s = s_next;
            if (!ROW && !MX) s_next = load_s(kb + 1);
            ok = mbar_wait_bounded(&done[kb % kRing], (kb / kRing) & 1);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(ERRBIT_FULL_WAIT);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_addr = lane_base + kTileX * (kb & 1);
#pragma unroll
            for (int c = 0; c < kHalfX / 16; ++c) {
                if (MOE && 16 * c >= live_cols) break;
                uint32_t dv[16];
                tc_ld16(d_addr + 16 * c, dv);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) tot[16 * c + i] = fmaf(s, __uint_as_float(dv[i]), tot[16 * c + i]);
            }
            // D_b has been read: the MMAs of K block kb + 2 may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[kb & 1]);
        }
        if (!MOE && ksplit > 1) {
            // K split over the cluster: the CTA of rank q owns the tile's x
            // columns [q C, q C + C), C = 256 / ksplit.  Every CTA sends its
            // partial totals of each column to the owner's receive buffer
            // (its x ring, idle once every CTA's MMAs are done), laid out
            // [source rank][weight row][column] with the row's 16-byte column
            // groups XOR-swizzled by row & 7 (so that a warp's 32 rows hit
            // distinct banks); the owner sums the ksplit partials in rank
            // order and stores them.
            const int C = kTileX / ksplit;  // 32, 64 or 128
            const uint32_t rank = cluster_ctarank();
            const int r = q * 32 + lane;
            const uint32_t recv = smem_u32(xring);
            cluster_sync_all();  // every CTA of the cluster is past its MMAs
#pragma unroll
            for (int j = 0; j < kHalfX; j += 4) {
                const int col = h * kHalfX + j;
                const uint32_t dst = static_cast<uint32_t>(col / C);
                const int g = ((col % C) >> 2) ^ (r & 7);
                const uint32_t local = recv + (((rank * 128 + r) * C + (g << 2)) << 2);
                dsmem_st_f32x4(dsmem_map(local, dst), tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
            }
            cluster_sync_all();  // every partial delivered
            const float *buf = reinterpret_cast<const float *>(xring);
            const int t = (warp - kWarpEpi0) * 32 + lane;  // 0..255
            const int rr = t & 127, rowg = n0 + rr;
            const float rs = (ROW && rowg < n) ? __ldg(scales + static_cast<int64_t>(rowg) * row_stride) : 1.0f;
            for (int g = t >> 7; g < C / 4; g += 2) {
                float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                for (int src = 0; src < ksplit; ++src) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(buf + (src * 128 + rr) * C + ((g ^ (rr & 7)) << 2));
                    sum.x += v.x;
                    sum.y += v.y;
                    sum.z += v.z;
                    sum.w += v.w;
                }
                const float out[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int mi = m0 + static_cast<int>(rank) * C + 4 * g + i;
                    if (ok && rowg < n && mi < m)
                        y[static_cast<int64_t>(mi) * n + rowg] = __float2bfloat16_rn(ROW ? out[i] * rs : out[i]);
                }
            }
        } else if (ok && row < n) {
            // thread = weight row, total j = y[m0 + 128 h + j][row]
            const float rs = ROW ? __ldg(scales + static_cast<int64_t>(row) * row_stride) : 1.0f;
#pragma unroll
            for (int j = 0; j < kHalfX; ++j) {
                if (MOE) {
                    const int pr = s_pair[h * kHalfX + j];  // y row = pair index t * topk + slot
                    if (pr >= 0) y[static_cast<int64_t>(pr) * n + row] = __float2bfloat16_rn(tot[j]);
                } else {
                    const int mi = m0 + h * kHalfX + j;
                    if (mi < m) y[static_cast<int64_t>(mi) * n + row] = __float2bfloat16_rn(ROW ? tot[j] * rs : tot[j]);
                }
            }
        }
    }

    // the other warps' share of the epilogue's two cluster barriers
    if (!MOE && ksplit > 1 && (warp < kWarpEpi0 || warp >= kWarpMma)) {
        cluster_sync_all();
        cluster_sync_all();
    }
    if (pdl_mode == 2) pdl_wait();
    if (pdl_mode != 1) pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tc_dealloc(tmem, kTmemCols);
}

std::mutex g_setup_mu;
bool g_setup_done[64] = {};
cudaError_t g_setup_err[64] = {};
int g_sms[64] = {};

}  // namespace

// One-time set-up per device: shared-memory opt-in for every instantiation,
// and a check that each was compiled with the registers the setmaxnreg split
// is planned against.
static cudaError_t prefill_setup(int *sms = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_setup_done[dev]) {
            // The register split (setmaxnreg) draws on the registers the
            // block is launched with: never launch a build compiled with
            // fewer than the split was planned against (its epilogue warps
            // would wait forever for registers).
            cudaError_t e = cudaSuccess;
            using Kern = decltype(&prefill_kernel<kScaleBlock>);
            const struct {
                Kern kern;
                int smem;
            } forms[] = {{prefill_kernel<kScaleBlock>, Geo<256>::kSmemBytes},
                         {prefill_kernel<kScaleRow>, Geo<256>::kSmemBytes},
                         {prefill_kernel<kScaleMx>, Geo<256>::kSmemBytes},
                         {prefill_kernel<kScaleBlock, true, 256>, Geo<256>::kSmemBytes},
                         {prefill_kernel<kScaleBlock, true, 128>, Geo<128>::kSmemBytes}};
            for (const auto &f : forms) {
                cudaFuncAttributes fa = {};
                if (e == cudaSuccess) e = cudaFuncSetAttribute(f.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, f.smem);
                if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, f.kern);
                if (e == cudaSuccess && fa.numRegs < kRegLaunch) e = cudaErrorInvalidConfiguration;
            }
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
            g_setup_err[dev] = e;
            g_setup_done[dev] = true;
        }
        if (g_setup_err[dev] != cudaSuccess) return g_setup_err[dev];
        if (sms) *sms = g_sms[dev];
    }
    return cudaSuccess;
}

cudaError_t launch_prefill(const DecodeArgs &a, cudaStream_t stream) {
    if (a.kind != kScaleBlock && a.kind != kScaleRow && a.kind != kScaleMx) return cudaErrorNotSupported;
    int sms = 0;
    {
        const cudaError_t e = prefill_setup(&sms);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm_x;
    const uint64_t k = static_cast<uint64_t>(a.k), m = static_cast<uint64_t>(a.m);
    // one TMA box = the x rows of one MMA unit: all 256 of the CTA's rows
    constexpr int kTileX = Geo<256>::kTileX;
    constexpr int kSmemBytes = Geo<256>::kSmemBytes;
    if (!encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, k, m, k * 2, 64,
                              static_cast<uint32_t>(kTileX), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // one box = one K block of the CTA's 128 weight rows
    CUtensorMap tm_codes;
    if (!encode_tensor_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, k, static_cast<uint64_t>(a.n), k,
                              kKB, kTileW, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    // x tiles fastest when the codes are too large to stay in L2 (half of
    // its 129 MB) beside the x tiles; weight tiles fastest otherwise
    // (measured: [18432, 7168] at M = 4096 1184 us vs 1474; [12288, 4096]
    // 386 us vs 433).  A tile count past an int takes the decode kernel in
    // chunks.
    const int64_t wtiles = (a.n + kTileW - 1) / kTileW, xtiles = (a.m + kTileX - 1) / kTileX;
    const int64_t tiles = wtiles * xtiles;
    const int xfast = a.n * a.k > (int64_t{64} << 20) ? 1 : 0;
    if (tiles > INT32_MAX / 8) return cudaErrorNotSupported;
    // One CTA per SM at a time: the last wave of a call holds `rem` tiles on
    // an otherwise idle GPU.  When it fills at most half the SMs, its tiles
    // run split over K in clusters of ksplit CTAs (a power of two, at most 4:
    // a split CTA still pays a whole tile's pipeline fill and drain, and
    // eight-way splits measured slower than four-way), launched after the
    // full waves and overlapping their end.  Same-box A/B against one launch
    // of every tile: [12288, 4096] M = 512 / 2048 / 4096 59.9 / 182.0 /
    // 339.8 us vs 66.8 / 191.7 / 347.2; MXFP8 [18432, 7168] M = 4096 853 vs
    // 910 us.
    const int64_t rem = tiles % sms, full = tiles - rem;
    int ksplit = 1;
    if (rem > 0 && 2 * rem <= sms)
        while (2 * ksplit <= 4 && 2 * ksplit * rem <= sms && 2 * ksplit <= kblocks) ksplit *= 2;
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(a.y);
    const int mi = static_cast<int>(a.m), ni = static_cast<int>(a.n), ki = static_cast<int>(a.k);
    auto kern = a.kind == kScaleRow ? prefill_kernel<kScaleRow>
                                    : (a.kind == kScaleMx ? prefill_kernel<kScaleMx> : prefill_kernel<kScaleBlock>);
    const int groups = static_cast<int>((a.k + 31) / 32);
    const int fast = static_cast<int>(xfast ? xtiles : wtiles);
    const int rstride = a.kind == kScaleRow ? a.row_stride : 0;
    const MoeTiles none{nullptr, nullptr, nullptr, 0, 0};
    const int64_t main_tiles = ksplit > 1 ? full : tiles;
    const bool split = ksplit > 1;
    if (main_tiles > 0) {
        kern<<<static_cast<unsigned>(main_tiles), kThreads, kSmemBytes, stream>>>(
            tm_x, tm_codes, a.scales, a.e8m0, groups, y, mi, ni, ki, kblocks, rstride, xfast, fast, 0, 1,
            split ? 1 : 0, none);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (!split) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rem * ksplit));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = main_tiles > 0 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_codes, a.scales, a.e8m0, groups, y, mi, ni, ki, kblocks, rstride,
                              xfast, fast, static_cast<int>(full), ksplit, main_tiles > 0 ? 2 : 0, none);
}

cudaError_t launch_prefill_moe(const DecodeArgs &a, const MoeArgs &g, const MoeRoute &r, cudaStream_t stream) {
    {
        const cudaError_t e = prefill_setup();
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tm_x;
    const int64_t pairs = a.m * g.topk;
    const uint64_t k = static_cast<uint64_t>(a.k);
    // the x rows in pair order (r.xs [pairs, k]); a tile loads the boxes of
    // kMoeXBox rows that hold its pairs
    if (!encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r.xs, k, static_cast<uint64_t>(pairs), k * 2,
                              64, static_cast<uint32_t>(kMoeXBox), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    CUtensorMap tm_codes;  // the stacked experts' codes [E * n, k]
    if (!encode_tensor_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.codes, k,
                              static_cast<uint64_t>(g.num_experts) * static_cast<uint64_t>(a.n), k, kKB, kTileW,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int64_t wtiles = (a.n + kTileW - 1) / kTileW;
    // at most ceil(pairs / tile) full tiles plus one partial tile per expert;
    // the CTAs past the routing's actual tile count leave at once
    // one routing tile is one CTA's x rows
    static_assert(Geo<kMoeGemmTileNarrow>::kTileX == kMoeGemmTileNarrow, "narrow tiles");
    static_assert(Geo<kMoeGemmTileWide>::kTileX == kMoeGemmTileWide, "wide tiles");
    const bool narrow = r.gemm_tile == kMoeGemmTileNarrow;
    if (!narrow && r.gemm_tile != kMoeGemmTileWide) return cudaErrorInvalidValue;
    const int64_t tbound = moe_gemm_tile_bound(pairs, g.num_experts, r.gemm_tile);
    if (tbound > 65535) return cudaErrorNotSupported;
    const dim3 grid(static_cast<unsigned>(wtiles), static_cast<unsigned>(tbound));
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const MoeTiles tiles{r.tile_off, r.tile_info, r.perm, static_cast<int>(g.topk), static_cast<int>(g.num_experts)};
    auto y = static_cast<__nv_bfloat16 *>(a.y);
    const int pi = static_cast<int>(pairs), ni = static_cast<int>(a.n), ki = static_cast<int>(a.k);
    if (narrow)
        prefill_kernel<kScaleBlock, true, kMoeGemmTileNarrow>
            <<<grid, kThreads, Geo<kMoeGemmTileNarrow>::kSmemBytes, stream>>>(
                tm_x, tm_codes, a.scales, nullptr, 0, y, pi, ni, ki, kblocks, 0, 0, 0, 0, 1, 0, tiles);
    else
        prefill_kernel<kScaleBlock, true, kMoeGemmTileWide>
            <<<grid, kThreads, Geo<kMoeGemmTileWide>::kSmemBytes, stream>>>(
                tm_x, tm_codes, a.scales, nullptr, 0, y, pi, ni, ki, kblocks, 0, 0, 0, 0, 1, 0, tiles);
    return cudaGetLastError();
}

uint32_t take_prefill_error() {
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill_err, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_prefill_err, &zero, sizeof zero);
    return v;
}

}  // namespace fp8bs
