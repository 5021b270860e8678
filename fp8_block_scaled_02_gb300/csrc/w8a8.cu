// w8a8.cu -- W8A8 linear: e4m3 activations (dynamic per-tensor scale s_x)
// times an e4m3 weight with one per-tensor scale s_w,
//   y[m, n] = bf16_rn( s_x * s_w * sum_k dec(qx[m, k]) * dec(qw[n, k]) ),
// the route of FreeToken PR #389 (What this adds: a dynamic per-tensor
// activation scale, then the FP8 GEMM).  Products of two e4m3 values are
// exact in fp32; the sum accumulates in fp32 and both scales multiply it
// once before the bf16 rounding.
//
//  * w8a8_decode_kernel (m <= 32 per launch): the e4m3 tensor-core MMA
//    (mma.sync m16n8k32 e4m3 x e4m3 -> fp32) takes both operands straight
//    from the staged codes -- no conversion at all.  One CTA owns 128 weight
//    rows; a TMA warp streams 128x128 code tiles plus the matching x code
//    tile (128-byte swizzle) into a 4-stage ring; eight consumer warps each
//    own a 16-row tile over the whole K block.  With few row tiles the K
//    blocks are split over a thread-block cluster and reduced through DSMEM
//    in rank order, as in the W8A16 decode kernel.
//  * w8a8_prefill_kernel: tcgen05.mma.kind::f8f6f4 (M=128, N=256, K=32),
//    both operands loaded by TMA into a 4-stage ring; persistent CTAs (one
//    per SM) loop over 128 x 256 output tiles, each tile accumulating over
//    the whole K range in one of two 256-column TMEM accumulators, so one
//    tile's epilogue overlaps the next tile's MMAs.
//  * w8a8_generic_kernel: plain loads, any shape or alignment.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

#include <mutex>

namespace fp8bs {

namespace {

__device__ uint32_t g_w8a8_err;

constexpr int kKB = 128;  // K (bytes = elements) per stage

__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ================================================================= decode
constexpr int kDBN = 128;          // weight rows per CTA
constexpr int kDStages = 4;
constexpr int kDConsumers = 8;     // one 16-row tile each
constexpr int kDWarpTma = kDConsumers;
constexpr int kMaxSplit = 8;       // portable cluster size limit

// named barrier of the eight consumer warps (the TMA warp is not waited for)
__device__ __forceinline__ void w8a8_consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kDConsumers * 32) : "memory");
}

template <int MT>
struct DCfg {
    static constexpr int kXRows = 8 * MT;                 // x rows staged (zero-padded by TMA)
    static constexpr int kCodeBytes = kDBN * kKB;         // 16 KB
    static constexpr int kXBytes = kXRows * kKB;          // 1-4 KB, a multiple of 1024
    static constexpr int kStageBytes = kCodeBytes + kXBytes;
    static constexpr int kRedStride = kXRows + 1;
    // split-K receive buffer: [source rank][row of this CTA's slice][m];
    // splits * ceil(128 / splits) <= 135 rows
    static constexpr int kRecvFloats = (kDBN + kMaxSplit) * kRedStride;
    static constexpr int kThreads = (kDConsumers + 1) * 32;
    static constexpr int kSmemBytes = 1024 + kDStages * kStageBytes + kRecvFloats * 4 + 2 * kDStages * 8;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert((kRecvFloats * 4) % 8 == 0, "barriers must stay 8-byte aligned");
    static_assert(kDBN * kRedStride * 4 <= kStageBytes, "split-K partials fit in ring stage 0");
    static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
};

// One CTA processes row tiles blockIdx.x, blockIdx.x + gridDim.x, ... for
// its K range; splits > 1: one row tile per CTA, cluster reduction over K.
//
// Fragments (m16n8k32, 8-bit operands): thread (g = lane / 4, t = lane % 4)
// holds A rows g and g + 8 at k = 4t..4t+3 (a0, a1) and 16+4t..16+4t+3
// (a2, a3), B column g at the same k.  The logical k order inside each
// 32-wide slice is a fixed permutation of the physical bytes, applied to A
// and B alike: thread t's 8 logical bytes are physical bytes 8t..8t+7, so
// every fragment is one 8-byte shared-memory load.
template <int MT>
__global__ void __launch_bounds__(DCfg<MT>::kThreads, 2) w8a8_decode_kernel(
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, const float *__restrict__ sx_p,
    const float *__restrict__ sw_p, __nv_bfloat16 *__restrict__ y, int m, int n, int kblocks, int splits,
    int ntiles) {
    using C = DCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    float *recv = reinterpret_cast<float *>(smem + kDStages * C::kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(recv + C::kRecvFloats);
    uint64_t *empty = full + kDStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.y;
    const int kb0 = static_cast<int>((static_cast<int64_t>(split) * kblocks) / splits);
    const int kb1 = static_cast<int>((static_cast<int64_t>(split + 1) * kblocks) / splits);
    const int nkb = kb1 - kb0;
    const int tile0 = blockIdx.x, tstep = gridDim.x;
    const int my_tiles = tile0 < ntiles ? (ntiles - tile0 + tstep - 1) / tstep : 0;
    const int total = my_tiles * nkb;
    const int mm = min(m, C::kXRows);
    // split-K: CTA r of the cluster finishes rows [r * rows_per, (r + 1) * rows_per)
    const int rank = splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int rows_per = (kDBN + splits - 1) / splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDConsumers);
        }
        fence_mbarrier_init();
    }
    if (warp == kDWarpTma && lane == 0) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(&tm_x);
        // the first ring-depth of weight tiles on their way into L2 while the
        // previous kernel drains (an L2 prefetch never observes stale data)
        const int npf = min(total, kDStages);
        for (int it = 0; it < npf; ++it) {
            const int ti = it / nkb;
            tma_prefetch_l2_2d(&tm_w, (kb0 + (it - ti * nkb)) * kKB, (tile0 + ti * tstep) * kDBN);
        }
    }
    __syncthreads();
    // nothing above reads what an earlier kernel writes: let the next kernel
    // in the stream be scheduled (it waits for this one before its reads)
    pdl_launch_dependents();
    pdl_wait();  // x codes and s_x may come from the previous kernel in the stream

    if (warp == kDWarpTma) {
        // ------------------------------------------------------ TMA producer
        const uint64_t stream_policy = policy_evict_first();
        for (int it = 0; it < total; ++it) {
            const int s = it % kDStages;
            int good = 1;
            if (it >= kDStages && lane == 0) good = mbar_wait_bounded(&empty[s], ((it / kDStages) - 1) & 1);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                if (lane == 0) atomicOr(&g_w8a8_err, ERRBIT_EMPTY_WAIT);
                break;
            }
            if (lane == 0) {
                const int ti = it / nkb;
                const int n0 = (tile0 + ti * tstep) * kDBN;
                const int kx = (kb0 + (it - ti * nkb)) * kKB;
                uint8_t *st = smem + s * C::kStageBytes;
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                tma_load_2d_hint(st, &tm_w, &full[s], kx, n0, stream_policy);
                tma_load_2d(st + C::kCodeBytes, &tm_x, &full[s], kx, 0);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------ consumers
        const int g = lane >> 2, t = lane & 3;
        const int ra = warp * 16 + g, rb = ra + 8;  // this thread's weight rows
        const int coff = (t & 1) * 8;
        const float scale = __ldg(sx_p) * __ldg(sw_p);
        bool failed = false;
        float acc[MT][4];  // split-K: read again after the tile loop
        for (int ti = 0; ti < my_tiles && !failed; ++ti) {
            const int n0 = (tile0 + ti * tstep) * kDBN;
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[j][q] = 0.0f;
            for (int kbi = 0; kbi < nkb; ++kbi) {
                const int it = ti * nkb + kbi;
                const int s = it % kDStages;
                const bool ready = mbar_wait_bounded(&full[s], (it / kDStages) & 1);
                if (!__all_sync(0xffffffffu, ready)) {
                    if (lane == 0) atomicOr(&g_w8a8_err, ERRBIT_FULL_WAIT);
                    failed = true;
                    break;
                }
                const uint8_t *cs = smem + s * C::kStageBytes;
                const uint8_t *xs = cs + C::kCodeBytes;
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    const int chunk = 2 * sl + (t >> 1);
                    const uint2 qa = *reinterpret_cast<const uint2 *>(cs + ra * 128 + ((chunk ^ (ra & 7)) << 4) + coff);
                    const uint2 qb = *reinterpret_cast<const uint2 *>(cs + rb * 128 + ((chunk ^ (rb & 7)) << 4) + coff);
#pragma unroll
                    for (int j = 0; j < MT; ++j) {
                        const int xr = 8 * j + g;
                        const uint2 bx =
                            *reinterpret_cast<const uint2 *>(xs + xr * 128 + ((chunk ^ (xr & 7)) << 4) + coff);
                        mma_e4m3_16832(acc[j], qa.x, qb.x, qa.y, qb.y, bx.x, bx.y);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (failed) break;
            // acc[j][q] is y[m = 8j + 2t + (q & 1)][n_local = (q < 2 ? ra : rb)]
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int mi = 8 * j + 2 * t + (q & 1);
                    const int nl = q < 2 ? ra : rb;
                    if (splits == 1 && mi < m && n0 + nl < n)
                        y[static_cast<int64_t>(mi) * n + n0 + nl] = __float2bfloat16_rn(acc[j][q] * scale);
                }
        }
        if (splits > 1) {
            // Split-K (one row tile): stage the partials in ring stage 0, free
            // once every consumer has left the ring, then push each row's
            // partial into its finisher's receive slot with coalesced DSMEM
            // stores (faster than scattering them from the MMA fragments).
            float *red = reinterpret_cast<float *>(smem);
            w8a8_consumer_bar();
#pragma unroll
            for (int j = 0; j < MT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int mi = 8 * j + 2 * t + (q & 1);
                    red[(q < 2 ? ra : rb) * C::kRedStride + mi] = acc[j][q];
                }
            w8a8_consumer_bar();
            const uint32_t recv_base =
                smem_u32(recv) + static_cast<uint32_t>(rank * rows_per * C::kRedStride * 4);
            for (int e = threadIdx.x; e < mm * kDBN; e += kDConsumers * 32) {
                const int nl = e / mm;
                const int mi = e - nl * mm;
                const int owner = nl / rows_per;
                const uint32_t off = static_cast<uint32_t>(((nl - owner * rows_per) * C::kRedStride + mi) * 4);
                dsmem_st_f32(dsmem_map(recv_base + off, static_cast<uint32_t>(owner)), red[nl * C::kRedStride + mi]);
            }
        }
    }
    if (splits == 1) return;

    // Split-K: one row tile per CTA; reduce across the cluster in rank order.
    // The consumers pushed each row's partial into its finisher's receive
    // buffer (slot = source rank); one release / acquire cluster barrier
    // makes them visible, and each CTA sums its rows locally in rank order
    // (no remote reads, so no second barrier before exit).
    const int n0 = tile0 * kDBN;
    cluster_sync_all();
    const float scale = __ldg(sx_p) * __ldg(sw_p);
    const int r_begin = rank * rows_per;
    const int r_end = min(kDBN, r_begin + rows_per);
    const int my_rows = max(0, r_end - r_begin);
    for (int e = threadIdx.x; e < mm * my_rows; e += C::kThreads) {
        const int mi = e / my_rows;
        const int rl = e - mi * my_rows;
        const int nn = n0 + r_begin + rl;
        if (nn >= n) continue;
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxSplit; ++q)
            if (q < splits) sum += recv[(q * rows_per + rl) * C::kRedStride + mi];
        y[static_cast<int64_t>(mi) * n + nn] = __float2bfloat16_rn(sum * scale);
    }
}

struct Setup {
    std::mutex mu;
    bool done[64] = {};
    cudaError_t err[64] = {};
    int resident[64] = {};
    ClusterFit fit;
};

template <int MT>
cudaError_t launch_decode_t(const W8A8Args &a, cudaStream_t stream) {
    using C = DCfg<MT>;
    auto kern = w8a8_decode_kernel<MT>;
    static Setup setup;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int resident = 1;
    {
        std::lock_guard<std::mutex> lock(setup.mu);
        if (!setup.done[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
            int blocks = 0;
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, C::kThreads, C::kSmemBytes);
            setup.err[dev] = e;
            setup.resident[dev] = blocks > 0 ? blocks : 1;
            setup.done[dev] = true;
        }
        if (setup.err[dev] != cudaSuccess) return setup.err[dev];
        resident = setup.resident[dev];
    }
    CUtensorMap tm_w, tm_x;
    const uint64_t n = static_cast<uint64_t>(a.n), k = static_cast<uint64_t>(a.k), m = static_cast<uint64_t>(a.m);
    if (!encode_tensor_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq, k, n, k, kKB, kDBN,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.xq, k, m, k, kKB, C::kXRows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const int ntiles = static_cast<int>((a.n + kDBN - 1) / kDBN);
    const int capacity = device_sm_count() * resident;
    int splits = 1;
    if (ntiles < capacity) {
        // as many K splits as fill the SMs, in clusters that all fit at once
        int cap = capacity / ntiles;
        if (cap > kMaxSplit) cap = kMaxSplit;
        if (cap > kblocks) cap = kblocks;
        splits = pick_split(setup.fit, reinterpret_cast<const void *>(kern), C::kThreads, C::kSmemBytes, ntiles, cap);
    }
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
    return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, a.sx, a.sw, static_cast<__nv_bfloat16 *>(a.y),
                              static_cast<int>(a.m), static_cast<int>(a.n), kblocks, splits, ntiles);
}

// ================================================================ prefill
constexpr int kPTileW = 128;              // weight rows per CTA (MMA M)
constexpr int kPTileX = 256;              // x rows per CTA (MMA N)
constexpr int kPStages = 4;
constexpr int kPABytes = kPTileW * kKB;   // 16 KB
constexpr int kPBBytes = kPTileX * kKB;   // 32 KB
constexpr int kPStage = kPABytes + kPBBytes;
constexpr int kPTmemCols = 512;           // accumulators D_0, D_1: columns [0, 256), [256, 512)
constexpr int kPWarpMma = 0, kPWarpTma = 1, kPWarpEpi0 = 2, kPNumEpi = 8;
constexpr int kPThreads = (kPWarpEpi0 + kPNumEpi) * 32;
constexpr int kPSmemBytes = 1024 + kPStages * kPStage + 256;
static_assert(kPSmemBytes <= 227 * 1024, "shared memory per CTA");

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3
// (format 0 at bits 7-9 and 10-12), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdescF8 = (1u << 4) | (static_cast<uint32_t>(kPTileX >> 3) << 17) |
                              (static_cast<uint32_t>(kPTileW >> 4) << 24);

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %4, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(kIdescF8)
        : "memory");
}

// Persistent: CTA b takes output tiles b, b + gridDim.x, ... (tile t = weight
// tile t % tiles_w, x tile t / tiles_w).  The TMA ring streams straight across
// tile boundaries and consecutive tiles accumulate into alternate TMEM
// accumulators, so the epilogue of one tile overlaps the MMAs of the next.
__global__ void __launch_bounds__(kPThreads, 1) w8a8_prefill_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                                   const __grid_constant__ CUtensorMap tm_x,
                                                                   const float *__restrict__ sx_p,
                                                                   const float *__restrict__ sw_p,
                                                                   __nv_bfloat16 *__restrict__ y, int m, int n,
                                                                   int kblocks, int tiles_w, int tiles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kPStages * kPStage);  // [kPStages]
    uint64_t *empty = full + kPStages;                                         // [kPStages]
    uint64_t *d_full = empty + kPStages;                                       // [2] a tile's MMAs done
    uint64_t *d_empty = d_full + 2;                                            // [2] a tile's epilogue done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(d_empty + 2);
    int *s_fail = reinterpret_cast<int *>(d_empty + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile0 = blockIdx.x, tstep = gridDim.x;
    const int my_tiles = tile0 < tiles ? (tiles - tile0 + tstep - 1) / tstep : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);  // tcgen05.commit
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);          // tcgen05.commit
            mbar_init(&d_empty[i], kPNumEpi);  // every epilogue warp
        }
        *s_fail = 0;
        fence_mbarrier_init();
    }
    if (warp == kPWarpTma && lane == 0) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(&tm_x);
    }
    if (warp == kPWarpMma) tc_alloc(tmem_slot, kPTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    if (warp == kPWarpMma) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int u = 0;  // stages consumed (all tiles)
            bool failed = false;
            for (int i = 0; i < my_tiles && !failed; ++i) {
                const int b = i & 1;
                // accumulator b was last read by the epilogue of tile i - 2
                if (i >= 2 && !mbar_wait_bounded(&d_empty[b], ((i - 2) >> 1) & 1)) {
                    atomicOr(&g_w8a8_err, ERRBIT_MMA_WAIT);
                    failed = true;
                } else {
                    tc_fence_after();
                    const uint32_t d = tmem + 256 * b;
                    for (int kb = 0; kb < kblocks; ++kb, ++u) {
                        const int s = u % kPStages;
                        if (!mbar_wait_bounded(&full[s], (u / kPStages) & 1)) {
                            atomicOr(&g_w8a8_err, ERRBIT_MMA_WAIT);
                            failed = true;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t adesc = sw128_desc(smem_u32(smem + s * kPStage));
                        const uint64_t bdesc = sw128_desc(smem_u32(smem + s * kPStage + kPABytes));
#pragma unroll
                        for (int kk = 0; kk < kKB / 32; ++kk)
                            tc_mma_f8(d, adesc + 2 * kk, bdesc + 2 * kk, (kb > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(&empty[s]);
                    }
                }
                if (failed) *reinterpret_cast<volatile int *>(s_fail) = 1;
                // the epilogue's wait for this tile (also after a failure, so
                // that it does not sit out its whole time limit)
                tc_commit(&d_full[b]);
            }
            // drain: wait for the last committed stage before TMEM can be freed
            if (u > 0 && !mbar_wait_bounded(&empty[(u - 1) % kPStages], ((u - 1) / kPStages) & 1))
                atomicOr(&g_w8a8_err, ERRBIT_MMA_WAIT);
        }
        __syncwarp();
    } else if (warp == kPWarpTma) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int u = 0;  // stages issued (all tiles)
            bool stop = false;
            for (int i = 0; i < my_tiles && !stop; ++i) {
                const int t = tile0 + i * tstep;
                const int n0 = (t % tiles_w) * kPTileW, m0 = (t / tiles_w) * kPTileX;
                for (int kb = 0; kb < kblocks; ++kb, ++u) {
                    const int s = u % kPStages;
                    if (u >= kPStages && !mbar_wait_bounded(&empty[s], ((u - kPStages) / kPStages) & 1)) {
                        atomicOr(&g_w8a8_err, ERRBIT_EMPTY_WAIT);
                        stop = true;
                        break;
                    }
                    if (*reinterpret_cast<volatile int *>(s_fail)) {
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + s * kPStage;
                    mbar_arrive_expect_tx(&full[s], kPStage);
                    tma_load_2d(st, &tm_w, &full[s], kb * kKB, n0);
                    tma_load_2d(st + kPABytes, &tm_x, &full[s], kb * kKB, m0);
                }
            }
            // never leave with copies in flight: wait for the last stages issued
            for (int v = u - kPStages < 0 ? 0 : u - kPStages; v < u; ++v)
                if (!mbar_wait_bounded(&full[v % kPStages], (v / kPStages) & 1))
                    atomicOr(&g_w8a8_err, ERRBIT_FULL_WAIT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        // thread = one weight row (TMEM lane of quarter q); columns
        // [128 ch, 128 ch + 128) of a tile's accumulator are rows
        // m0 + 128 ch + j of x
        const int q = warp & 3;
        const int ch = (warp - kPWarpEpi0) >> 2;
        const float scale = __ldg(sx_p) * __ldg(sw_p);
        for (int i = 0; i < my_tiles; ++i) {
            const int b = i & 1;
            const int t = tile0 + i * tstep;
            const int n0 = (t % tiles_w) * kPTileW, m0 = (t / tiles_w) * kPTileX;
            const int row = n0 + q * 32 + lane;
            const bool ok = mbar_wait_bounded(&d_full[b], (i >> 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) atomicOr(&g_w8a8_err, ERRBIT_FULL_WAIT);
                break;
            }
            if (*reinterpret_cast<volatile int *>(s_fail)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + 256 * b + ch * 128;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[16];
                tc_ld16(taddr + 16 * c, v);
                tc_wait_ld();
                if (row < n) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int mi = m0 + ch * 128 + 16 * c + j;
                        if (mi < m)
                            y[static_cast<int64_t>(mi) * n + row] = __float2bfloat16_rn(__uint_as_float(v[j]) * scale);
                    }
                }
            }
            // accumulator b has been read: the MMAs of tile i + 2 may reuse it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[b]);
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPWarpMma) tc_dealloc(tmem, kPTmemCols);
}

std::mutex g_prefill_mu;
bool g_prefill_done[64] = {};
cudaError_t g_prefill_err_set[64] = {};

// ================================================================ generic
constexpr int kGRows = 8;  // warps per CTA, one weight row each

__device__ __forceinline__ float e4m3_value(uint8_t code) {
    return bf16lo_to_f32(e4m3x2_to_bf16x2(code, 0x9180u));
}

__global__ void __launch_bounds__(kGRows * 32) w8a8_generic_kernel(const uint8_t *__restrict__ xq, int64_t m,
                                                                   const float *__restrict__ sx_p,
                                                                   const uint8_t *__restrict__ wq,
                                                                   const float *__restrict__ sw_p,
                                                                   uint16_t *__restrict__ y, int64_t n, int64_t k) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kGRows + (threadIdx.x >> 5);
    if (row >= n) return;
    pdl_wait();
    const float scale = __ldg(sx_p) * __ldg(sw_p);
    const uint8_t *wrow = wq + row * k;
    for (int64_t m0 = 0; m0 < m; m0 += 8) {
        const int mc = static_cast<int>(min(static_cast<int64_t>(8), m - m0));
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int64_t c = lane; c < k; c += 32) {
            const float wv = e4m3_value(wrow[c]);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < mc) acc[i] = fmaf(e4m3_value(xq[(m0 + i) * k + c]), wv, acc[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0 && i < mc) {
                const __nv_bfloat16 b = __float2bfloat16_rn(v * scale);
                y[(m0 + i) * n + row] = *reinterpret_cast<const uint16_t *>(&b);
            }
        }
    }
}

}  // namespace

cudaError_t launch_w8a8_decode(const W8A8Args &a, cudaStream_t stream) {
    switch ((a.m + 7) / 8) {
        case 1: return launch_decode_t<1>(a, stream);
        case 2: return launch_decode_t<2>(a, stream);
        case 3: return launch_decode_t<3>(a, stream);
        case 4: return launch_decode_t<4>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_w8a8_prefill(const W8A8Args &a, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_prefill_mu);
        if (!g_prefill_done[dev]) {
            g_prefill_err_set[dev] =
                cudaFuncSetAttribute(w8a8_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
            g_prefill_done[dev] = true;
        }
        if (g_prefill_err_set[dev] != cudaSuccess) return g_prefill_err_set[dev];
    }
    CUtensorMap tm_w, tm_x;
    const uint64_t n = static_cast<uint64_t>(a.n), k = static_cast<uint64_t>(a.k), m = static_cast<uint64_t>(a.m);
    if (!encode_tensor_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.wq, k, n, k, kKB, kPTileW,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.xq, k, m, k, kKB, kPTileX,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const int64_t tiles_w = (a.n + kPTileW - 1) / kPTileW;
    const int64_t tiles = tiles_w * ((a.m + kPTileX - 1) / kPTileX);
    // one CTA per SM (the ring takes most of its shared memory), each looping
    // over its tiles; its stage counter runs over all of them (an int)
    const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 1;
    if (tiles >= (int64_t(1) << 31) || (tiles / sms + 1) * kblocks >= (int64_t(1) << 31))
        return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
    w8a8_prefill_kernel<<<grid, kPThreads, kPSmemBytes, stream>>>(tm_w, tm_x, a.sx, a.sw,
                                                                  static_cast<__nv_bfloat16 *>(a.y),
                                                                  static_cast<int>(a.m), static_cast<int>(a.n),
                                                                  kblocks, static_cast<int>(tiles_w),
                                                                  static_cast<int>(tiles));
    return cudaGetLastError();
}

cudaError_t launch_w8a8_generic(const W8A8Args &a, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((a.n + kGRows - 1) / kGRows);
    w8a8_generic_kernel<<<blocks, kGRows * 32, 0, stream>>>(a.xq, a.m, a.sx, a.wq, a.sw,
                                                            static_cast<uint16_t *>(a.y), a.n, a.k);
    return cudaGetLastError();
}

uint32_t take_w8a8_error() {
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_w8a8_err, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_w8a8_err, &zero, sizeof zero);
    return v;
}

}  // namespace fp8bs
