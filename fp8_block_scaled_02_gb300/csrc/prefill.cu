// prefill.cu -- block-FP8 W8A16 GEMM for prefill-shaped batches on the
// 5th-generation tensor cores (tcgen05), y[M, N] = x[M, K] . dequant(W)^T.
//
// Design (sm_103a, one CTA per 128 weight rows x 128 rows of x, 18 warps):
//  * Weights are the MMA's A operand and live in tensor memory: eight
//    "decoder" warps stream their rows' e4m3 codes from global memory (each
//    thread owns one weight row = one TMEM lane and one 64-wide K half,
//    loading two K blocks ahead), convert them exactly to bf16 pairs in
//    registers and tcgen05.st them into a double-buffered 64-column A slot
//    (128 K of bf16 per K block).  The decoded weight never touches shared
//    memory or HBM.
//  * x is the B operand: one producer thread brings each K block's
//    [128 rows x 128 K] bf16 tile in with 2-D TMA (128-byte swizzle, two
//    64-column panels) into a 4-stage shared-memory ring.
//  * One thread issues tcgen05.mma.kind::f16 (bf16 x bf16 -> fp32, M=128,
//    N=128, K=16; 8 per K block).  Each K block accumulates from zero into
//    one of two 128-column TMEM accumulators.
//  * Eight epilogue warps (two per TMEM lane quarter, one per 64-column
//    half) read each finished K-block accumulator with tcgen05.ld, multiply
//    it by that block's fp32 scale and add it into 64 fp32 registers per
//    thread ("promotion"), so the scale is applied once per 128-wide K
//    block to an fp32 partial and never folded into a rounded bf16 weight.
//    At the end each thread stores its weight row's outputs as bf16.
//  * With one scale per weight row (or per tensor) there is nothing to
//    promote per K block: all K blocks accumulate into one TMEM
//    accumulator, and the epilogue reads it once after the last MMA,
//    multiplies each row by its scale and stores bf16.
//  * mbarriers: x_full (TMA ring), a_full (TMEM A slots), d_empty (TMEM
//    accumulators), and a ring of "MMA done" barriers, one tcgen05.commit
//    per K block, that frees x stages, A slots and accumulators alike.  Every wait is bounded; a kernel that gives up sets an error
//    word, drains what it issued and still frees its TMEM.
#include "common.cuh"
#include "internal.h"

#include <mutex>

namespace fp8bs {

namespace {

__device__ uint32_t g_prefill_err;

constexpr int kTileW = 128;       // weight rows per CTA (= one scale row block, = MMA M)
constexpr int kTileX = 128;       // x rows per CTA (= MMA N)
constexpr int kKB = 128;          // K per block
constexpr int kXStages = 4;
constexpr int kRing = 4;          // MMA-completion barriers (>= x stages, > A slots, > accumulators)
static_assert(kXStages <= kRing, "the x producer waits on a block kXStages back");
constexpr int kXPanel = kTileX * 128;     // 64 bf16 per row, 16 KB
constexpr int kXStage = 2 * kXPanel;      // 32 KB
constexpr int kTmemCols = 512;
constexpr int kColA = 0;                  // A slots: [0, 64) and [64, 128)
constexpr int kColD = 128;                // accumulators: [128, 256) and [256, 384)

// warp roles
constexpr int kWarpMma = 0;       // also allocates / frees TMEM
constexpr int kWarpTma = 1;
constexpr int kWarpDec0 = 2;      // 2..9 decoders: lane quarter warp % 4, K half (warp - 2) / 4
constexpr int kNumDec = 8;
constexpr int kWarpEpi0 = kWarpDec0 + kNumDec;  // 10..17 epilogue: lane quarter warp % 4, column half (warp - 10) / 4
constexpr int kNumEpi = 8;
constexpr int kThreads = (kWarpEpi0 + kNumEpi) * 32;
constexpr int kSmemBytes = 1024 + kXStages * kXStage + 256;

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kTileX >> 3) << 17) |
                            (static_cast<uint32_t>(kTileW >> 4) << 24);

// Shared-memory matrix descriptor for a K-major operand stored in the
// canonical 128-byte-swizzle layout (rows of 128 bytes, 8-row atoms of 1024
// bytes stacked along M/N): start address >> 4 (bits 0-13), leading byte
// offset (unused for this layout; 16 bytes) at bits 16-29, stride byte
// offset 1024 >> 4 at bits 32-45, descriptor version 1 (bits 46-47), layout
// type 2 = 128-byte swizzle (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    return static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(accumulate), "r"(kIdesc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
          "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
          "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_codes16(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void fail(uint32_t bit) { atomicOr(&g_prefill_err, bit); }

// ROW: scales[row * row_stride] per weight row (stride 0: one per tensor)
// instead of 128x128 block scales.
template <bool ROW>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                              const uint8_t *__restrict__ codes,
                                                              const float *__restrict__ scales,
                                                              __nv_bfloat16 *__restrict__ y, int m, int n,
                                                              int k, int kblocks, int row_stride) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kXStages * kXStage);
    // done[kb % kRing] completes when the MMAs of K block kb have finished
    // (one tcgen05.commit per block); the x producer, the decoders and the
    // epilogue all wait on it, each before its ring slot could be reused
    uint64_t *x_full = bars;                 // [kXStages]
    uint64_t *done = bars + kXStages;        // [kRing]
    uint64_t *a_full = done + kRing;         // [2]
    uint64_t *d_empty = a_full + 2;          // [2]
    uint64_t *d_full = d_empty + 2;          // ROW: all MMAs of the tile done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(d_full + 1);
    int *s_fail = reinterpret_cast<int *>(d_full + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileW;
    const int m0 = blockIdx.y * kTileX;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kXStages; ++i) mbar_init(&x_full[i], 1);
        for (int i = 0; i < kRing; ++i) mbar_init(&done[i], 1);  // tcgen05.commit
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_full[i], kNumDec);   // one arrival per decoder warp
            mbar_init(&d_empty[i], kNumEpi);  // one arrival per epilogue warp
        }
        mbar_init(d_full, 1);  // tcgen05.commit
        *s_fail = 0;
        fence_mbarrier_init();
    }
    if (warp == kWarpTma && lane == 0) prefetch_tensormap(&tm_x);
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        int issued = 0;  // K blocks whose MMAs were committed
        if (lane == 0) {
            for (int kb = 0; kb < kblocks; ++kb) {
                const int xs = kb % kXStages, as = kb & 1, db = ROW ? 0 : (kb & 1);
                bool ok = mbar_wait_bounded(&x_full[xs], (kb / kXStages) & 1) &&
                          mbar_wait_bounded(&a_full[as], (kb >> 1) & 1) &&
                          (ROW || kb < 2 || mbar_wait_bounded(&d_empty[db], ((kb >> 1) - 1) & 1));
                if (!ok) {
                    fail(ERRBIT_MMA_WAIT);
                    *reinterpret_cast<volatile int *>(s_fail) = 1;
                    break;
                }
                tc_fence_after();
                // descriptor of the stage's first 16-column slice; the others
                // are 32 bytes (2 in address/16 units) apart within a 64-column
                // panel, and panels are kXPanel bytes apart
                const uint64_t desc0 = sw128_desc(smem_u32(smem + xs * kXStage));
                const uint32_t d_tmem = tmem + kColD + db * 128;
                const uint32_t a_tmem = tmem + kColA + as * 64;
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk)
                    tc_mma(d_tmem, a_tmem + kk * 8, desc0 + (kk >> 2) * (kXPanel >> 4) + (kk & 3) * 2,
                           (kk > 0 || (ROW && kb > 0)) ? 1u : 0u);
                tc_commit(&done[kb % kRing]);
                issued = kb + 1;
            }
            // ROW: the epilogue's single wait (also after a failure, so that
            // it does not sit out its whole time limit)
            if (ROW) tc_commit(d_full);
            // drain: wait for the last committed block before TMEM can be freed
            if (issued > 0 && !mbar_wait_bounded(&done[(issued - 1) % kRing], ((issued - 1) / kRing) & 1))
                fail(ERRBIT_MMA_WAIT);
        }
        __syncwarp();
    } else if (warp == kWarpTma) {
        // ------------------------------------------------------ x producer
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < kblocks; ++kb) {
                const int xs = kb % kXStages;
                if (kb >= kXStages && !mbar_wait_bounded(&done[(kb - kXStages) % kRing], ((kb - kXStages) / kRing) & 1)) {
                    fail(ERRBIT_EMPTY_WAIT);
                    break;
                }
                if (*reinterpret_cast<volatile int *>(s_fail)) break;
                uint8_t *st = smem + xs * kXStage;
                mbar_arrive_expect_tx(&x_full[xs], kXStage);
                tma_load_2d(st, &tm_x, &x_full[xs], kb * kKB, m0);
                tma_load_2d(st + kXPanel, &tm_x, &x_full[xs], kb * kKB + 64, m0);
                issued = kb + 1;
            }
            // never leave with copies in flight: wait for the last stages issued
            for (int kb = issued - kXStages < 0 ? 0 : issued - kXStages; kb < issued; ++kb)
                if (!mbar_wait_bounded(&x_full[kb % kXStages], (kb / kXStages) & 1)) fail(ERRBIT_FULL_WAIT);
        }
        __syncwarp();
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------ decoders
        // thread = one weight row (its TMEM lane); this warp converts the K
        // half kh (64 codes) of its rows for every K block, two blocks ahead
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int kh = (warp - kWarpDec0) >> 2;
        const int row = n0 + q * 32 + lane;
        const bool row_ok = row < n;
        const uint8_t *rp = codes + static_cast<int64_t>(row_ok ? row : 0) * k + kh * 64;
        auto load4 = [&](int kb, uint4 (&v)[4]) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = kb * kKB + kh * 64 + j * 16;
                v[j] = (kb < kblocks && row_ok && col < k) ? ld_codes16(rp + kb * kKB + j * 16) : make_uint4(0, 0, 0, 0);
            }
        };
        uint4 c0[4], c1[4], c2[4];
        load4(0, c0);
        load4(1, c1);
        for (int kb = 0; kb < kblocks; ++kb) {
            const int as = kb & 1;
            load4(kb + 2, c2);  // in flight while this block is converted
            bool ok = kb < 2 || mbar_wait_bounded(&done[(kb - 2) % kRing], ((kb - 2) / kRing) & 1);
            if (!__all_sync(0xffffffffu, ok) || *reinterpret_cast<volatile int *>(s_fail)) {
                if (lane == 0) fail(ERRBIT_EMPTY_WAIT);
                break;
            }
            tc_fence_after();
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 c = c0[j];
                v[8 * j + 0] = e4m3x2_to_bf16x2(c.x, 0x9180u);
                v[8 * j + 1] = e4m3x2_to_bf16x2(c.x, 0xB3A2u);
                v[8 * j + 2] = e4m3x2_to_bf16x2(c.y, 0x9180u);
                v[8 * j + 3] = e4m3x2_to_bf16x2(c.y, 0xB3A2u);
                v[8 * j + 4] = e4m3x2_to_bf16x2(c.z, 0x9180u);
                v[8 * j + 5] = e4m3x2_to_bf16x2(c.z, 0xB3A2u);
                v[8 * j + 6] = e4m3x2_to_bf16x2(c.w, 0x9180u);
                v[8 * j + 7] = e4m3x2_to_bf16x2(c.w, 0xB3A2u);
            }
            tc_st32(tmem + (static_cast<uint32_t>(q * 32) << 16) + kColA + as * 64 + kh * 32, v);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[as]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                c0[j] = c1[j];
                c1[j] = c2[j];
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        // thread = one weight row (TMEM lane); this warp promotes the 64
        // accumulator columns (rows of x) of half ch
        const int q = warp & 3;
        const int ch = (warp - kWarpEpi0) >> 2;
        float acc[kTileX / 2];
#pragma unroll
        for (int i = 0; i < kTileX / 2; ++i) acc[i] = 0.0f;
        const float *srow = scales + (ROW ? 0 : static_cast<int64_t>(blockIdx.x) * kblocks);
        bool ok = true;
        if (ROW) {
            ok = mbar_wait_bounded(d_full, 0);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(ERRBIT_FULL_WAIT);
                ok = false;
            } else {
                ok = *reinterpret_cast<volatile int *>(s_fail) == 0;
                tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + kColD + ch * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[16];
                    tc_ld16(taddr + 16 * c, v);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[16 * c + i] = __uint_as_float(v[i]);
                }
                const int row = n0 + q * 32 + lane;
                const float rs = row < n ? __ldg(scales + static_cast<int64_t>(row) * row_stride) : 0.0f;
#pragma unroll
                for (int i = 0; i < kTileX / 2; ++i) acc[i] *= rs;
            }
        }
        for (int kb = 0; ROW ? false : kb < kblocks; ++kb) {
            const int db = kb & 1;
            const float s = __ldg(srow + kb);
            ok = mbar_wait_bounded(&done[kb % kRing], (kb / kRing) & 1);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(ERRBIT_FULL_WAIT);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + kColD + db * 128 + ch * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[16];
                tc_ld16(taddr + 16 * c, v);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[16 * c + i] = fmaf(s, __uint_as_float(v[i]), acc[16 * c + i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[db]);
        }
        // thread = weight row, acc[i] = y[m0 + 64 ch + i][row]
        const int row = n0 + q * 32 + lane;
        if (ok && row < n) {
#pragma unroll
            for (int i = 0; i < kTileX / 2; ++i) {
                const int mi = m0 + ch * 64 + i;
                if (mi < m) y[static_cast<int64_t>(mi) * n + row] = __float2bfloat16_rn(acc[i]);
            }
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

std::mutex g_setup_mu;
bool g_setup_done[64] = {};
cudaError_t g_setup_err[64] = {};

}  // namespace

cudaError_t launch_prefill(const DecodeArgs &a, cudaStream_t stream) {
    if (a.kind != kScaleBlock && a.kind != kScaleRow) return cudaErrorNotSupported;
    const bool row = a.kind == kScaleRow;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_setup_done[dev]) {
            cudaError_t e =
                cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
            g_setup_err[dev] = e;
            g_setup_done[dev] = true;
        }
        if (g_setup_err[dev] != cudaSuccess) return g_setup_err[dev];
    }
    CUtensorMap tm_x;
    const uint64_t k = static_cast<uint64_t>(a.k), m = static_cast<uint64_t>(a.m);
    if (!encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, k, m, k * 2, 64, kTileX,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int kblocks = static_cast<int>((a.k + kKB - 1) / kKB);
    const dim3 grid(static_cast<unsigned>((a.n + kTileW - 1) / kTileW), static_cast<unsigned>((a.m + kTileX - 1) / kTileX));
    auto kern = row ? prefill_kernel<true> : prefill_kernel<false>;
    kern<<<grid, kThreads, kSmemBytes, stream>>>(tm_x, a.codes, a.scales, static_cast<__nv_bfloat16 *>(a.y),
                                                 static_cast<int>(a.m), static_cast<int>(a.n), static_cast<int>(a.k),
                                                 kblocks, row ? a.row_stride : 0);
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
