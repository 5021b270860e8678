// prefill.cu -- block-FP8 / per-row FP8 W8A16 GEMM for prefill-shaped
// batches on the 5th-generation tensor cores (tcgen05),
// y[M, N] = x[M, K] . dequant(W)^T.
//
// Design (sm_103a, one CTA per 128 weight rows x 256 rows of x, 18 warps):
//  * Weights are the MMA's A operand.  Eight "decoder" warps stream their
//    rows' e4m3 codes from global memory (each thread owns one weight row
//    and one 64-wide K half, loading two K blocks ahead), convert them
//    exactly to bf16 pairs in registers and store them into a
//    double-buffered shared-memory A slot in the 128-byte-swizzled K-major
//    layout the tensor core reads.  The decoded weight never reaches HBM.
//    Each decoded 128 x 128 block feeds both 128-row halves of x, so the
//    decode work per flop is half that of a 128 x 128 tile.
//  * x is the B operand: one producer thread brings each unit's x rows
//    (block scales: one (K block, half), 128 rows; one scale per row: one K
//    block, all 256 rows) with 2-D TMA (128-byte swizzle, two 64-column
//    panels) into a 128 KB shared-memory ring.
//  * One thread issues tcgen05.mma.kind::f16 (bf16 x bf16 -> fp32, M=128,
//    K=16, 8 per unit, both operands from shared memory; N = 128 per half
//    with block scales, N = 256 with one scale per row, which reads each
//    decoded A fragment once for both halves) and one tcgen05.commit per
//    unit into a ring of "MMA done" barriers that frees x stages, A slots and
//    accumulators alike.
//  * Block scales: each (K block, half) accumulates from zero into that
//    half's 128-column TMEM partial D_h; eight epilogue warps (one per TMEM
//    lane quarter and half) read it with tcgen05.ld, multiply it by the
//    block's fp32 scale and add it into the half's running total T_h, which
//    also lives in TMEM (tcgen05.st), with packed fp32x2 FMAs ("promotion":
//    the scale is applied once per 128-wide K block to an fp32 partial and
//    never folded into a rounded bf16 weight).  TMEM: T_0, T_1, D_0, D_1 =
//    512 columns.
//  * With one scale per weight row (or per tensor) nothing is promoted per
//    K block: the MMAs accumulate straight into T_h across all of K, and the
//    epilogue reads it once after a final commit, multiplies each row by its
//    scale and stores bf16.
//  * Every wait is bounded; a kernel that gives up sets an error word,
//    drains what it issued and still frees its TMEM.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

#include <mutex>

namespace fp8bs {

namespace {

__device__ uint32_t g_prefill_err;

constexpr int kTileW = 128;       // weight rows per CTA (= one scale row block, = MMA M)
constexpr int kHalfX = 128;       // x rows per MMA group (= MMA N)
constexpr int kTileX = 2 * kHalfX;  // x rows per CTA
constexpr int kKB = 128;          // K per block
constexpr int kPanel = 128 * 128;           // one 64-column bf16 panel of 128 rows, 16 KB
constexpr int kXBytes = 4 * 2 * kPanel;     // x ring: 128 KB

// The x ring and the MMA shape.  Block scales: one unit = (K block, half of
// x), N = 128, into that half's partial D_h, so one half's promotion overlaps
// the other half's MMAs.  One scale per row: nothing to promote, one unit =
// K block, N = 256 straight into T = [T_0 | T_1]: each decoded A fragment is
// read from shared memory once for both halves.
template <bool ROW>
struct PCfg {
    static constexpr int kN = ROW ? kTileX : kHalfX;      // MMA N = x rows per unit
    static constexpr int kUnitsPerKb = ROW ? 1 : 2;
    static constexpr int kXPanel = kN * 128;              // one 64-column panel of the unit's x rows
    static constexpr int kXStage = 2 * kXPanel;           // 32 KB / 64 KB
    static constexpr int kXStages = kXBytes / kXStage;    // 4 / 2
};
constexpr int kASlots = 2;                  // decoded weight blocks in flight
constexpr int kASlot = 2 * kPanel;          // 32 KB
constexpr int kRing = 8;  // MMA-completion barriers, one per unit; >= every look-back
static_assert(4 <= kRing && 2 * kASlots <= kRing, "a wait must never reach back a full ring");
constexpr int kTmemCols = 512;
constexpr int kColT = 0;                  // running totals T_0, T_1: [0, 128), [128, 256)
constexpr int kColD = 256;                // per-K-block partials D_0, D_1: [256, 384), [384, 512)

// warp roles
constexpr int kWarpMma = 0;       // also allocates / frees TMEM
constexpr int kWarpTma = 1;
constexpr int kWarpDec0 = 2;      // 2..9 decoders: weight rows 32 (warp % 4) .. +31, K half (warp - 2) / 4
constexpr int kNumDec = 8;
constexpr int kWarpEpi0 = kWarpDec0 + kNumDec;  // 10..17 epilogue: TMEM lane quarter warp % 4, half (warp - 10) / 4
constexpr int kNumEpi = 8;
constexpr int kThreads = (kWarpEpi0 + kNumEpi) * 32;
constexpr int kSmemBytes = 1024 + kXBytes + kASlots * kASlot + 256;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
template <int N>
__host__ __device__ constexpr uint32_t idesc_f16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(kTileW >> 4) << 24);
}

__device__ __forceinline__ uint4 ld_codes16(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void fail(uint32_t bit) { atomicOr(&g_prefill_err, bit); }

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

// t = s * d + t on two packed fp32 lanes (one instruction for two outputs)
__device__ __forceinline__ void ffma2(uint32_t &t_lo, uint32_t &t_hi, uint64_t s2, uint32_t d_lo, uint32_t d_hi) {
    uint64_t t, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(t) : "r"(t_lo), "r"(t_hi));
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(d_lo), "r"(d_hi));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(t) : "l"(s2), "l"(d));
    asm("mov.b64 {%0, %1}, %2;" : "=r"(t_lo), "=r"(t_hi) : "l"(t));
}

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
    using P = PCfg<ROW>;
    constexpr int kXStages = P::kXStages, kXStage = P::kXStage, kXPanel = P::kXPanel;
    constexpr int kPerKb = P::kUnitsPerKb;
    uint8_t *xring = smem;                              // [kXStages][2 panels][N rows][128 B]
    uint8_t *aring = smem + kXBytes;                    // [kASlots][2 panels][128 rows][128 B]
    uint64_t *bars = reinterpret_cast<uint64_t *>(aring + kASlots * kASlot);
    // done[u % kRing] completes when the MMAs of unit u have finished (one
    // tcgen05.commit per unit; u = 2 kb + half with block scales, u = kb
    // with one scale per row); the x producer, the decoders and the
    // epilogue all wait on it, each before its slot could be reused
    uint64_t *x_full = bars;                 // [kXStages]
    uint64_t *done = x_full + kXStages;      // [kRing]
    uint64_t *a_full = done + kRing;         // [kASlots]
    uint64_t *d_empty = a_full + kASlots;    // [2] one per half
    uint64_t *d_full = d_empty + 2;          // ROW: every MMA of the tile done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(d_full + 1);
    int *s_fail = reinterpret_cast<int *>(d_full + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kTileW;
    const int m0 = blockIdx.y * kTileX;
    const int units = kPerKb * kblocks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kXStages; ++i) mbar_init(&x_full[i], 1);
        for (int i = 0; i < kRing; ++i) mbar_init(&done[i], 1);  // tcgen05.commit
        for (int i = 0; i < kASlots; ++i) mbar_init(&a_full[i], kNumDec);  // one arrival per decoder warp
        for (int i = 0; i < 2; ++i) mbar_init(&d_empty[i], kNumEpi / 2);   // the half's epilogue warps
        mbar_init(d_full, 1);
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
        int issued = 0;  // units whose MMAs were committed
        if (lane == 0) {
            for (int u = 0; u < units; ++u) {
                const int kb = u / kPerKb, h = u % kPerKb, xs = u % kXStages, as = kb % kASlots;
                bool ok = mbar_wait_bounded(&x_full[xs], (u / kXStages) & 1) &&
                          (h == 1 || mbar_wait_bounded(&a_full[as], (kb / kASlots) & 1)) &&
                          (ROW || kb == 0 || mbar_wait_bounded(&d_empty[h], (kb - 1) & 1));
                if (!ok) {
                    fail(ERRBIT_MMA_WAIT);
                    *reinterpret_cast<volatile int *>(s_fail) = 1;
                    break;
                }
                tc_fence_after();
                // descriptors of the first 16-column slices; the others are 32
                // bytes (2 in address/16 units) apart within a 64-column panel
                const uint64_t adesc = sw128_desc(smem_u32(aring + as * kASlot));
                const uint64_t bdesc = sw128_desc(smem_u32(xring + xs * kXStage));
                const uint32_t d_tmem = tmem + (ROW ? kColT : kColD + h * 128);
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk) {
                    const uint64_t aoff = static_cast<uint64_t>((kk >> 2) * (kPanel >> 4) + (kk & 3) * 2);
                    const uint64_t boff = static_cast<uint64_t>((kk >> 2) * (kXPanel >> 4) + (kk & 3) * 2);
                    tc_mma_ss<idesc_f16<P::kN>()>(d_tmem, adesc + aoff, bdesc + boff,
                                                  (kk > 0 || (ROW && kb > 0)) ? 1u : 0u);
                }
                tc_commit(&done[u % kRing]);
                issued = u + 1;
            }
            // ROW: the epilogue's single wait (also after a failure, so that
            // it does not sit out its whole time limit)
            if (ROW) tc_commit(d_full);
            // drain: wait for the last committed unit before TMEM can be freed
            if (issued > 0 && !mbar_wait_bounded(&done[(issued - 1) % kRing], ((issued - 1) / kRing) & 1))
                fail(ERRBIT_MMA_WAIT);
        }
        __syncwarp();
    } else if (warp == kWarpTma) {
        // ------------------------------------------------------ x producer
        if (lane == 0) {
            int issued = 0;
            for (int u = 0; u < units; ++u) {
                const int xs = u % kXStages;
                if (u >= kXStages &&
                    !mbar_wait_bounded(&done[(u - kXStages) % kRing], ((u - kXStages) / kRing) & 1)) {
                    fail(ERRBIT_EMPTY_WAIT);
                    break;
                }
                if (*reinterpret_cast<volatile int *>(s_fail)) break;
                uint8_t *st = xring + xs * kXStage;
                const int kx = (u / kPerKb) * kKB, mx = m0 + (u % kPerKb) * kHalfX;
                mbar_arrive_expect_tx(&x_full[xs], kXStage);
                tma_load_2d(st, &tm_x, &x_full[xs], kx, mx);
                tma_load_2d(st + kXPanel, &tm_x, &x_full[xs], kx + 64, mx);
                issued = u + 1;
            }
            // never leave with copies in flight: wait for the last stages issued
            for (int u = issued - kXStages < 0 ? 0 : issued - kXStages; u < issued; ++u)
                if (!mbar_wait_bounded(&x_full[u % kXStages], (u / kXStages) & 1)) fail(ERRBIT_FULL_WAIT);
        }
        __syncwarp();
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------ decoders
        // thread = one weight row r; this warp converts the K half kh (64
        // codes = one 128-byte swizzled row of A panel kh) for every K block,
        // two blocks ahead of the conversion
        const int r = (warp & 3) * 32 + lane;
        const int kh = (warp - kWarpDec0) >> 2;
        const int row = n0 + r;
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
            const int as = kb % kASlots;
            load4(kb + 2, c2);  // in flight while this block is converted
            // slot `as` was last read by the MMAs of K block kb - kASlots,
            // whose last unit is kPerKb (kb - kASlots + 1) - 1
            const int prev = kPerKb * (kb - kASlots + 1) - 1;
            bool ok = kb < kASlots || mbar_wait_bounded(&done[prev % kRing], (prev / kRing) & 1);
            if (!__all_sync(0xffffffffu, ok) || *reinterpret_cast<volatile int *>(s_fail)) {
                if (lane == 0) fail(ERRBIT_EMPTY_WAIT);
                break;
            }
            uint8_t *arow = aring + as * kASlot + kh * kPanel + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 c = c0[j];
                // 16 codes -> two 16-byte chunks (2j, 2j + 1) of this row
                uint4 lo, hi;
                lo.x = e4m3x2_to_bf16x2(c.x, 0x9180u);
                lo.y = e4m3x2_to_bf16x2(c.x, 0xB3A2u);
                lo.z = e4m3x2_to_bf16x2(c.y, 0x9180u);
                lo.w = e4m3x2_to_bf16x2(c.y, 0xB3A2u);
                hi.x = e4m3x2_to_bf16x2(c.z, 0x9180u);
                hi.y = e4m3x2_to_bf16x2(c.z, 0xB3A2u);
                hi.z = e4m3x2_to_bf16x2(c.w, 0x9180u);
                hi.w = e4m3x2_to_bf16x2(c.w, 0xB3A2u);
                *reinterpret_cast<uint4 *>(arow + (((2 * j) ^ (r & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(arow + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
            }
            fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
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
        // thread = one weight row (TMEM lane of quarter q); this warp owns
        // the 128 accumulator columns (rows of x) of half h
        const int q = warp & 3;
        const int h = (warp - kWarpEpi0) >> 2;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t t_addr = lane_base + kColT + h * 128;
        const uint32_t d_addr = lane_base + kColD + h * 128;
        const int row = n0 + q * 32 + lane;
        bool ok = true;
        if (ROW) {
            ok = mbar_wait_bounded(d_full, 0);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail(ERRBIT_FULL_WAIT);
                ok = false;
            } else {
                ok = *reinterpret_cast<volatile int *>(s_fail) == 0;
            }
        } else {
            const float *srow = scales + static_cast<int64_t>(blockIdx.x) * kblocks;
            for (int kb = 0; kb < kblocks; ++kb) {
                const float s = __ldg(srow + kb);
                uint64_t s2;
                asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(s));
                const int u = 2 * kb + h;
                ok = mbar_wait_bounded(&done[u % kRing], (u / kRing) & 1);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) fail(ERRBIT_FULL_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                // T_h += s * D_h, 16 columns at a time; the loads of chunk
                // c + 1 are in flight while chunk c is combined and stored
                uint32_t dv[2][16], tv[2][16];
                tc_ld16(d_addr, dv[0]);
                if (kb > 0) tc_ld16(t_addr, tv[0]);
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int cur = c & 1, nxt = cur ^ 1;
                    if (c + 1 < 8) {
                        tc_ld16(d_addr + 16 * (c + 1), dv[nxt]);
                        if (kb > 0) tc_ld16(t_addr + 16 * (c + 1), tv[nxt]);
                    }
                    if (kb > 0) {
#pragma unroll
                        for (int i = 0; i < 16; i += 2) ffma2(tv[cur][i], tv[cur][i + 1], s2, dv[cur][i], dv[cur][i + 1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) tv[cur][i] = __float_as_uint(s * __uint_as_float(dv[cur][i]));
                    }
                    tc_st16(t_addr + 16 * c, tv[cur]);
                    tc_wait_ld();
                }
                // D_h has been read: the next unit of this half may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_empty[h]);
                tc_wait_st();  // T_h is read again by the next K block
            }
        }
        // thread = weight row, column j of T_h = y[m0 + 128 h + j][row]
        if (ok) {
            tc_fence_after();
            const float rs = !ROW ? 1.0f : (row < n ? __ldg(scales + static_cast<int64_t>(row) * row_stride) : 0.0f);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[16];
                tc_ld16(t_addr + 16 * c, v);
                tc_wait_ld();
                if (row < n) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int mi = m0 + h * kHalfX + 16 * c + i;
                        const float val = ROW ? __uint_as_float(v[i]) * rs : __uint_as_float(v[i]);
                        if (mi < m) y[static_cast<int64_t>(mi) * n + row] = __float2bfloat16_rn(val);
                    }
                }
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
    // one TMA box = the x rows of one MMA unit (a half with block scales, all
    // 256 with one scale per row)
    const uint32_t box_rows = row ? static_cast<uint32_t>(PCfg<true>::kN) : static_cast<uint32_t>(PCfg<false>::kN);
    if (!encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, k, m, k * 2, 64, box_rows,
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
