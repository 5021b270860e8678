// quantize.cu -- load-time requantization kernels.
//
//  * block_quantize_kernel: bf16 [n,k] -> e4m3 codes + one fp32 scale per
//    128x128 tile (Atlas spark_model/weight_map/quantize_fp8_bs.rs: one CTA
//    per tile, grid [k_blocks, n_blocks]; FreeToken PR #636
//    per_block_quant_fp8).  Each thread keeps its 32 elements in registers
//    between the amax reduction and the encode, so the tile is read from HBM
//    exactly once.
//  * mx_quantize_kernel: bf16 [n,k] -> e4m3 codes + one e8m0 exponent per 32
//    consecutive k of a row (FreeToken issue #624).  Four lanes own one
//    32-element group (16 bytes each, fully coalesced), the group amax comes
//    from two shuffles, and no fp32 copy of the weight is ever formed.
//  * row_quantize_kernel / tensor_*_kernel: one fp32 scale per output row
//    or per weight (FreeToken PR #389, What this adds / Why), the same rule
//    as a tile: s = amax / 448 over the row (tensor), s = 1 if all zero.
//    Per row is one CTA per row; per tensor is a grid-wide amax (atomicMax
//    on the fp32 bit pattern, which orders like the value for |w| >= 0, so
//    the result is the exact maximum whatever the order) into the scale
//    slot, an encode pass that derives s from it, and a one-thread pass
//    that replaces the amax by s.
//  * *_generic kernels: scalar versions of the same arithmetic for shapes or
//    pointers the vector kernels cannot take (k % 8 != 0, unaligned w).
//
// The arithmetic is fixed by the definition: amax in fp32, s = amax / 448.f
// as an IEEE fp32 division, the code of the IEEE quotient w / s,
// cvt.rn.satfinite to e4m3.  MX scales are exact powers of two, so
// w * 2^(127-E) is exact wherever it matters.
//
// The vector kernels form w / s with Markstein's correction (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): y = RN(1/s) once per tile,
// q0 = RN(w y), r = w - s q0 exactly by fma, q = RN(q0 + r y), sign copied
// from w.  Over every positive finite bf16 amax with s >= 2^-92 and every
// bf16 |w| <= amax (1.03e9 pairs, checked exhaustively on the host) the e4m3
// code of q equals the code of the IEEE quotient; the quotients themselves
// differ only where the residual falls below the normal range, far below the
// first e4m3 rounding boundary.  Tiles with s < 2^-92 take the IEEE division.
#include "common.cuh"
#include "internal.h"

namespace fp8bs {

namespace {

constexpr int kTile = 128;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Two bf16 values (as fp32) divided by s with Markstein's correction (see
// above), q0 = RN(w y), r = w - s q0, q = RN(q0 + r y), the sign copied from
// w, on both values at once with packed fp32x2 fma (each lane rounds exactly
// like the scalar fma; q0 = fma(w, y, -0) = RN(w y)): ns2 = (-s, -s),
// y2 = (y, y), y = RN(1/s).  Returns the two e4m3 codes.
__device__ __forceinline__ uint16_t encode2_mk(float wlo, float whi, uint64_t ns2, uint64_t y2) {
    const uint64_t negzero2 = 0x8000000080000000ull;
    uint64_t w2, q0, r, q;
    asm("mov.b64 %0, {%1, %2};" : "=l"(w2) : "f"(wlo), "f"(whi));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q0) : "l"(w2), "l"(y2), "l"(negzero2));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(ns2), "l"(q0), "l"(w2));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(y2), "l"(q0));
    float qlo, qhi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(qlo), "=f"(qhi) : "l"(q));
    return f32x2_to_e4m3x2(copysignf(qlo, wlo), copysignf(qhi, whi));
}

// Encode 8 bf16 values divided by s into 8 e4m3 bytes.
__device__ __forceinline__ uint2 encode8_mk(const uint4 v, float s, float y) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint64_t ns2, y2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(ns2) : "f"(-s));
    asm("mov.b64 %0, {%1, %1};" : "=l"(y2) : "f"(y));
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint16_t c0 = encode2_mk(bf16lo_to_f32(w[2 * h]), bf16hi_to_f32(w[2 * h]), ns2, y2);
        const uint16_t c1 = encode2_mk(bf16lo_to_f32(w[2 * h + 1]), bf16hi_to_f32(w[2 * h + 1]), ns2, y2);
        out[h] = static_cast<uint32_t>(c0) | (static_cast<uint32_t>(c1) << 16);
    }
    return make_uint2(out[0], out[1]);
}

// The code of v / s for 8 values: Markstein's quotient where it is exact
// for the encode (s >= 2^-92), the IEEE division otherwise; `y` is RN(1/s)
// or anything when s < 2^-92.  s is uniform over a tile, row or tensor.
__device__ __forceinline__ uint2 encode8_quot(const uint4 v, float s, float y) {
    return s >= 0x1p-92f ? encode8_mk(v, s, y) : encode8_div(v, s);
}

__device__ __forceinline__ float recip_for(float s) { return s >= 0x1p-92f ? __frcp_rn(s) : 0.0f; }

__device__ __forceinline__ uint2 encode8_mul(const uint4 v, float f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint16_t c0 = f32x2_to_e4m3x2(bf16lo_to_f32(w[2 * h]) * f, bf16hi_to_f32(w[2 * h]) * f);
        const uint16_t c1 =
            f32x2_to_e4m3x2(bf16lo_to_f32(w[2 * h + 1]) * f, bf16hi_to_f32(w[2 * h + 1]) * f);
        out[h] = static_cast<uint32_t>(c0) | (static_cast<uint32_t>(c1) << 16);
    }
    return make_uint2(out[0], out[1]);
}

// max |w| over 8 bf16 values, folded into m.  Magnitudes of finite bf16
// values order like their 15-bit patterns, so the maximum is taken on the
// packed integer halves.
__device__ __forceinline__ float absmax8(const uint4 v, float m) {
    uint32_t mx = max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    mx = max_u16x2(mx, v.z & 0x7FFF7FFFu);
    mx = max_u16x2(mx, v.w & 0x7FFF7FFFu);
    const uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);
    return fmaxf(m, __uint_as_float(m16 << 16));
}

// MX exponent from the group amax (a non-negative bf16 value held in fp32):
// e = smallest integer with 448 * 2^e >= amax.  Writing amax = m * 2^p with
// m in [1, 2): 448 * 2^(p-8) = 1.75 * 2^p >= amax iff m <= 1.75, so
// e = p - 8 + (m > 1.75).  In the fp32 encoding p = field - 127 and
// m > 1.75 iff the 23-bit mantissa exceeds 0x600000.  Subnormal amax gives
// e + 127 < 0 and clamps to E = 0; amax = 0 gives E = 127 by definition.
__device__ __forceinline__ int mx_exponent(float amax) {
    if (amax == 0.0f) return 127;
    const uint32_t u = __float_as_uint(amax);
    const int field = static_cast<int>(u >> 23);
    if (field == 0) return 0;
    const int E = field - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return E < 0 ? 0 : (E > 254 ? 254 : E);
}

// 2^(127 - E) as an fp32 value, exact for E in [0, 254].
__device__ __forceinline__ float mx_inv_scale(int E) {
    const int t = 254 - E;  // biased exponent of 2^(127-E)
    return t >= 1 ? __uint_as_float(static_cast<uint32_t>(t) << 23) : __uint_as_float(0x00400000u);
}

// ------------------------------------------------------------ block, fast
// 256 threads per 128x128 tile: thread t owns the 16-byte chunk t % 16 of
// rows t / 16 + 16 i (i < 8), i.e. 64 elements kept in registers between the
// tile-amax reduction and the encode; four CTAs per SM keep four tiles'
// loads in flight while others reduce and encode (measured against 512 x 2,
// 256 x 3, 128 x 8 and 1024 x 1 threads x CTAs per SM: 69.6 us vs 94.7 /
// 76.8 / 99.0 / 143 us for the [18432, 7168] weight).
constexpr int kQThreads = 256;
constexpr int kQRows = kQThreads / 16;  // rows covered per pass

__global__ void __launch_bounds__(kQThreads, 4) block_quantize_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                    uint8_t *__restrict__ codes,
                                                                    float *__restrict__ scales,
                                                                    int64_t n, int64_t k) {
    __shared__ float warp_amax[kQThreads / 32];
    const int bk = blockIdx.x, bn = blockIdx.y;
    const int chunk = threadIdx.x & 15;  // 8 bf16 = 16 bytes
    const int rg = threadIdx.x >> 4;     // rows rg + kQRows i
    const int64_t col = static_cast<int64_t>(bk) * kTile + chunk * 8;
    const bool col_ok = col < k;  // k % 8 == 0: a chunk is all in or all out

    uint4 v[kTile / kQRows];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kTile / kQRows; ++i) {
        const int64_t row = static_cast<int64_t>(bn) * kTile + rg + kQRows * i;
        if (col_ok && row < n)
            v[i] = ld_nc_v4(w + row * k + col);
        else
            v[i] = make_uint4(0, 0, 0, 0);  // padding: |0| never raises amax
    }
#pragma unroll
    for (int i = 0; i < kTile / kQRows; ++i) amax = absmax8(v[i], amax);
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) warp_amax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = warp_amax[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, warp_amax[i]);
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    const float y = recip_for(s);
    if (threadIdx.x == 0) scales[static_cast<int64_t>(bn) * gridDim.x + bk] = s;
#pragma unroll
    for (int i = 0; i < kTile / kQRows; ++i) {
        const int64_t row = static_cast<int64_t>(bn) * kTile + rg + kQRows * i;
        if (col_ok && row < n) {
            const uint2 c = encode8_quot(v[i], s, y);
            *reinterpret_cast<uint2 *>(codes + row * k + col) = c;
        }
    }
}

// --------------------------------------------------------- block, generic
__global__ void __launch_bounds__(256) block_quantize_generic_kernel(
    const __nv_bfloat16 *__restrict__ w, uint8_t *__restrict__ codes, float *__restrict__ scales,
    int64_t n, int64_t k) {
    __shared__ float warp_amax[8];
    const int bk = blockIdx.x, bn = blockIdx.y;
    const int64_t r0 = static_cast<int64_t>(bn) * kTile, c0 = static_cast<int64_t>(bk) * kTile;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), n - r0));
    const int cols = static_cast<int>(min(static_cast<int64_t>(kTile), k - c0));
    const uint16_t *wb = reinterpret_cast<const uint16_t *>(w);
    float amax = 0.0f;
    for (int e = threadIdx.x; e < rows * cols; e += blockDim.x) {
        const int r = e / cols, c = e % cols;
        amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(wb[(r0 + r) * k + c0 + c]) << 16)));
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) warp_amax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = warp_amax[0];
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_amax[i]);
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    if (threadIdx.x == 0) scales[static_cast<int64_t>(bn) * gridDim.x + bk] = s;
    for (int e = threadIdx.x; e < rows * cols; e += blockDim.x) {
        const int r = e / cols, c = e % cols;
        const float q = __uint_as_float(static_cast<uint32_t>(wb[(r0 + r) * k + c0 + c]) << 16) / s;
        codes[(r0 + r) * k + c0 + c] = static_cast<uint8_t>(f32x2_to_e4m3x2(q, 0.0f) & 0xFF);
    }
}

// --------------------------------------------------------------- MX, fast
// Thread layout: each row of k bf16 is cut into 4*G chunks of 8 elements
// (G = ceil(k/32) groups); chunks past k are padding.  A block of 256 threads
// covers kMxUnroll consecutive 256-chunk slabs (that many independent 16-byte
// loads in flight per thread; 2 measured faster than 4 or 8).  Lanes
// 4j..4j+3 hold one group.
constexpr int kMxThreads = 256;
constexpr int kMxUnroll = 2;

// Unsigned 32-bit division by a divisor fixed for the launch, by a multiply
// high and shifts (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994, the round-down-with-add form): for divisor
// d >= 2, l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1 (< 2^32), and
// q / d = (t + ((q - t) >> 1)) >> (l - 1) with t = umulhi(m, q), exact for
// every 32-bit q.  The host computes m and l (div_magic below).
struct DivMagic {
    uint32_t m, l;
};

DivMagic div_magic(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return {static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ uint32_t div_by(uint32_t q, DivMagic dm) {
    const uint32_t t = __umulhi(dm.m, q);
    return (t + ((q - t) >> 1)) >> (dm.l - 1);
}

// One thread per 16-byte chunk (8 elements; four chunks = one 32-element
// group, reduced with two shuffles).  The flat chunk index fits 32 bits
// (the launcher sends larger tensors to the generic kernel).
__global__ void __launch_bounds__(kMxThreads) mx_quantize_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                 uint8_t *__restrict__ codes,
                                                                 uint8_t *__restrict__ e8m0,
                                                                 int64_t n, int64_t k,
                                                                 int64_t groups, DivMagic per_row) {
    const uint32_t chunks_per_row = static_cast<uint32_t>(groups * 4);
    const uint32_t total = static_cast<uint32_t>(n * chunks_per_row);
    const uint32_t base = blockIdx.x * (kMxThreads * kMxUnroll) + threadIdx.x;
    uint4 v[kMxUnroll];
    int64_t row[kMxUnroll], col[kMxUnroll];
    bool ok[kMxUnroll];
#pragma unroll
    for (int u = 0; u < kMxUnroll; ++u) {
        const uint32_t q = base + u * kMxThreads;
        const bool in = q < total;
        const uint32_t r = in ? div_by(q, per_row) : 0u;
        row[u] = r;
        col[u] = in ? static_cast<int64_t>(q - r * chunks_per_row) * 8 : 0;
        ok[u] = in && col[u] < k;
        v[u] = ok[u] ? ld_nc_v4(w + row[u] * k + col[u]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kMxUnroll; ++u) {
        float amax = absmax8(v[u], 0.0f);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int E = mx_exponent(amax);
        if (ok[u]) {
            const uint2 c = encode8_mul(v[u], mx_inv_scale(E));
            *reinterpret_cast<uint2 *>(codes + row[u] * k + col[u]) = c;
            if ((threadIdx.x & 3) == 0) e8m0[row[u] * groups + col[u] / 32] = static_cast<uint8_t>(E);
        }
    }
}

// k a multiple of 32: chunk q of the flat [n, k] array starts at element 8q
// and lies in 32-element group q / 4 of the flat [n, k / 32] exponent array,
// so no row or column is formed (the per-chunk division and 64-bit index
// arithmetic of the kernel above made it issue-bound).  The flat chunk index
// fits 32 bits (the launcher checks).
constexpr int kMxFlatUnroll = 4;
__global__ void __launch_bounds__(kMxThreads) mx_quantize_flat_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                      uint8_t *__restrict__ codes,
                                                                      uint8_t *__restrict__ e8m0, uint32_t total) {
    const uint32_t base = blockIdx.x * (kMxThreads * kMxFlatUnroll) + threadIdx.x;
    uint4 v[kMxFlatUnroll];
#pragma unroll
    for (int u = 0; u < kMxFlatUnroll; ++u) {
        const uint32_t q = base + u * kMxThreads;
        v[u] = q < total ? ld_nc_v4(w + 8 * static_cast<uint64_t>(q)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kMxFlatUnroll; ++u) {
        const uint32_t q = base + u * kMxThreads;
        float amax = absmax8(v[u], 0.0f);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int E = mx_exponent(amax);
        if (q < total) {
            *reinterpret_cast<uint2 *>(codes + 8 * static_cast<uint64_t>(q)) = encode8_mul(v[u], mx_inv_scale(E));
            if ((threadIdx.x & 3) == 0) e8m0[q >> 2] = static_cast<uint8_t>(E);
        }
    }
}

// ------------------------------------------------------------ MX, generic
__global__ void __launch_bounds__(256) mx_quantize_generic_kernel(
    const __nv_bfloat16 *__restrict__ w, uint8_t *__restrict__ codes, uint8_t *__restrict__ e8m0,
    int64_t n, int64_t k, int64_t groups) {
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (g >= n * groups) return;
    const int64_t r = g / groups, c0 = (g - r * groups) * 32;
    const int len = static_cast<int>(min(static_cast<int64_t>(32), k - c0));
    const uint16_t *wb = reinterpret_cast<const uint16_t *>(w) + r * k + c0;
    float amax = 0.0f;
    for (int i = 0; i < len; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(wb[i]) << 16)));
    const int E = mx_exponent(amax);
    const float f = mx_inv_scale(E);
    for (int i = 0; i < len; ++i) {
        const float q = __uint_as_float(static_cast<uint32_t>(wb[i]) << 16) * f;
        codes[r * k + c0 + i] = static_cast<uint8_t>(f32x2_to_e4m3x2(q, 0.0f) & 0xFF);
    }
    e8m0[g] = static_cast<uint8_t>(E);
}

// --------------------------------------------------------------- per row
// One CTA per weight row.  The row's 16-byte chunks are dealt round-robin to
// 256 threads; the first kRowHeld chunks of each thread stay in registers
// between the amax reduction and the encode, so rows of up to
// 256 * 8 * kRowHeld = 8192 elements are read from HBM once (longer rows
// read the remainder a second time, from L2).
constexpr int kRowThreads = 256;
constexpr int kRowHeld = 4;

__device__ __forceinline__ float cta_max(float v, float *warp_slots) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) warp_slots[threadIdx.x >> 5] = v;
    __syncthreads();
    v = warp_slots[0];
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) v = fmaxf(v, warp_slots[i]);
    return v;
}

__global__ void __launch_bounds__(kRowThreads) row_quantize_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                 uint8_t *__restrict__ codes,
                                                                 float *__restrict__ scales, int64_t k) {
    __shared__ float warp_amax[kRowThreads / 32];
    const int64_t row = blockIdx.x;
    const __nv_bfloat16 *wr = w + row * k;
    uint8_t *cr = codes + row * k;
    const int64_t chunks = k / 8;  // k % 8 == 0 on this path
    uint4 v[kRowHeld];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kRowHeld; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * kRowThreads;
        v[i] = c < chunks ? ld_nc_v4(wr + c * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kRowHeld; ++i) amax = absmax8(v[i], amax);
    for (int64_t c = threadIdx.x + kRowHeld * kRowThreads; c < chunks; c += kRowThreads)
        amax = absmax8(ld_nc_v4(wr + c * 8), amax);
    amax = cta_max(amax, warp_amax);
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    const float y = recip_for(s);
    if (threadIdx.x == 0) scales[row] = s;
#pragma unroll
    for (int i = 0; i < kRowHeld; ++i) {
        const int64_t c = threadIdx.x + static_cast<int64_t>(i) * kRowThreads;
        if (c < chunks) *reinterpret_cast<uint2 *>(cr + c * 8) = encode8_quot(v[i], s, y);
    }
    for (int64_t c = threadIdx.x + kRowHeld * kRowThreads; c < chunks; c += kRowThreads)
        *reinterpret_cast<uint2 *>(cr + c * 8) = encode8_quot(ld_nc_v4(wr + c * 8), s, y);
}

__global__ void __launch_bounds__(kRowThreads) row_quantize_generic_kernel(
    const __nv_bfloat16 *__restrict__ w, uint8_t *__restrict__ codes, float *__restrict__ scales, int64_t k) {
    __shared__ float warp_amax[kRowThreads / 32];
    const int64_t row = blockIdx.x;
    const uint16_t *wb = reinterpret_cast<const uint16_t *>(w) + row * k;
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < k; c += kRowThreads)
        amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(wb[c]) << 16)));
    amax = cta_max(amax, warp_amax);
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    if (threadIdx.x == 0) scales[row] = s;
    for (int64_t c = threadIdx.x; c < k; c += kRowThreads) {
        const float q = __uint_as_float(static_cast<uint32_t>(wb[c]) << 16) / s;
        codes[row * k + c] = static_cast<uint8_t>(f32x2_to_e4m3x2(q, 0.0f) & 0xFF);
    }
}

// ------------------------------------------------------------ per tensor
// The weight is one flat array of total = n*k elements.  VEC: total % 8 == 0
// and 16-byte aligned w / 8-byte aligned codes, 16-byte chunks.
constexpr int kTensorThreads = 256;

template <bool VEC>
__global__ void __launch_bounds__(kTensorThreads) tensor_amax_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                   int64_t total,
                                                                   uint32_t *__restrict__ amax_bits) {
    __shared__ float warp_amax[kTensorThreads / 32];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTensorThreads;
    float amax = 0.0f;
    if (VEC) {
        // four independent 16-byte loads in flight per thread per step
        const int64_t n8 = total / 8;
        for (int64_t c = static_cast<int64_t>(blockIdx.x) * kTensorThreads + threadIdx.x; c < n8; c += 4 * stride) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = c + u * stride < n8 ? ld_nc_v4(w + (c + u * stride) * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) amax = absmax8(v[u], amax);
        }
    } else {
        const uint16_t *wb = reinterpret_cast<const uint16_t *>(w);
        for (int64_t e = static_cast<int64_t>(blockIdx.x) * kTensorThreads + threadIdx.x; e < total; e += stride)
            amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(wb[e]) << 16)));
    }
    amax = cta_max(amax, warp_amax);
    if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(amax));
}

template <bool VEC>
__global__ void __launch_bounds__(kTensorThreads) tensor_encode_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                     int64_t total, uint8_t *__restrict__ codes,
                                                                     const uint32_t *__restrict__ amax_bits) {
    const float amax = __uint_as_float(*amax_bits);
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    const float y = recip_for(s);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTensorThreads;
    // Walk the tensor back to front: the amax pass just read it front to
    // back, so its last part is still in L2 when this pass starts.
    if (VEC) {
        const int64_t n8 = total / 8;
        for (int64_t c = static_cast<int64_t>(blockIdx.x) * kTensorThreads + threadIdx.x; c < n8; c += 4 * stride) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = c + u * stride < n8 ? ld_nc_v4(w + (n8 - 1 - (c + u * stride)) * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c + u * stride < n8)
                    *reinterpret_cast<uint2 *>(codes + (n8 - 1 - (c + u * stride)) * 8) = encode8_quot(v[u], s, y);
        }
    } else {
        const uint16_t *wb = reinterpret_cast<const uint16_t *>(w);
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * kTensorThreads + threadIdx.x; i < total; i += stride) {
            const int64_t e = total - 1 - i;
            const float q = __uint_as_float(static_cast<uint32_t>(wb[e]) << 16) / s;
            codes[e] = static_cast<uint8_t>(f32x2_to_e4m3x2(q, 0.0f) & 0xFF);
        }
    }
}

// Replace the accumulated amax in the scale slot by s (after every encode
// CTA has read it: stream order).
__global__ void tensor_finalize_kernel(float *scale) {
    if (threadIdx.x == 0) {
        const float amax = *scale;
        *scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    }
}

// ------------------------------------------------- small per-tensor (one CTA)
// Activations at decode sizes: amax and cast in one launch of one CTA (the
// per-call cost, not the bytes, dominates there); same arithmetic as the
// grid-wide per-tensor path, so a tensor quantizes to the same bits either way.
constexpr int kActThreads = 1024;

template <bool VEC>
__global__ void __launch_bounds__(kActThreads) tensor_quantize_small_kernel(const __nv_bfloat16 *__restrict__ w,
                                                                          int64_t total, uint8_t *__restrict__ codes,
                                                                          float *__restrict__ scale) {
    __shared__ float warp_amax[kActThreads / 32];
    const uint16_t *wb = reinterpret_cast<const uint16_t *>(w);
    float amax = 0.0f;
    if (VEC) {
        for (int64_t c = threadIdx.x; c < total / 8; c += kActThreads) amax = absmax8(ld_nc_v4(w + c * 8), amax);
    } else {
        for (int64_t e = threadIdx.x; e < total; e += kActThreads)
            amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(wb[e]) << 16)));
    }
    amax = cta_max(amax, warp_amax);
    const float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
    const float y = recip_for(s);
    if (threadIdx.x == 0) *scale = s;
    if (VEC) {
        for (int64_t c = threadIdx.x; c < total / 8; c += kActThreads)
            *reinterpret_cast<uint2 *>(codes + c * 8) = encode8_quot(ld_nc_v4(w + c * 8), s, y);
    } else {
        for (int64_t e = threadIdx.x; e < total; e += kActThreads) {
            const float q = __uint_as_float(static_cast<uint32_t>(wb[e]) << 16) / s;
            codes[e] = static_cast<uint8_t>(f32x2_to_e4m3x2(q, 0.0f) & 0xFF);
        }
    }
}

}  // namespace

cudaError_t launch_block_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                                  float *scales, bool vector_ok, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((k + kTile - 1) / kTile),
                    static_cast<unsigned>((n + kTile - 1) / kTile));
    if (vector_ok)
        block_quantize_kernel<<<grid, kQThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w), codes,
                                                              scales, n, k);
    else
        block_quantize_generic_kernel<<<grid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(w), codes, scales, n, k);
    return cudaGetLastError();
}

cudaError_t launch_mx_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                               uint8_t *e8m0, bool vector_ok, cudaStream_t stream) {
    const int64_t groups = (k + 31) / 32;
    const int64_t per_block = kMxThreads * kMxUnroll;
    const int64_t total = n * groups * 4;
    const int64_t flat_block = kMxThreads * kMxFlatUnroll;
    if (vector_ok && k % 32 == 0 && total + flat_block < (int64_t(1) << 32)) {
        const unsigned blocks = static_cast<unsigned>((total + flat_block - 1) / flat_block);
        mx_quantize_flat_kernel<<<blocks, kMxThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w), codes,
                                                                    e8m0, static_cast<uint32_t>(total));
    } else if (vector_ok && total + per_block < (int64_t(1) << 32)) {
        const unsigned blocks = static_cast<unsigned>((total + per_block - 1) / per_block);
        mx_quantize_kernel<<<blocks, kMxThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w),
                                                               codes, e8m0, n, k, groups,
                                                               div_magic(static_cast<uint32_t>(groups * 4)));
    } else {
        const int64_t total = n * groups;
        const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
        mx_quantize_generic_kernel<<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(w), codes, e8m0, n, k, groups);
    }
    return cudaGetLastError();
}

cudaError_t launch_row_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                                float *scales, bool vector_ok, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>(n);
    if (vector_ok)
        row_quantize_kernel<<<blocks, kRowThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w), codes,
                                                                scales, k);
    else
        row_quantize_generic_kernel<<<blocks, kRowThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(w),
                                                                        codes, scales, k);
    return cudaGetLastError();
}

cudaError_t launch_tensor_quantize(const void *w, int64_t n, int64_t k, uint8_t *codes,
                                   float *scale, bool vector_ok, cudaStream_t stream) {
    const int64_t total = n * k;
    const int64_t units = vector_ok ? total / 8 : total;
    // enough CTAs to fill every SM several times over, never more than the work
    int64_t blocks = static_cast<int64_t>(device_sm_count()) * 8;
    const int64_t need = (units + kTensorThreads - 1) / kTensorThreads;
    if (blocks > need) blocks = need;
    if (blocks < 1) blocks = 1;
    const __nv_bfloat16 *wb = static_cast<const __nv_bfloat16 *>(w);
    uint32_t *amax_bits = reinterpret_cast<uint32_t *>(scale);
    cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    const unsigned g = static_cast<unsigned>(blocks);
    if (vector_ok) {
        tensor_amax_kernel<true><<<g, kTensorThreads, 0, stream>>>(wb, total, amax_bits);
        tensor_encode_kernel<true><<<g, kTensorThreads, 0, stream>>>(wb, total, codes, amax_bits);
    } else {
        tensor_amax_kernel<false><<<g, kTensorThreads, 0, stream>>>(wb, total, amax_bits);
        tensor_encode_kernel<false><<<g, kTensorThreads, 0, stream>>>(wb, total, codes, amax_bits);
    }
    tensor_finalize_kernel<<<1, 32, 0, stream>>>(scale);
    return cudaGetLastError();
}

cudaError_t launch_act_quantize(const void *x, int64_t m, int64_t k, uint8_t *codes, float *scale,
                                bool vector_ok, cudaStream_t stream) {
    const int64_t total = m * k;
    if (total > kActSmall) return launch_tensor_quantize(x, m, k, codes, scale, vector_ok, stream);
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    if (vector_ok)
        tensor_quantize_small_kernel<true><<<1, kActThreads, 0, stream>>>(xb, total, codes, scale);
    else
        tensor_quantize_small_kernel<false><<<1, kActThreads, 0, stream>>>(xb, total, codes, scale);
    return cudaGetLastError();
}

namespace {

// Test hook: the quantizers' e4m3 encode step (f32x2_to_e4m3x2) over
// consecutive binary32 bit patterns, four per thread and one 32-bit store.
__global__ void encode_probe_kernel(uint32_t first, int64_t quads, uint32_t *__restrict__ out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < quads; i += stride) {
        const uint32_t b = first + static_cast<uint32_t>(4 * i);
        const uint32_t lo = f32x2_to_e4m3x2(__uint_as_float(b), __uint_as_float(b + 1u));
        const uint32_t hi = f32x2_to_e4m3x2(__uint_as_float(b + 2u), __uint_as_float(b + 3u));
        out[i] = lo | (hi << 16);
    }
}

}  // namespace

cudaError_t launch_encode_probe(uint32_t first, int64_t count, uint8_t *codes, cudaStream_t stream) {
    const int64_t quads = count / 4;
    int64_t blocks = (quads + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    encode_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(first, quads,
                                                                          reinterpret_cast<uint32_t *>(codes));
    return cudaGetLastError();
}

}  // namespace fp8bs
