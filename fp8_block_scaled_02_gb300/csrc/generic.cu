// generic.cu -- plain-load W8A16 GEMV for any shape and alignment (k not a
// multiple of 16, unaligned x or codes).  Same arithmetic as the decode
// kernel: exact e4m3 -> bf16 -> fp32 decode, fp32 partial sums per scale
// group (128 columns for block FP8, 32 for MXFP8) multiplied by that group's
// scale, bf16 rounding once at the end.  With one scale per row (or tensor)
// the whole row sums unscaled and its scale multiplies the total.  One warp per weight row; rows of x
// in chunks of 8.  Correctness path only -- the fast paths are decode.cu and
// prefill.cu.
#include "common.cuh"
#include "internal.h"

namespace fp8bs {

namespace {

constexpr int kRowsPerBlock = 8;  // warps per CTA, one weight row each

__device__ __forceinline__ float decode_e4m3(uint8_t code) {
    return bf16lo_to_f32(e4m3x2_to_bf16x2(code, 0x9180u));
}

template <int SC>
__global__ void __launch_bounds__(kRowsPerBlock * 32) generic_gemv_kernel(
    const uint16_t *__restrict__ x, int64_t m, const uint8_t *__restrict__ codes,
    const float *__restrict__ scales, const uint8_t *__restrict__ e8m0, uint16_t *__restrict__ y,
    int64_t n, int64_t k, int row_stride) {
    constexpr bool MX = SC == kScaleMx, ROW = SC == kScaleRow;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= n) return;  // whole warp leaves together
    pdl_wait();
    const int64_t kblocks = (k + 127) / 128, groups = (k + 31) / 32;
    const int gsz = MX ? 32 : 128;
    const uint8_t *wrow = codes + row * k;
    for (int64_t m0 = 0; m0 < m; m0 += 8) {
        const int mc = static_cast<int>(min(static_cast<int64_t>(8), m - m0));
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int64_t c0 = 0; c0 < k; c0 += gsz) {
            float part[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = 0.0f;
            const int64_t c1 = min(static_cast<int64_t>(k), c0 + gsz);
            for (int64_t c = c0 + lane; c < c1; c += 32) {
                const float wv = decode_e4m3(wrow[c]);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < mc)
                        part[i] = fmaf(__uint_as_float(static_cast<uint32_t>(x[(m0 + i) * k + c]) << 16), wv,
                                       part[i]);
            }
            float s;
            if (ROW) {
                s = 1.0f;
            } else if (MX) {
                const uint32_t E = e8m0[row * groups + c0 / 32];
                s = E ? __uint_as_float(E << 23) : __uint_as_float(0x00400000u);
            } else {
                s = scales[(row / 128) * kblocks + c0 / 128];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(s, part[i], acc[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0 && i < mc) {
                const __nv_bfloat16 b = __float2bfloat16_rn(ROW ? v * scales[row * row_stride] : v);
                y[(m0 + i) * n + row] = *reinterpret_cast<const uint16_t *>(&b);
            }
        }
    }
}

}  // namespace

cudaError_t launch_generic_gemv(const DecodeArgs &a, cudaStream_t stream) {
    const unsigned blocks = static_cast<unsigned>((a.n + kRowsPerBlock - 1) / kRowsPerBlock);
    const uint16_t *x = static_cast<const uint16_t *>(a.x);
    uint16_t *y = static_cast<uint16_t *>(a.y);
    constexpr int kT = kRowsPerBlock * 32;
    switch (a.kind) {
        case kScaleBlock:
            generic_gemv_kernel<kScaleBlock><<<blocks, kT, 0, stream>>>(x, a.m, a.codes, a.scales, nullptr, y, a.n,
                                                                        a.k, 0);
            break;
        case kScaleMx:
            generic_gemv_kernel<kScaleMx><<<blocks, kT, 0, stream>>>(x, a.m, a.codes, nullptr, a.e8m0, y, a.n, a.k,
                                                                     0);
            break;
        case kScaleRow:
            generic_gemv_kernel<kScaleRow><<<blocks, kT, 0, stream>>>(x, a.m, a.codes, a.scales, nullptr, y, a.n,
                                                                      a.k, a.row_stride);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace fp8bs
