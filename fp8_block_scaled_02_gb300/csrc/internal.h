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

// decode.cu -- TMA-staged skinny GEMM, m <= 32 per launch.
struct DecodeArgs {
    const void *x;           // bf16 [m, k] (row offset already applied)
    const uint8_t *codes;    // e4m3 [n, k]
    const float *scales;     // block scales [ceil(n/128), ceil(k/128)] or nullptr
    const uint8_t *e8m0;     // MX exponents [n, ceil(k/32)] or nullptr
    void *y;                 // bf16 [m, n] (row offset already applied)
    int64_t m, n, k;
};
cudaError_t launch_decode(const DecodeArgs &a, bool mx, cudaStream_t stream);
uint32_t take_decode_error();  // reads and clears the decode kernels' error word

// generic.cu -- plain-load kernels for any shape / alignment.
cudaError_t launch_generic_gemv(const DecodeArgs &a, bool mx, cudaStream_t stream);

// prefill.cu -- tcgen05 block-FP8 GEMM for larger m.
cudaError_t launch_prefill(const DecodeArgs &a, cudaStream_t stream);
uint32_t take_prefill_error();

// tensormap.cu -- cuTensorMapEncodeTiled through the runtime's driver entry
// point (no link against libcuda).
bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Multiprocessor count of the current device (cached per device).
int device_sm_count();

}  // namespace fp8bs
