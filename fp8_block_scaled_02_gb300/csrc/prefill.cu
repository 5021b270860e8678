// prefill.cu -- tcgen05 block-FP8 GEMM for prefill-shaped batches (placeholder
// until the tensor-core kernel lands; the dispatcher falls back to the
// decode kernel in 32-row chunks while this reports "not supported").
#include "internal.h"

namespace fp8bs {

cudaError_t launch_prefill(const DecodeArgs &, cudaStream_t) { return cudaErrorNotSupported; }
uint32_t take_prefill_error() { return 0; }

}  // namespace fp8bs
