// noalloc.cu -- fp8bs_gemv_noalloc: the workspace GEMV (fp8bs_gemv_ws) for
// callers that cannot allocate device memory.
//
// fp8bs_gemv_ws needs a scratch buffer from its caller (the f16 copy of x and
// its per-block factors).  Some callers have no way to provide one: a plugin
// whose host framework owns every byte of device memory through its own pool
// and forbids other allocations, a real-time decode loop that cannot afford
// cudaMalloc / cudaFree (cudaFree synchronises the whole device), or a C
// caller with no place to keep a buffer alive between calls.  This entry
// point takes its scratch from a fixed array in the library's own device
// memory instead, so it allocates nothing, ever.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoallocScratchBytes until the process exits.  In host
// code its name only stands for the variable; the device address comes from
// cudaGetSymbolAddress, looked up once per device (with that device
// current) the first time the entry point runs there, and passed to the
// kernels like any workspace pointer.
#include "fp8bs.h"
#include "internal.h"

#include <mutex>

namespace fp8bs {

constexpr int64_t kNoallocScratchBytes = FP8BS_NOALLOC_SCRATCH_BYTES;

// The shared scratch.  Every call uses it from its first byte on, and each
// call writes every byte it later reads before reading it (the x
// preparation fills the f16 copy and the factors; the GEMV reads rows past m
// as zeros through its tensor map, never from memory), so nothing here
// needs to start at zero or be cleared between calls.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

namespace {

struct ScratchAddr {
    std::mutex mu;
    bool done[64] = {};
    cudaError_t err[64] = {};
    void *ptr[64] = {};
};
ScratchAddr g_addr;

// Device address of the scratch on the current device (looked up once).
cudaError_t scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_addr.mu);
    if (!g_addr.done[dev]) {
        void *p = nullptr;
        g_addr.err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        g_addr.ptr[dev] = p;
        g_addr.done[dev] = true;
    }
    *out = g_addr.ptr[dev];
    return g_addr.err[dev];
}

inline bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace fp8bs

extern "C" int fp8bs_gemv_noalloc(const void *x_bf16, int64_t m, const uint8_t *codes, const float *scales,
                                  int64_t n, int64_t k, void *y_bf16, void *stream) {
    using namespace fp8bs;
    constexpr int64_t kMaxDim = int64_t{1} << 31;
    if (m < 0 || n <= 0 || k <= 0 || m >= kMaxDim || n >= kMaxDim || k >= kMaxDim) return FP8BS_ERR_SHAPE;
    if (m == 0) return FP8BS_OK;
    if (!x_bf16 || !codes || !scales || !y_bf16) return FP8BS_ERR_NULL;
    if (!aligned_to(x_bf16, 2) || !aligned_to(y_bf16, 2) || !aligned_to(scales, 4)) return FP8BS_ERR_ALIGN;
    // only the decode path uses scratch; every other path is fp8bs_gemv's
    if (fp8bs_select_path(m, n, k, x_bf16, codes, 0) != FP8BS_PATH_DECODE)
        return fp8bs_gemv(x_bf16, m, codes, scales, n, k, y_bf16, stream);
    if (xprep_bytes(m, k) > kNoallocScratchBytes) return FP8BS_ERR_SHAPE;
    void *scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess || !scratch) return FP8BS_ERR_CUDA;
    const DecodeArgs a{x_bf16, codes, scales, nullptr, y_bf16, m, n, k, kScaleBlock, 0};
    return launch_decode_xprep(a, scratch, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FP8BS_OK
                                                                                            : FP8BS_ERR_CUDA;
}
