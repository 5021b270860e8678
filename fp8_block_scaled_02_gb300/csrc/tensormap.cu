// tensormap.cu -- TMA descriptor encoding and device queries.
//
// cuTensorMapEncodeTiled is a driver API entry point; it is fetched once
// through the runtime (cudaGetDriverEntryPointByVersion) so the library
// needs no link against libcuda.  Encoding is pure host work (no device
// call, no synchronisation), so it is safe inside stream capture.
#include "internal.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

namespace fp8bs {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void resolve_encode() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices] = {};

}  // namespace

bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, resolve_encode);
    if (!g_encode) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, const uint64_t (&dims)[3],
                          const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, resolve_encode);
    if (!g_encode) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = g_encode(map, dtype, 3, const_cast<void *>(base), d, st, bx, elem_strides,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int pick_split(ClusterFit &fit, const void *kern, int threads, int smem, int tiles, int max_split) {
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || dev >= 64) return 1;
    if (max_split > 16) max_split = 16;
    for (int s = max_split; s > 1; --s) {
        int fits;
        {
            std::lock_guard<std::mutex> lock(mu);
            fits = fit.max_clusters[dev][s];
            if (fits == 0) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(1, static_cast<unsigned>(s), 1);
                cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
                cfg.dynamicSmemBytes = static_cast<size_t>(smem);
                cudaLaunchAttribute attr;
                attr.id = cudaLaunchAttributeClusterDimension;
                attr.val.clusterDim.x = 1;
                attr.val.clusterDim.y = static_cast<unsigned>(s);
                attr.val.clusterDim.z = 1;
                cfg.attrs = &attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                    (void)cudaGetLastError();
                    n = -1;
                }
                fit.max_clusters[dev][s] = fits = n;
            }
        }
        if (fits >= tiles) return s;
    }
    return 1;
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 1;
        g_sm_count[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

}  // namespace fp8bs
