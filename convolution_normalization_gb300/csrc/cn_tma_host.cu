// Host side of TMA: encodes tiled tensor maps through the driver entry point
// (fetched once through the runtime, so the library does not link libcuda);
// and the kernels' dynamic shared-memory limits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "cn_internal.h"

namespace cn {
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_once;

void fetch_encode() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    else
        cudaGetLastError();
}
}  // namespace

bool tma_available() {
    std::call_once(g_once, fetch_encode);
    return g_encode != nullptr;
}

cudaError_t raise_dyn_smem(const void *kern, int bytes) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.maxDynamicSharedSizeBytes >= bytes) return cudaSuccess;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// fp32 tensor of rank 4 (dims innermost first, strides in bytes for dims
// 1..3), tile box `box`, zero fill outside the tensor, no swizzle.
int encode_tmap_f32_4d(CUtensorMap *map, const float *base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4]) {
    if (!tma_available()) return CN_ERR_UNSUPPORTED;
    cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gs[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(base), gd, gs,
                          bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? CN_OK : CN_ERR_CUDA;
}

// fp32 tensor of rank 5 (dims innermost first, strides in bytes for dims
// 1..4), tile box `box`, zero fill outside the tensor, no swizzle.
int encode_tmap_f32_5d(CUtensorMap *map, const float *base, const uint64_t dims[5],
                       const uint64_t strides_bytes[4], const uint32_t box[5]) {
    if (!tma_available()) return CN_ERR_UNSUPPORTED;
    cuuint64_t gd[5] = {dims[0], dims[1], dims[2], dims[3], dims[4]};
    cuuint64_t gs[4] = {strides_bytes[0], strides_bytes[1], strides_bytes[2], strides_bytes[3]};
    cuuint32_t bx[5] = {box[0], box[1], box[2], box[3], box[4]};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, const_cast<float *>(base), gd, gs,
                          bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? CN_OK : CN_ERR_CUDA;
}

}  // namespace cn
