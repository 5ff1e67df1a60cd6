// fa_tmap.cu - TMA tensor-map encoding through the driver entry point (no
// link-time dependency on libcuda).

#include "fa_tmap.h"

#include <cudaTypedefs.h>
#include <mutex>

namespace fa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;

cudaError_t encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::call_once(g_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_init_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                      cudaEnableDefault, &q);
        if (g_init_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn))
            g_init_err = cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    *out = g_encode;
    return g_init_err;
}

}  // namespace

cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w,
                              int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = encoder(&enc);
    if (e != cudaSuccess) return e;
    const int inner_bytes = box_w * 2;
    CUtensorMapSwizzle swz = inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                           : inner_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                           : inner_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * d * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = encoder(&enc);
    if (e != cudaSuccess) return e;
    const int inner_bytes = box_w * 4;
    CUtensorMapSwizzle swz = inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                           : inner_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                           : inner_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)S * d * 4};
    cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace fa
