// fa_tmap.cu - TMA tensor-map encoding through the driver entry point (no
// link-time dependency on libcuda), with a small host-side cache: a tensor
// map only encodes an address, a shape and a box, so a cached map stays valid
// for any buffer that later occupies the same address with the same shape.

#include "fa_tmap.h"

#include <cudaTypedefs.h>
#include <cstring>
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

struct Key {
    const void* base;
    int elt_bytes, d, rows, pitch, BH, box_w, box_rows;
    bool operator==(const Key& o) const {
        return base == o.base && elt_bytes == o.elt_bytes && d == o.d && rows == o.rows && pitch == o.pitch &&
               BH == o.BH && box_w == o.box_w && box_rows == o.box_rows;
    }
};

constexpr int kCache = 64;
struct Entry {
    Key key;
    CUtensorMap map;
    bool used;
};
std::mutex g_mu;
Entry g_cache[kCache];
int g_next = 0;

// Encode a 3-D tiled map over `rows` rows of d bf16 (2-byte) or fp32 (4-byte)
// elements per head, heads `pitch` rows apart; swizzle chosen from the box's
// inner bytes.
cudaError_t encode_3d(CUtensorMap* map, const void* base, int elt_bytes, int d, int rows, int pitch, int BH,
                      int box_w, int box_rows) {
    const Key key{base, elt_bytes, d, rows, pitch, BH, box_w, box_rows};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < kCache; ++i) {
            if (g_cache[i].used && g_cache[i].key == key) {
                *map = g_cache[i].map;
                return cudaSuccess;
            }
        }
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = encoder(&enc);
    if (e != cudaSuccess) return e;
    const int inner_bytes = box_w * elt_bytes;
    CUtensorMapSwizzle swz = inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                           : inner_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                           : inner_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * elt_bytes, (cuuint64_t)pitch * d * elt_bytes};
    cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, elt_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lk(g_mu);
    g_cache[g_next] = Entry{key, *map, true};
    g_next = (g_next + 1) % kCache;
    return cudaSuccess;
}

}  // namespace

cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w,
                              int box_rows) {
    return encode_3d(map, base, 2, d, S, S, BH, box_w, box_rows);
}

cudaError_t make_tmap_bf16_3d_rows(CUtensorMap* map, const void* base, int d, int rows, int pitch, int BH,
                                   int box_w, int box_rows) {
    return encode_3d(map, base, 2, d, rows, pitch, BH, box_w, box_rows);
}

cudaError_t make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w, int box_rows) {
    return encode_3d(map, base, 4, d, S, S, BH, box_w, box_rows);
}

}  // namespace fa
