// fa_tmap.cu - TMA tensor-map encoding through the driver entry point (no
// link-time dependency on libcuda), with a small host-side cache: a tensor
// map only encodes an address, a shape, strides and a box, so a cached map
// stays valid for any buffer that later occupies the same address with the
// same shape and strides.

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
    int elt_bytes, rank;
    cuuint64_t dims[4];
    cuuint64_t strides[3];
    cuuint32_t box[4];
    bool operator==(const Key& o) const {
        if (base != o.base || elt_bytes != o.elt_bytes || rank != o.rank) return false;
        for (int i = 0; i < rank; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i] || (i > 0 && strides[i - 1] != o.strides[i - 1]))
                return false;
        return true;
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

// Encode a tiled map of rank 3 or 4 over bf16 (2-byte) or fp32 (4-byte)
// elements: dims innermost first, strides in bytes for dims 1..rank-1, box
// {box_w, box_rows, 1, ...}; swizzle chosen from the box's inner bytes.
cudaError_t encode(CUtensorMap* map, const Key& key) {
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
    const int inner_bytes = (int)key.box[0] * key.elt_bytes;
    CUtensorMapSwizzle swz = inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                           : inner_bytes == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                           : inner_bytes == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
    for (int i = 0; i < key.rank; ++i) {
        dims[i] = key.dims[i];
        box[i] = key.box[i];
        if (i > 0) strides[i - 1] = key.strides[i - 1];
    }
    CUresult r = enc(map, key.elt_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                     key.rank, const_cast<void*>(key.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lk(g_mu);
    g_cache[g_next] = Entry{key, *map, true};
    g_next = (g_next + 1) % kCache;
    return cudaSuccess;
}

Key key_3d(const void* base, int elt_bytes, int d, int rows, int pitch, int BH, int box_w, int box_rows) {
    Key k{};
    k.base = base;
    k.elt_bytes = elt_bytes;
    k.rank = 3;
    k.dims[0] = (cuuint64_t)d;
    k.dims[1] = (cuuint64_t)rows;
    k.dims[2] = (cuuint64_t)BH;
    k.strides[0] = (cuuint64_t)d * elt_bytes;
    k.strides[1] = (cuuint64_t)pitch * d * elt_bytes;
    k.box[0] = (cuuint32_t)box_w;
    k.box[1] = (cuuint32_t)box_rows;
    k.box[2] = 1;
    return k;
}

}  // namespace

cudaError_t make_tmap_bf16_4d(CUtensorMap* map, const void* base, int d, int rows, int H, int B, View v,
                              int box_w, int box_rows) {
    // A dimension of extent 1 is never stepped: give it a stride the encoder
    // accepts whatever the caller's value was.
    const long long s = v.s;
    const long long h = H > 1 ? v.h : s * rows;
    const long long b = B > 1 ? v.b : h * H;
    Key k{};
    k.base = base;
    k.elt_bytes = 2;
    k.rank = 4;
    k.dims[0] = (cuuint64_t)d;
    k.dims[1] = (cuuint64_t)rows;
    k.dims[2] = (cuuint64_t)H;
    k.dims[3] = (cuuint64_t)B;
    k.strides[0] = (cuuint64_t)s * 2;
    k.strides[1] = (cuuint64_t)h * 2;
    k.strides[2] = (cuuint64_t)b * 2;
    k.box[0] = (cuuint32_t)box_w;
    k.box[1] = (cuuint32_t)box_rows;
    k.box[2] = 1;
    k.box[3] = 1;
    return encode(map, k);
}

cudaError_t make_tmap_bf16_view(CUtensorMap* map, bool* rank3, const void* base, int d, int rows, int H, int B,
                                View v, int box_w, int box_rows) {
    // Batch and head merge into one dimension of B*H indices when stepping
    // the batch index is H steps of the head index.
    const long long h = H > 1 ? v.h : v.s * rows;
    if (B == 1 || v.b == h * H) {
        Key k{};
        k.base = base;
        k.elt_bytes = 2;
        k.rank = 3;
        k.dims[0] = (cuuint64_t)d;
        k.dims[1] = (cuuint64_t)rows;
        k.dims[2] = (cuuint64_t)B * H;
        k.strides[0] = (cuuint64_t)v.s * 2;
        k.strides[1] = (cuuint64_t)h * 2;
        k.box[0] = (cuuint32_t)box_w;
        k.box[1] = (cuuint32_t)box_rows;
        k.box[2] = 1;
        *rank3 = true;
        return encode(map, k);
    }
    *rank3 = false;
    return make_tmap_bf16_4d(map, base, d, rows, H, B, v, box_w, box_rows);
}

cudaError_t make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w, int box_rows) {
    return encode(map, key_3d(base, 4, d, S, S, BH, box_w, box_rows));
}

}  // namespace fa
