// fa_bwd_aux.cu - the two memory-bound kernels around the backward pass.
//
// preprocess: D_i = rowsum(O * dO)_i in fp32 ("Stanford CS336 Assignment 2
//   (Systems)" handout, section 4, "backward pass with recomputation": D is
//   precomputed in global memory; Algorithm 2, before its loops), and zeroing of the fp32
//   dQ accumulator that the key-tile-outer kernel adds into (skipped when
//   there is none: the deterministic backward sums dQ in its own pass).
// dq_convert: dq = dQacc * scale rounded to the storage dtype (Eq. 18's 1/sqrt(d)
//   is applied here once instead of on every partial product).
//
// Both are streaming kernels sized to the SM count: a lane group of G lanes
// reads one row (16 bytes per lane; the preprocess reduces it with shuffles),
// and every lane keeps U rows in flight.  O, dO and dq are [B, H, S, d] views
// with any strides (16-byte aligned rows; contiguous ones skip the index
// arithmetic); D and dQacc are contiguous.  Both are launched as programmatic
// dependents of the kernel before them: they wait for it (griddepcontrol.wait)
// before touching memory and let the next kernel launch early.

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int AUX_NT = 256;

template <int CPR>
struct RowGroup {
    // Lanes per row: the 16-byte chunks of a row, rounded up to a power of two.
    static constexpr int G = CPR <= 2 ? 2 : CPR <= 4 ? 4 : CPR <= 8 ? 8 : CPR <= 16 ? 16 : 32;
    static constexpr int RPW = 32 / G;      // rows per warp and step
    static_assert(CPR <= 32, "row wider than a warp");
};

// Element offset of query row `row` (flat over B*H*S, below 2^31) in a view.
__device__ __forceinline__ long long row_off(const View& v, long long row, int S, int H) {
    const unsigned r32 = (unsigned)row;
    const unsigned bh = r32 / (unsigned)S;
    const unsigned b = bh / (unsigned)H;
    return v.off((int)b, (int)(bh - b * H), (long long)(r32 - bh * (unsigned)S));
}

template <typename T, int D>
__global__ void __launch_bounds__(AUX_NT)
bwd_preprocess_kernel(const T* __restrict__ o, View vo, const T* __restrict__ dO, View vdo,
                      float* __restrict__ Dvec, float* __restrict__ dQacc, long long n_rows, int S, int H,
                      bool contig) {
    constexpr int VN = Vec16<T>::N;           // elements per 16-byte chunk
    constexpr int CPR = D / VN;               // chunks per row
    using RG = RowGroup<CPR>;
    constexpr int U = 2;                      // row steps in flight per warp
    constexpr int Z4 = D / 4;                 // float4s of one dQ accumulator row
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int sub = lane / RG::G;             // row of this lane within a warp step
    const int c = lane % RG::G;               // chunk of this lane within the row
    const long long warp_id = ((long long)blockIdx.x * AUX_NT + threadIdx.x) >> 5;
    const long long n_warps = ((long long)gridDim.x * AUX_NT) >> 5;
    constexpr int ROWS_PER_ITER = RG::RPW * U;
    float4* z = reinterpret_cast<float4*>(dQacc);
    for (long long r0 = warp_id * ROWS_PER_ITER; r0 < n_rows; r0 += n_warps * ROWS_PER_ITER) {
        float part[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long row = r0 + u * RG::RPW + sub;
            part[u] = 0.f;
            if (row < n_rows) {
                if (c < CPR) {
                    float a[VN], b[VN];
                    const long long oo = contig ? row * D : row_off(vo, row, S, H);
                    const long long od = contig ? row * D : row_off(vdo, row, S, H);
                    Vec16<T>::load(o + oo + c * VN, a);
                    Vec16<T>::load(dO + od + c * VN, b);
#pragma unroll
                    for (int i = 0; i < VN; ++i) part[u] = fmaf(a[i], b[i], part[u]);
                }
                // This row of the dQ accumulator starts at zero (no accumulator
                // in the deterministic backward).
                if (z != nullptr) {
#pragma unroll
                    for (int k = c; k < Z4; k += RG::G) z[row * Z4 + k] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int off = RG::G / 2; off > 0; off >>= 1) part[u] += __shfl_xor_sync(0xffffffffu, part[u], off);
            const long long row = r0 + u * RG::RPW + sub;
            if (c == 0 && row < n_rows) Dvec[row] = part[u];
        }
    }
}

// Four fp32 values times scale stored as T (one 16-byte or 8-byte store).
template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v, float scale) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * scale, v.y * scale);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * scale, v.w * scale);
        uint2 packed;
        packed.x = *reinterpret_cast<unsigned int*>(&lo);
        packed.y = *reinterpret_cast<unsigned int*>(&hi);
        *reinterpret_cast<uint2*>(dst) = packed;
    }
}

// dq = dQacc * scale for a contiguous dq: grid-stride over float4s, U loads
// in flight per thread.
template <typename T>
__global__ void __launch_bounds__(AUX_NT)
dq_convert_flat_kernel(const float* __restrict__ dQacc, T* __restrict__ dq, long long n4, float scale) {
    constexpr int U = 4;
    griddep_wait();
    griddep_launch();
    const long long stride = (long long)gridDim.x * AUX_NT;
    for (long long i0 = (long long)blockIdx.x * AUX_NT + threadIdx.x; i0 < n4; i0 += stride * U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long i = i0 + u * stride;
            if (i < n4) v[u] = __ldcs(reinterpret_cast<const float4*>(dQacc) + i);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long i = i0 + u * stride;
            if (i < n4) store4(dq + 4 * i, v[u], scale);
        }
    }
}

// dq = dQacc * scale for a strided dq: lane groups of G lanes per row (one
// float4 of the contiguous accumulator per lane), U rows in flight per lane.
template <typename T, int D>
__global__ void __launch_bounds__(AUX_NT)
dq_convert_kernel(const float* __restrict__ dQacc, T* __restrict__ dq, View vdq, long long n_rows, int S, int H,
                  float scale) {
    constexpr int CPR = D / 4;                // float4s per accumulator row
    using RG = RowGroup<CPR>;
    constexpr int U = 4;
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int sub = lane / RG::G;
    const int c = lane % RG::G;
    const long long warp_id = ((long long)blockIdx.x * AUX_NT + threadIdx.x) >> 5;
    const long long n_warps = ((long long)gridDim.x * AUX_NT) >> 5;
    constexpr int ROWS_PER_ITER = RG::RPW * U;
    for (long long r0 = warp_id * ROWS_PER_ITER; r0 < n_rows; r0 += n_warps * ROWS_PER_ITER) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long row = r0 + u * RG::RPW + sub;
            if (row < n_rows && c < CPR) v[u] = __ldcs(reinterpret_cast<const float4*>(dQacc + row * D) + c);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long row = r0 + u * RG::RPW + sub;
            if (row >= n_rows || c >= CPR) continue;
            store4(dq + row_off(vdq, row, S, H) + 4 * c, v[u], scale);
        }
    }
}

// dK = dV = 0 on key rows [row0, row0 + rows) of every head (keys no query
// attends): 16-byte zero stores over both views.
__global__ void __launch_bounds__(AUX_NT)
zero_rows_kernel(char* dk, View vdk, char* dv, View vdv, long long n_rows, int row0, int rows, int H, int units,
                 int elt) {
    griddep_wait();
    griddep_launch();
    const long long n = n_rows * units;
    for (long long i = (long long)blockIdx.x * AUX_NT + threadIdx.x; i < n; i += (long long)gridDim.x * AUX_NT) {
        const long long row = i / units;
        const int u = (int)(i - row * units);
        const int bh = (int)(row / rows);
        const int r = row0 + (int)(row - (long long)bh * rows);
        const int b = bh / H, h = bh - b * H;
        *reinterpret_cast<uint4*>(dk + vdk.off(b, h, r) * elt + 16 * u) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dv + vdv.off(b, h, r) * elt + 16 * u) = make_uint4(0, 0, 0, 0);
    }
}

bool is_contig(const View& v, const BwdArgs& a) {
    const View c = contiguous_view(a.H, a.S, a.d);
    return (a.B == 1 || v.b == c.b) && (a.H == 1 || v.h == c.h) && v.s == c.s;
}

int sm_count() {
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <typename T, int D>
cudaError_t preprocess_launch(const BwdArgs& a) {
    constexpr int CPR = D / Vec16<T>::N;
    const long long n_rows = (long long)a.B * a.H * a.S;
    const long long rows_per_cta = (AUX_NT / 32) * RowGroup<CPR>::RPW * 2;
    const long long want = (n_rows + rows_per_cta - 1) / rows_per_cta;
    const unsigned grid = (unsigned)std::max(1LL, std::min(want, (long long)sm_count() * 8));
    return launch_pdl(bwd_preprocess_kernel<T, D>, dim3(grid), dim3(AUX_NT), 0, a.stream, (const T*)a.o, a.vo,
                      (const T*)a.dO, a.vdo, a.Dvec, a.dQacc, n_rows, a.S, a.H,
                      is_contig(a.vo, a) && is_contig(a.vdo, a));
}

template <typename T>
cudaError_t preprocess_dispatch(const BwdArgs& a) {
    switch (a.d) {
        case 16: return preprocess_launch<T, 16>(a);
        case 32: return preprocess_launch<T, 32>(a);
        case 64: return preprocess_launch<T, 64>(a);
        case 80: return preprocess_launch<T, 80>(a);
        case 96: return preprocess_launch<T, 96>(a);
        case 128: return preprocess_launch<T, 128>(a);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int D>
cudaError_t convert_launch(const BwdArgs& a) {
    constexpr int CPR = D / 4;
    const long long n_rows = (long long)a.B * a.H * a.S;
    const long long rows_per_cta = (AUX_NT / 32) * RowGroup<CPR>::RPW * 4;
    const long long want = (n_rows + rows_per_cta - 1) / rows_per_cta;
    const unsigned grid = (unsigned)std::max(1LL, std::min(want, (long long)sm_count() * 8));
    return launch_pdl(dq_convert_kernel<T, D>, dim3(grid), dim3(AUX_NT), 0, a.stream, (const float*)a.dQacc,
                      (T*)a.dq, a.vdq, n_rows, a.S, a.H, a.scale);
}

template <typename T>
cudaError_t convert_dispatch(const BwdArgs& a) {
    if (is_contig(a.vdq, a)) {
        const long long n4 = (long long)a.B * a.H * a.S * a.d / 4;
        const long long want = (n4 + AUX_NT * 4 - 1) / (AUX_NT * 4);
        const unsigned grid = (unsigned)std::max(1LL, std::min(want, (long long)sm_count() * 8));
        return launch_pdl(dq_convert_flat_kernel<T>, dim3(grid), dim3(AUX_NT), 0, a.stream, (const float*)a.dQacc,
                          (T*)a.dq, n4, a.scale);
    }
    switch (a.d) {
        case 16: return convert_launch<T, 16>(a);
        case 32: return convert_launch<T, 32>(a);
        case 64: return convert_launch<T, 64>(a);
        case 80: return convert_launch<T, 80>(a);
        case 96: return convert_launch<T, 96>(a);
        case 128: return convert_launch<T, 128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a) {
    return a.dtype == DT_FP32 ? preprocess_dispatch<float>(a) : preprocess_dispatch<__nv_bfloat16>(a);
}

cudaError_t launch_zero_rows(const BwdArgs& a, int row0) {
    if (row0 >= a.Sk) return cudaSuccess;
    const int elt = a.dtype == DT_FP32 ? 4 : 2;
    const int units = a.d * elt / 16;
    const int rows = a.Sk - row0;
    const long long n_rows = (long long)a.B * a.H * rows;
    const long long want = (n_rows * units + AUX_NT - 1) / AUX_NT;
    const unsigned grid = (unsigned)std::max(1LL, std::min(want, (long long)sm_count() * 8));
    return launch_pdl(zero_rows_kernel, dim3(grid), dim3(AUX_NT), 0, a.stream, (char*)a.dk, a.vdk, (char*)a.dv, a.vdv,
                      n_rows, row0, rows, a.H, units, elt);
}

cudaError_t launch_dq_convert(const BwdArgs& a) {
    return a.dtype == DT_FP32 ? convert_dispatch<float>(a) : convert_dispatch<__nv_bfloat16>(a);
}

}  // namespace fa
