// fa_bwd_aux.cu - the two memory-bound kernels around the backward pass.
//
// preprocess: D_i = rowsum(O * dO)_i in fp32 ("Stanford CS336 Assignment 2
//   (Systems)" handout, section 4, "backward pass with recomputation": D is
//   precomputed in global memory; Algorithm 2 step 2), and zeroing of the fp32
//   dQ accumulator that the key-tile-outer kernel adds into (skipped when
//   there is none: the deterministic backward sums dQ in its own pass).
// dq_convert: dq = dQacc * scale rounded to the storage dtype (Eq. 18's 1/sqrt(d)
//   is applied here once instead of on every partial product).
//
// Both are streaming kernels sized to the SM count: a lane group of G lanes
// reads one row (16 bytes per lane) and reduces it with shuffles, and every
// lane keeps U rows in flight.  Both are launched as programmatic dependents
// of the kernel before them: they wait for it (griddepcontrol.wait) before
// touching memory and let the next kernel launch early.

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

template <typename T, int D>
__global__ void __launch_bounds__(AUX_NT)
bwd_preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dO, float* __restrict__ Dvec,
                      float* __restrict__ dQacc, long long n_rows) {
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
                    Vec16<T>::load(o + row * D + c * VN, a);
                    Vec16<T>::load(dO + row * D + c * VN, b);
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

template <typename T>
__global__ void __launch_bounds__(AUX_NT)
dq_convert_kernel(const float* __restrict__ dQacc, T* __restrict__ dq, long long n4, float scale) {
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
            if (i >= n4) continue;
            if constexpr (sizeof(T) == 4) {
                reinterpret_cast<float4*>(dq)[i] =
                    make_float4(v[u].x * scale, v[u].y * scale, v[u].z * scale, v[u].w * scale);
            } else {
                __nv_bfloat162 lo = __floats2bfloat162_rn(v[u].x * scale, v[u].y * scale);
                __nv_bfloat162 hi = __floats2bfloat162_rn(v[u].z * scale, v[u].w * scale);
                uint2 packed;
                packed.x = *reinterpret_cast<unsigned int*>(&lo);
                packed.y = *reinterpret_cast<unsigned int*>(&hi);
                reinterpret_cast<uint2*>(dq)[i] = packed;
            }
        }
    }
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
    return launch_pdl(bwd_preprocess_kernel<T, D>, dim3(grid), dim3(AUX_NT), 0, a.stream, (const T*)a.o,
                      (const T*)a.dO, a.Dvec, a.dQacc, n_rows);
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

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a) {
    return a.dtype == DT_FP32 ? preprocess_dispatch<float>(a) : preprocess_dispatch<__nv_bfloat16>(a);
}

cudaError_t launch_dq_convert(const BwdArgs& a) {
    const long long n4 = (long long)a.B * a.H * a.S * a.d / 4;
    const long long want = (n4 + AUX_NT * 4 - 1) / (AUX_NT * 4);
    const unsigned grid = (unsigned)std::max(1LL, std::min(want, (long long)sm_count() * 8));
    if (a.dtype == DT_FP32)
        return launch_pdl(dq_convert_kernel<float>, dim3(grid), dim3(AUX_NT), 0, a.stream, (const float*)a.dQacc,
                          (float*)a.dq, n4, a.scale);
    return launch_pdl(dq_convert_kernel<__nv_bfloat16>, dim3(grid), dim3(AUX_NT), 0, a.stream,
                      (const float*)a.dQacc, (__nv_bfloat16*)a.dq, n4, a.scale);
}

}  // namespace fa
