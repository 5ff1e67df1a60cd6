// fa_bwd_aux.cu - the two memory-bound kernels around the backward pass.
//
// preprocess: D_i = rowsum(O * dO)_i in fp32 ("Stanford CS336 Assignment 2
//   (Systems)" handout, section 4, "backward pass with recomputation": D is
//   precomputed in global memory; Algorithm 2 step 2), and zeroing of the fp32
//   dQ accumulator that the key-tile-outer kernel adds into.
// dq_convert: dq = dQacc * scale rounded to the storage dtype (Eq. 18's 1/sqrt(d)
//   is applied here once instead of on every partial product).
//
// Both stream rows with 16-byte vector accesses; one CTA owns 64 consecutive
// rows so that every warp reads contiguous memory.

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int PRE_ROWS = 64;
constexpr int PRE_NT = 256;

template <typename T, int D>
__global__ void __launch_bounds__(PRE_NT)
bwd_preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dO, float* __restrict__ Dvec,
                      float* __restrict__ dQacc, long long n_rows) {
    constexpr int VN = Vec16<T>::N;
    constexpr int CPR = D / VN;               // 16-byte chunks per row
    __shared__ float part[PRE_ROWS][CPR + 1];
    const long long row0 = (long long)blockIdx.x * PRE_ROWS;
    const int nr = (int)min((long long)PRE_ROWS, n_rows - row0);

    for (int idx = threadIdx.x; idx < nr * CPR; idx += PRE_NT) {
        const int r = idx / CPR, c = idx % CPR;
        const size_t off = (size_t)(row0 + r) * D + (size_t)c * VN;
        float a[VN], b[VN];
        Vec16<T>::load(o + off, a);
        Vec16<T>::load(dO + off, b);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < VN; ++i) s = fmaf(a[i], b[i], s);
        part[r][c] = s;
    }
    // Zero this CTA's rows of the dQ accumulator.
    float4* z = reinterpret_cast<float4*>(dQacc + (size_t)row0 * D);
    const int nz = nr * D / 4;
    for (int i = threadIdx.x; i < nz; i += PRE_NT) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    if (threadIdx.x < nr) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < CPR; ++c) s += part[threadIdx.x][c];
        Dvec[row0 + threadIdx.x] = s;
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
dq_convert_kernel(const float* __restrict__ dQacc, T* __restrict__ dq, long long n4, float scale) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (long long)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(dQacc)[i];
        if constexpr (sizeof(T) == 4) {
            reinterpret_cast<float4*>(dq)[i] = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * scale, v.y * scale);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * scale, v.w * scale);
            uint2 packed;
            packed.x = *reinterpret_cast<unsigned int*>(&lo);
            packed.y = *reinterpret_cast<unsigned int*>(&hi);
            reinterpret_cast<uint2*>(dq)[i] = packed;
        }
    }
}

template <typename T, int D>
cudaError_t preprocess_launch(const BwdArgs& a) {
    const long long n_rows = (long long)a.B * a.H * a.S;
    const unsigned grid = (unsigned)((n_rows + PRE_ROWS - 1) / PRE_ROWS);
    bwd_preprocess_kernel<T, D><<<grid, PRE_NT, 0, a.stream>>>((const T*)a.o, (const T*)a.dO, a.Dvec,
                                                                a.dQacc, n_rows);
    return cudaGetLastError();
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
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long want = (n4 + 255) / 256;
    const unsigned grid = (unsigned)max(1LL, min(want, (long long)sms * 8));
    if (a.dtype == DT_FP32)
        dq_convert_kernel<float><<<grid, 256, 0, a.stream>>>(a.dQacc, (float*)a.dq, n4, a.scale);
    else
        dq_convert_kernel<__nv_bfloat16><<<grid, 256, 0, a.stream>>>(a.dQacc, (__nv_bfloat16*)a.dq, n4, a.scale);
    return cudaGetLastError();
}

}  // namespace fa
