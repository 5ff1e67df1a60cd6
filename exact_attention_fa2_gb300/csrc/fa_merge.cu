// fa_merge.cu - merge of two partial attention results over disjoint key
// sets ("[Attention] FlashAttention/Ring-Attention/...统一原理": the
// two-half merge).  For one query row with partial outputs o_a, o_b (each
// normalised over its own keys) and partial logsumexps L_a, L_b:
//   L = log(e^L_a + e^L_b),  o = e^(L_a - L) o_a + e^(L_b - L) o_b.
// A side with no admissible key carries L = -inf and weight 0; a row with
// none on either side gets o = 0, L = -inf.  Streaming kernel: one thread
// per four consecutive elements of a row, launched as a programmatic
// dependent of the kernel before it.

#include "fa_common.cuh"
#include "fa_launch.h"

#include <cmath>

namespace fa {
namespace {

constexpr int MERGE_NT = 256;

template <typename T>
__global__ void __launch_bounds__(MERGE_NT)
merge_kernel(const float* __restrict__ o_a, const float* __restrict__ l_a, const float* __restrict__ o_b,
             const float* __restrict__ l_b, T* __restrict__ o, float* __restrict__ lse, long long rows, int d4) {
    griddep_wait();
    griddep_launch();
    const long long n = rows * d4;
    const long long stride = (long long)gridDim.x * MERGE_NT;
    for (long long i = (long long)blockIdx.x * MERGE_NT + threadIdx.x; i < n; i += stride) {
        const long long r = i / d4;
        const float la = l_a[r], lb = l_b[r];
        const float m = fmaxf(la, lb);
        float wa = 0.f, wb = 0.f, L = -INFINITY;
        if (m != -INFINITY) {
            const float ea = expf(la - m), eb = expf(lb - m);
            const float sum = ea + eb;
            wa = ea / sum;
            wb = eb / sum;
            L = m + logf(sum);
        }
        const float4 a = reinterpret_cast<const float4*>(o_a)[i];
        const float4 b = reinterpret_cast<const float4*>(o_b)[i];
        const float v0 = wa * a.x + wb * b.x, v1 = wa * a.y + wb * b.y;
        const float v2 = wa * a.z + wb * b.z, v3 = wa * a.w + wb * b.w;
        if constexpr (sizeof(T) == 4) {
            reinterpret_cast<float4*>(o)[i] = make_float4(v0, v1, v2, v3);
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v0, v1);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v2, v3);
            uint2 packed;
            packed.x = *reinterpret_cast<unsigned int*>(&lo);
            packed.y = *reinterpret_cast<unsigned int*>(&hi);
            reinterpret_cast<uint2*>(o)[i] = packed;
        }
        if (i - r * d4 == 0) lse[r] = L;
    }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a) {
    const int d4 = a.d / 4;
    const long long n = a.rows * d4;
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (n + MERGE_NT - 1) / MERGE_NT;
    const unsigned grid = (unsigned)std::max(1LL, std::min(want, (long long)sms * 8));
    if (a.dtype == DT_FP32)
        return launch_pdl(merge_kernel<float>, dim3(grid), dim3(MERGE_NT), 0, a.stream, a.o_a, a.lse_a, a.o_b,
                          a.lse_b, static_cast<float*>(a.o), a.lse, a.rows, d4);
    return launch_pdl(merge_kernel<__nv_bfloat16>, dim3(grid), dim3(MERGE_NT), 0, a.stream, a.o_a, a.lse_a, a.o_b,
                      a.lse_b, static_cast<__nv_bfloat16*>(a.o), a.lse, a.rows, d4);
}

}  // namespace fa
