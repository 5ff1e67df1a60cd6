// fa_tc_common.cuh - pieces shared by the tensor-core forward and backward
// kernels: head-dimension chunking for TMA boxes and MMA descriptors, warp
// waits and register fences for Tensor Memory loads.
#pragma once

#include "sm103_ptx.cuh"

namespace fa {
namespace tc {

using namespace sm103;

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // every mbarrier wait gives up after 2 s

// The head dimension is split into 64-column chunks (128-byte rows, 128-byte
// swizzle) and one remainder chunk of 16 or 32 columns (32/64-byte swizzle),
// each its own TMA box and MMA descriptor family.
template <int D>
struct Chunks {
    static constexpr int N64 = D / 64;
    static constexpr int REM = D % 64;
    static constexpr int NCH = N64 + (REM ? 1 : 0);
    __host__ __device__ static constexpr int width(int c) { return c < N64 ? 64 : REM; }
    __host__ __device__ static constexpr int tile_off(int c, int rows) { return c * rows * 128; }
    __host__ __device__ static constexpr uint32_t swz(int c) {
        return width(c) == 64 ? SW_128B : (width(c) == 32 ? SW_64B : SW_32B);
    }
    __host__ __device__ static constexpr int row_bytes(int c) { return width(c) * 2; }
    __host__ __device__ static constexpr int map_index(int c) { return width(c) == 64 ? 0 : 1; }
};

// Lane 0 waits, the rest of the warp learns the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
    int ok = 1;
    if (lane_id() == 0) ok = mbar_wait(bar, parity, abort, status, WAIT_LIMIT_NS) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Keeps later uses of TMEM-loaded registers after tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

}  // namespace tc
}  // namespace fa
