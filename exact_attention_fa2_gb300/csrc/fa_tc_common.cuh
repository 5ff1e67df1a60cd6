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
// swizzle), each its own TMA box and MMA descriptor family.  d = 16 and 32
// are one narrower chunk (32/64-byte swizzle).  For d = 80 and 96 the
// remainder chunk is stored like a full one (a 64-column box whose columns
// past d the TMA fills with zeros): every operand then has the uniform
// 128-byte layout, so a product whose N is the head dim is ONE instruction of
// N = d instead of one per chunk (the k-steps over d still stop at d).
template <int D>
struct Chunks {
    static constexpr int N64 = D / 64;
    static constexpr int REM = D % 64;
    static constexpr int NCH = N64 + (REM ? 1 : 0);
    static constexpr bool PAD = REM != 0 && N64 > 0;
    static constexpr int COLS = PAD ? 64 * NCH : D;          // head-dim columns stored per row
    __host__ __device__ static constexpr int width(int c) { return c < N64 ? 64 : REM; }
    __host__ __device__ static constexpr int tile_off(int c, int rows) { return c * rows * 128; }
    __host__ __device__ static constexpr int tile_bytes(int rows) { return rows * COLS * 2; }
    __host__ __device__ static constexpr uint32_t swz(int c) {
        return (PAD || width(c) == 64) ? SW_128B : (width(c) == 32 ? SW_64B : SW_32B);
    }
    __host__ __device__ static constexpr int row_bytes(int c) { return PAD ? 128 : width(c) * 2; }
    __host__ __device__ static constexpr int map_index(int c) { return (PAD || width(c) == 64) ? 0 : 1; }
    // One instruction covers N = d for the products whose N is the head dim.
    static constexpr bool SINGLE_N = D == 128 || PAD;
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
