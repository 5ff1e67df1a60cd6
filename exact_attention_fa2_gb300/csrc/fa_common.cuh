// fa_common.cuh - small helpers shared by the attention kernels (device side).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#ifndef FA_LOG2E
#define FA_LOG2E 1.4426950408889634f
#define FA_LN2 0.6931471805599453f
#endif

// Status codes a kernel may leave in the device status word.
#define FA_DEV_STATUS_TIMEOUT 1u
#define FA_DEV_STATUS_BOUNDS 2u

namespace fa {

struct bf16x8 { __nv_bfloat162 h[4]; };

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Round an fp32 value to the storage precision of T and back (identity for fp32).
template <typename T> __device__ __forceinline__ float round_to(float x) {
    return to_f32(from_f32<T>(x));
}

// Load 16 bytes of T from global memory and widen to fp32.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float* p, float* out) {
        float4 v = *reinterpret_cast<const float4*>(p);
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
    __device__ __forceinline__ static void store(float* p, const float* in) {
        *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float* out) {
        uint4 raw = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x; out[2 * i + 1] = f.y;
        }
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, const float* in) {
        uint4 raw;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = raw;
    }
};

// Programmatic dependent launch: wait until the previous kernel on the stream
// has completed and its writes are visible (returns at once when the kernel
// was launched without the attribute); let the next kernel start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void set_status(unsigned int* status, unsigned int code) {
    if (status) atomicOr(status, code);
}

}  // namespace fa
