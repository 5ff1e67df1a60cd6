// fa_tc_common.cuh - pieces shared by the tensor-core forward and backward
// kernels: head-dimension chunking for TMA boxes and MMA descriptors, warp
// waits, register fences for Tensor Memory loads, and the two product shapes
// (N = head dim, K = head dim) issued on 128-row tiles.
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
    __host__ __device__ static constexpr int col(int c) { return 64 * c; }
    // Box widths of the two TMA maps (0: map unused).
    static constexpr int MAP_W0 = N64 > 0 ? 64 : 0;
    static constexpr int MAP_W1 = (REM > 0 && !PAD) ? REM : 0;
    // One instruction covers N = d for the products whose N is the head dim.
    static constexpr bool SINGLE_N = D == 128 || PAD;
};

// The head dimension in W-column chunks (W = 16: 32-byte rows and swizzle;
// W = 32: 64-byte), the last one padded to W columns when W does not divide
// d (the TMA fills the columns past d with zeros).  A d = 80 tile of 128 rows
// takes 20 KB with W = 16 and 24 KB with W = 32 instead of 32 KB in 64-column
// chunks.  The chunks are uniform, so a product whose N is the head dim is
// still one instruction (N-direction atoms of W columns, one chunk apart); the
// k-steps over d stop at d.
template <int D, int W>
struct ChunksW {
    static_assert((W == 16 || W == 32) && D % 16 == 0, "16- or 32-column chunks, d a multiple of 16");
    static constexpr int NCH = (D + W - 1) / W;
    static constexpr int COLS = NCH * W;                      // head-dim columns stored per row
    __host__ __device__ static constexpr int width(int c) { return c < NCH - 1 ? W : D - W * (NCH - 1); }
    __host__ __device__ static constexpr int col(int c) { return W * c; }
    __host__ __device__ static constexpr int tile_off(int c, int rows) { return c * rows * W * 2; }
    __host__ __device__ static constexpr int tile_bytes(int rows) { return rows * COLS * 2; }
    __host__ __device__ static constexpr uint32_t swz(int) { return W == 16 ? SW_32B : SW_64B; }
    __host__ __device__ static constexpr int row_bytes(int) { return W * 2; }
    __host__ __device__ static constexpr int map_index(int) { return 1; }
    static constexpr int MAP_W0 = 0;
    static constexpr int MAP_W1 = W;
    static constexpr bool SINGLE_N = true;
};

// Block b of a flat grid of n_units units for each of BH heads, ordered in
// groups of grp heads: inside a group every head's unit 0 comes first, then
// every head's unit 1, and so on (grp = BH: one group, plain unit-major order).
__device__ __forceinline__ void grid_unit(int b, int BH, int n_units, int grp, int& unit, int& bh) {
    const int per = grp * n_units;
    const int g = b / per;
    const int g0 = g * grp;
    const int gsz = min(grp, BH - g0);
    const int r = b - g * per;
    unit = r / gsz;
    bh = g0 + r - unit * gsz;
}

// Heads per group of that order for a kernel whose CTAs each stream
// `bytes_per_head` of their head's data from L2.  All heads (the plain
// longest-first order) while every head's data fits `limit_mib` (160 MiB for
// the key-tile-outer backward with dQ, 128 MiB, about the L2, for the
// forward, the dK/dV-only backward and the dQ pass: the limits measured
// fastest for each); beyond that, as
// few heads as give the GPU two waves of units, within 64 MB, so the CTAs in
// flight re-read a few heads' tiles from L2 instead of DRAM.  Smaller groups
// than needed would cost more in load balance (the heaviest units of later
// groups start late) than they save.
inline int head_group(int BH, int n_units, double bytes_per_head, double limit_mib = 160.0,
                      bool only_many_heads = false) {
    constexpr double kMB = 1024.0 * 1024.0;
    if (BH * bytes_per_head <= limit_mib * kMB) return BH;
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // With fewer heads than a quarter of the SMs, the plain order already
    // keeps four or more units of every head in flight, which re-read that
    // head's tiles from L2, and grouping only delays later groups' heaviest
    // units.
    if (only_many_heads && 4 * BH < sms) return BH;
    int g = (2 * sms + n_units - 1) / n_units;
    const int cap = (int)(64.0 * kMB / bytes_per_head);
    g = g < cap ? g : cap;
    g = g < 1 ? 1 : g;
    return g < BH ? g : BH;
}

// Every lane of the warp waits on the barrier itself (the warp stays
// converged), then one vote makes the outcome uniform.  Measured against one
// lane waiting and a shuffle handing its outcome to the others: 5-14 % faster
// kernels, the hand-offs between warp roles being on their critical paths.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
    const bool ok = mbar_wait(bar, parity, abort, status, WAIT_LIMIT_NS);
    return __all_sync(0xffffffffu, ok);
}

// Keeps later uses of TMEM-loaded registers after tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// B operand of the products whose N dimension is the head dim: a [rows][d]
// tile (TMA layout, 128 rows, chunked as C) read MN-major, k-step of 16 rows
// `ks`.  `b_lo` is the low descriptor word of the tile (LBO = the chunk
// stride); the A operand is either Tensor Memory (`a_tm`) or shared memory
// (`a_desc`).
template <int D, bool A_TMEM, class C = Chunks<D>>
__device__ __forceinline__ void mma_n_is_d(uint32_t d_tmem, uint32_t a_tm, uint64_t a_desc, uint32_t b_lo, int ks,
                                           uint32_t a_mn, uint32_t acc) {
    if constexpr (C::SINGLE_N) {
        const uint64_t bdesc =
            desc_make(b_lo + ((ks * 16 * C::row_bytes(0)) >> 4), desc_hi(8 * C::row_bytes(0), C::swz(0)));
        if constexpr (A_TMEM) mma_ts(d_tmem, a_tm, bdesc, idesc_bf16(128, D, 0, 1), acc);
        else mma_ss(d_tmem, a_desc, bdesc, idesc_bf16(128, D, a_mn, 1), acc);
    } else {
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
            const uint32_t off = (C::tile_off(c, 128) + ks * 16 * C::row_bytes(c)) >> 4;
            const uint64_t bdesc = desc_make(b_lo + off, desc_hi(8 * C::row_bytes(c), C::swz(c)));
            if constexpr (A_TMEM) mma_ts(d_tmem + c * 64, a_tm, bdesc, idesc_bf16(128, C::width(c), 0, 1), acc);
            else mma_ss(d_tmem + c * 64, a_desc, bdesc, idesc_bf16(128, C::width(c), a_mn, 1), acc);
        }
    }
}

// C[128x128] = A[128 x d] B[128 x d]^T with both tiles K-major (head dim
// contiguous, chunked as C); a_lo / b_lo are the tiles' low descriptor words
// (LBO 16).
template <int D, class C = Chunks<D>>
__device__ __forceinline__ void mma_k_is_d(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc) {
    int step = 0;
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
        for (int s = 0; s < C::width(c) / 16; ++s, ++step) {
            const uint32_t off = (C::tile_off(c, 128) + s * 32) >> 4;
            const uint32_t hi = desc_hi(8 * C::row_bytes(c), C::swz(c));
            mma_ss(d_tmem, desc_make(a_lo + off, hi), desc_make(b_lo + off, hi), idesc, step > 0 ? 1u : 0u);
        }
    }
}

}  // namespace tc
}  // namespace fa
