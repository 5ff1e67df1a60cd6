// fa_fwd_tc.cu - bf16 FlashAttention-2 forward on the sm_103a tensor cores.
//
// Computes O = softmax(Q K^T * scale) V and L = logsumexp ("Stanford CS336
// Assignment 2 (Systems)" handout, section 4: Eq. 4-6, Eq. 12, Algorithm 1)
// with tcgen05.mma into Tensor Memory.
//
// One CTA owns one 128-row query tile of one (batch, head) and streams the
// 128-key K/V tiles it needs through a TMA/mbarrier ring.  Warp roles:
//   warps 0-3  softmax on score columns 0-63 (one query row per thread),
//   warps 4-7  softmax on score columns 64-127 (same rows),
//   warp  8    TMA producer (Q once, then the K and V rings),
//   warp  9    Tensor Memory allocation and the single-thread MMA issuer.
// Tensor Memory: two score buffers S_0, S_1 (columns [0,128) and [128,256))
// and the output accumulator O (columns [256, 256+d)).  The MMA issuer
// computes S_{j+1} = Q K_{j+1}^T into the free buffer while the softmax works
// on S_j, so the tensor cores and the softmax warps run concurrently.  P_j
// (bf16) overwrites the first 64 columns of its score buffer and the PV
// product reads it from there.
//
// Online softmax (Algorithm 1 lines 10-13) in base 2: scores are scaled by
// c = |scale| * log2(e); the two halves of a row exchange their maxima through
// shared memory; a warp rescales its rows of O only when some row's max grew.
// The running max is always the exact max so far, which keeps the dominant
// probability of a sharp row at exactly 1.0 before the bf16 rounding of P
// (letting the max lag by a few binades doubles the bf16 error of O for sharp
// softmax rows).  Fully masked causal tiles are never loaded or multiplied.

#include "fa_common.cuh"
#include "fa_launch.h"
#include "fa_tmap.h"
#include "sm103_ptx.cuh"
#include "fa_tc_common.cuh"

#include <cstring>

namespace fa {
namespace {

using namespace sm103;
using namespace tc;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int NTHREADS = 320;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 256;
constexpr int SMEM_FLOOR = 120 * 1024;   // keeps one CTA per SM (it owns all of TMEM)

template <int D>
struct FwdCfg {
    static constexpr int TILE = BM * D * 2;
    static constexpr int NS_RAW = (222 * 1024 - TILE) / (2 * TILE);
    static constexpr int NS = NS_RAW > 4 ? 4 : NS_RAW;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE;
    static constexpr int V_OFF = K_OFF + NS * TILE;
    static constexpr int X_OFF = V_OFF + NS * TILE;     // (value, tag) slots: max [2 parity][2 half][128], l [2 half][128]
    static constexpr int BAR_OFF = X_OFF + 6 * BM * 8;
    // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full, o_done, drain
    static constexpr int NBARS = 1 + 4 * NS + 5;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int DYN_SMEM = (BYTES + 1024) > SMEM_FLOOR ? (BYTES + 1024) : SMEM_FLOOR;
    static_assert(NS >= 2, "K/V ring needs two stages");
    static_assert(DYN_SMEM <= 227 * 1024, "shared memory budget");
};

struct FwdParams {
    CUtensorMap tq[2];
    CUtensorMap tk[2];
    CUtensorMap tv[2];
    __nv_bfloat16* o;
    float* lse;
    unsigned int* status;
    int S;
    int n_qt;
    int n_kv;
    int causal;
    float c;          // |scale| * log2(e), at least 1e-30
    uint32_t neg_a;   // 1 when scale < 0: the S product negates Q
};

// Exchange one float with the partner thread that owns the other column half
// of the same query row: publish (value, tag) with one 64-bit store, then poll
// the partner's slot until it carries the same tag.  The poll is bounded: on
// timeout (or when another role of the CTA gave up) it reports through the
// status word / abort flag and returns the thread's own value.
__device__ __forceinline__ float exchange_with_partner(uint32_t mine, uint32_t theirs, float val, int tag,
                                                       volatile int* abort, unsigned int* status, bool& ok) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" :: "r"(mine), "f"(val), "f"(__int_as_float(tag)) : "memory");
    uint64_t t0 = 0;
    for (uint32_t n = 0;; ++n) {
        float pv, pt;
        asm volatile("ld.volatile.shared.v2.f32 {%0, %1}, [%2];" : "=f"(pv), "=f"(pt) : "r"(theirs) : "memory");
        if (__float_as_int(pt) == tag) return pv;
        if ((n & 255) == 255) {
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            if (*abort || now - t0 > WAIT_LIMIT_NS) {
                if (!*abort) set_status(status, FA_DEV_STATUS_TIMEOUT);
                *abort = 1;
                ok = false;
                return val;
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_tc_kernel(const __grid_constant__ FwdParams p) {
    using C = Chunks<D>;
    using G = FwdCfg<D>;
    constexpr int NS = G::NS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + G::BAR_OFF;
    const uint32_t q_full = bar0;
    auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto k_empty = [&](int s) { return bar0 + 8u * (1 + NS + s); };
    auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * NS + s); };
    auto v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * NS + s); };
    auto s_full = [&](int b) { return bar0 + 8u * (1 + 4 * NS + b); };
    const uint32_t p_full = bar0 + 8u * (3 + 4 * NS);
    const uint32_t o_done = bar0 + 8u * (4 + 4 * NS);
    const uint32_t drain = bar0 + 8u * (5 + 4 * NS);
    const uint32_t xmax = sb + G::X_OFF;                               // float2 slots [2][2][128]
    const uint32_t xl = xmax + 4 * BM * 8;                              // float2 slots [2][128]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // One flat grid ordered tile-rank-major: every head's longest causal row
    // block is dispatched before any head's next one (longest job first).
    const int BH = (int)(gridDim.x / (unsigned)p.n_qt);
    const int rank = (int)blockIdx.x / BH;
    const int bh = (int)blockIdx.x - rank * BH;
    const int qt = p.causal ? (p.n_qt - 1 - rank) : rank;
    const int S = p.S;
    const int q0 = qt * BM;
    const int jmax = p.causal ? min(qt, p.n_kv - 1) : p.n_kv - 1;   // key tiles 0..jmax

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        mbar_init(s_full(0), 1);
        mbar_init(s_full(1), 1);
        mbar_init(p_full, 2 * BM);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort = 0;
    }
    for (int i = threadIdx.x; i < 6 * BM; i += NTHREADS)            // no slot carries a valid tag yet
        reinterpret_cast<int2*>(smem + G::X_OFF)[i] = make_int2(0, -1);
    if (threadIdx.x == 0) {
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == TMA_WARP) {
        // ------------------------------------------------------------ producer
        int issued_k = 0, issued_v = 0;
        if (lane == 0) {
            for (int i = 0; i < 2; ++i) {
                prefetch_tmap(&p.tq[i]);
                prefetch_tmap(&p.tk[i]);
                prefetch_tmap(&p.tv[i]);
            }
            mbar_arrive_expect_tx(q_full, G::TILE);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(sb + G::Q_OFF + C::tile_off(c, BM), &p.tq[C::map_index(c)], c * 64, q0, bh, q_full);
            for (int j = 0; j <= jmax; ++j) {
                const int st = j % NS;
                const uint32_t ph = (j / NS) & 1;
                if (!mbar_wait(k_empty(st), ph ^ 1, abort, p.status, WAIT_LIMIT_NS)) break;
                mbar_arrive_expect_tx(k_full(st), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sb + G::K_OFF + st * G::TILE + C::tile_off(c, BN), &p.tk[C::map_index(c)],
                                c * 64, j * BN, bh, k_full(st));
                issued_k = j + 1;
                if (!mbar_wait(v_empty(st), ph ^ 1, abort, p.status, WAIT_LIMIT_NS)) break;
                mbar_arrive_expect_tx(v_full(st), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sb + G::V_OFF + st * G::TILE + C::tile_off(c, BN), &p.tv[C::map_index(c)],
                                c * 64, j * BN, bh, v_full(st));
                issued_v = j + 1;
            }
            if (*abort) {
                // Let the copies already in flight land before the CTA exits.
                volatile int no_abort = 0;
                mbar_wait(q_full, 0, &no_abort, p.status, WAIT_LIMIT_NS);
                for (int j = max(0, issued_k - NS); j < issued_k; ++j)
                    mbar_wait(k_full(j % NS), (j / NS) & 1, &no_abort, p.status, WAIT_LIMIT_NS);
                for (int j = max(0, issued_v - NS); j < issued_v; ++j)
                    mbar_wait(v_full(j % NS), (j / NS) & 1, &no_abort, p.status, WAIT_LIMIT_NS);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0) | (p.neg_a << 13);
        // Low descriptor words of the operand buffers; k-steps add constants.
        const uint32_t q_lo = desc_lo(sb + G::Q_OFF, 16);
        const uint32_t k_lo0 = desc_lo(sb + G::K_OFF, 16);
        const uint32_t v_lo0 = desc_lo(sb + G::V_OFF, BN * 128);
        // S_j = Q K_j^T into score buffer j % 2.
        auto issue_s = [&](int j) {
            const int st = j % NS;
            const uint32_t d_s = tmem + (uint32_t)(j & 1) * 128;
            const uint32_t klo = k_lo0 + (uint32_t)st * (G::TILE >> 4);
            int step = 0;
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
                for (int s = 0; s < C::width(c) / 16; ++s, ++step) {
                    const uint32_t off = (C::tile_off(c, BM) + s * 32) >> 4;
                    const uint32_t hi = desc_hi(8 * C::row_bytes(c), C::swz(c));
                    mma_ss(d_s, desc_make(q_lo + off, hi), desc_make(klo + off, hi), idesc_s, step > 0 ? 1u : 0u);
                }
            }
            mma_commit(s_full(j & 1));
            mma_commit(k_empty(st));
        };
        // O += P_j V_j: A = P_j from Tensor Memory, B = V_j (MN-major, keys along K).
        auto issue_pv = [&](int j) {
            const int st = j % NS;
            const uint32_t vlo = v_lo0 + (uint32_t)st * (G::TILE >> 4);
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks) {
                const uint32_t a_tm = tmem + (uint32_t)(j & 1) * 128 + ks * 8;
                const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
                if constexpr (D == 128) {
                    mma_ts(tmem + TM_O, a_tm, desc_make(vlo + ks * 128, desc_hi(1024, SW_128B)),
                           idesc_bf16(BM, 128, 0, 1), acc);
                } else {
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c) {
                        const uint32_t off = (C::tile_off(c, BN) + ks * 16 * C::row_bytes(c)) >> 4;
                        mma_ts(tmem + TM_O + c * 64, a_tm, desc_make(vlo + off, desc_hi(8 * C::row_bytes(c), C::swz(c))),
                               idesc_bf16(BM, C::width(c), 0, 1), acc);
                    }
                }
            }
            mma_commit(o_done);
            mma_commit(v_empty(st));
        };
        bool ok = warp_wait(q_full, 0, abort, p.status);
        if (ok) ok = warp_wait(k_full(0), 0, abort, p.status);
        if (ok) {
            tc_fence_after();
            if (lane == 0) issue_s(0);
            __syncwarp();
        }
        for (int j = 0; j <= jmax && ok; ++j) {
            if (j + 1 <= jmax) {
                const int st = (j + 1) % NS;
                if (!(ok = warp_wait(k_full(st), ((j + 1) / NS) & 1, abort, p.status))) break;
                tc_fence_after();
                if (lane == 0) issue_s(j + 1);
                __syncwarp();
            }
            if (!(ok = warp_wait(v_full(j % NS), (j / NS) & 1, abort, p.status))) break;
            if (!(ok = warp_wait(p_full, j & 1, abort, p.status))) break;
            tc_fence_after();
            if (lane == 0) issue_pv(j);
            __syncwarp();
        }
        if (*abort) {
            // Wait until every MMA issued so far has finished before TMEM is freed.
            if (lane == 0) {
                volatile int no_abort = 0;
                mma_commit(drain);
                mbar_wait(drain, 0, &no_abort, p.status, WAIT_LIMIT_NS);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int h = warp >> 2;                 // column half of every score tile
        const int wq = warp & 3;                 // lane quarter of Tensor Memory
        const int row_local = wq * 32 + lane;
        const int row = q0 + row_local;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float c = p.c;
        const int key_lim = p.causal ? min(row, S - 1) : S - 1;
        float m_use = -INFINITY;
        float l_part = 0.f;                       // this half's share of the row sum
        bool ok = true;
        for (int j = 0; j <= jmax; ++j) {
            const int b = j & 1;
            if (!(ok = warp_wait(s_full(b), (j >> 1) & 1, abort, p.status))) break;
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + (uint32_t)b * 128;
            uint32_t r[64];
            tmem_ld32(tS + 64 * h, r);
            tmem_ld32(tS + 64 * h + 32, r + 32);
            tmem_wait_ld();
            reg_fence<64>(r);
            // Only the diagonal tile of a causal row block and a ragged last
            // tile need the per-element mask; masked scores become -inf.
            const int kbase = j * BN + 64 * h;
            if ((p.causal && j == jmax) || (j * BN + BN > S)) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (kbase + i > key_lim) r[i] = 0xff800000u;
            }
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 64; i += 8) {
                mx0 = max3f(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                mx1 = max3f(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                mx2 = max3f(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                mx3 = max3f(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
            }
            const float pmax = max3f(mx0, mx1, fmaxf(mx2, mx3));
            const uint32_t xm = xmax + (uint32_t)(b * 2 * BM) * 8;
            const float omax = exchange_with_partner(xm + (uint32_t)(h * BM + row_local) * 8,
                                                     xm + (uint32_t)((1 - h) * BM + row_local) * 8, pmax, j, abort,
                                                     p.status, ok);
            if (!ok) break;
            const float mx = fmaxf(pmax, omax);
            const float m_new = fmaxf(m_use, mx * c);
            const float alpha = (j == 0 || m_new == m_use) ? 1.f : ex2(m_use - m_new);
            m_use = m_new;
            const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
            const uint64_t c2 = f2pack(c, c);
            const uint64_t n2 = f2pack(neg, neg);
            // P = exp2(S*c - m) rounded to bf16 into columns [32h, 32h+32) of
            // the score buffer (both halves have read their scores: the
            // exchange above ordered it), and this half's fp32 row sum.
            uint64_t sum_a = f2pack(0.f, 0.f), sum_b = f2pack(0.f, 0.f);
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float x0, x1;
                f2unpack(fma2(f2pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, n2), x0, x1);
                const float p0 = ex2(x0);
                const float p1 = ex2(x1);
                if (i & 1) sum_b = add2(sum_b, f2pack(p0, p1));
                else sum_a = add2(sum_a, f2pack(p0, p1));
                pk[i] = pack_bf16(p0, p1);
            }
            tmem_st32(tS + 32 * h, pk);
            float s0, s1, s2, s3;
            f2unpack(sum_a, s0, s1);
            f2unpack(sum_b, s2, s3);
            l_part = l_part * alpha + ((s0 + s1) + (s2 + s3));
            // Rescale this half's O columns once the previous PV product has
            // landed (it was issued when the previous P was published).
            if (j > 0) {
                if (!(ok = warp_wait(o_done, (j - 1) & 1, abort, p.status))) break;
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    tc_fence_after();
                    const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
                    for (int u = h; u < D / 16; u += 2) {
                        uint32_t o[16];
                        tmem_ld16(tmem + lane_off + TM_O + 16 * u, o);
                        tmem_wait_ld();
                        reg_fence<16>(o);
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            float lo, hi;
                            f2unpack(mul2(f2pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), lo, hi);
                            o[i] = __float_as_uint(lo);
                            o[i + 1] = __float_as_uint(hi);
                        }
                        tmem_st16(tmem + lane_off + TM_O + 16 * u, o);
                    }
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // Epilogue (Algorithm 1 lines 15-18): O / l and L = (m + log2 l) ln 2.
        if (ok) {
            const float l_other = exchange_with_partner(xl + (uint32_t)(h * BM + row_local) * 8,
                                                        xl + (uint32_t)((1 - h) * BM + row_local) * 8, l_part, 0,
                                                        abort, p.status, ok);
            const float l_sum = l_part + l_other;
            if (ok && warp_wait(o_done, jmax & 1, abort, p.status)) {
                tc_fence_after();
                const float inv = 1.f / l_sum;
                __nv_bfloat16* orow = p.o + ((size_t)bh * S + row) * D;
#pragma unroll
                for (int u = h; u < D / 16; u += 2) {
                    uint32_t o[16];
                    tmem_ld16(tmem + lane_off + TM_O + 16 * u, o);
                    tmem_wait_ld();
                    reg_fence<16>(o);
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                    if (row < S) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + 16 * u);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
                if (h == 0 && row < S) p.lse[(size_t)bh * S + row] = (m_use + log2f(l_sum)) * FA_LN2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D>
cudaError_t fwd_tc_launch(const FwdArgs& a) {
    using C = Chunks<D>;
    using G = FwdCfg<D>;
    FwdParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    const void* src[3] = {a.q, a.k, a.v};
    CUtensorMap* maps[3] = {p.tq, p.tk, p.tv};
    for (int i = 0; i < 3; ++i) {
        cudaError_t e;
        if (C::N64 > 0 && (e = make_tmap_bf16_3d(&maps[i][0], src[i], D, a.S, BH, 64, BM)) != cudaSuccess) return e;
        if (C::REM > 0 && (e = make_tmap_bf16_3d(&maps[i][1], src[i], D, a.S, BH, C::REM, BM)) != cudaSuccess) return e;
    }
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.lse = a.lse;
    p.status = a.status;
    p.S = a.S;
    p.n_qt = (a.S + BM - 1) / BM;
    p.n_kv = (a.S + BN - 1) / BN;
    p.causal = a.causal;
    float c = fabsf(a.scale) * FA_LOG2E;
    p.c = c < 1e-30f ? 1e-30f : c;
    p.neg_a = a.scale < 0.f ? 1u : 0u;
    auto kern = fwd_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::DYN_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_qt * BH);
    kern<<<grid, NTHREADS, G::DYN_SMEM, a.stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a) {
    switch (a.d) {
        case 16: return fwd_tc_launch<16>(a);
        case 32: return fwd_tc_launch<32>(a);
        case 64: return fwd_tc_launch<64>(a);
        case 80: return fwd_tc_launch<80>(a);
        case 96: return fwd_tc_launch<96>(a);
        case 128: return fwd_tc_launch<128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
