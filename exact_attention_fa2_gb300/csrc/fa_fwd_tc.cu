// fa_fwd_tc.cu - bf16 FlashAttention-2 forward on the sm_103a tensor cores.
//
// Computes O = softmax(Q K^T * scale) V and L = logsumexp ("Stanford CS336
// Assignment 2 (Systems)" handout, section 4: Eq. 4-6, Eq. 12, Algorithm 1)
// with tcgen05.mma into Tensor Memory.
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams the
// 128-key K/V tiles they need through a TMA/mbarrier ring.  Warp roles:
//   warps 0-3  softmax for query tile 0 (one thread per query row),
//   warps 4-7  softmax for query tile 1,
//   warp  8    TMA producer (Q tiles once, then the K and V rings),
//   warp  9    Tensor Memory allocation and the single-thread MMA issuer.
// Tensor Memory (512 columns): S_t in columns [128t, 128t+128) for the two
// tiles, O_t in [256+128t, 256+128t+d).  P_t (bf16) overwrites the first 64
// columns of S_t and is read from there by the PV product.  While one tile's
// softmax runs, the tensor cores work on the other tile (ping-pong).
//
// Online softmax (Algorithm 1 lines 10-13) in base 2: scores are scaled by
// c = |scale| * log2(e).  A warp rescales its rows of O in Tensor Memory only
// when some row's running max grew; rows whose max did not grow multiply by 1.
// The running max is always the exact max so far, which keeps the dominant
// probability of a sharp row at exactly 1.0 before the bf16 rounding of P
// (letting the max lag by a few binades would double the bf16 error of O for
// sharp softmax rows).
// Fully masked causal tiles are never loaded or multiplied.

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
constexpr float RESCALE_THRESHOLD = 0.0f;
constexpr int SMEM_FLOOR = 120 * 1024;   // keeps one CTA per SM (it owns all of TMEM)

template <int D>
struct FwdCfg {
    static constexpr int TILE = BM * D * 2;
    static constexpr int NS_RAW = (225 * 1024 - 2 * TILE) / (2 * TILE);
    static constexpr int NS = NS_RAW > 4 ? 4 : NS_RAW;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + 2 * TILE;
    static constexpr int V_OFF = K_OFF + NS * TILE;
    static constexpr int BAR_OFF = V_OFF + NS * TILE;
    // q_full[2], k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[2], p_full[2], o_full[2], drain
    static constexpr int NBARS = 2 + 4 * NS + 7;
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
    int n_pairs;
    int n_kv;
    int causal;
    float c;          // |scale| * log2(e), at least 1e-30
    uint32_t neg_a;   // 1 when scale < 0: the S product negates Q
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_tc_kernel(const __grid_constant__ FwdParams p) {
    using C = Chunks<D>;
    using G = FwdCfg<D>;
    constexpr int NS = G::NS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + G::BAR_OFF;
    auto q_full = [&](int t) { return bar0 + 8u * t; };
    auto k_full = [&](int s) { return bar0 + 8u * (2 + s); };
    auto k_empty = [&](int s) { return bar0 + 8u * (2 + NS + s); };
    auto v_full = [&](int s) { return bar0 + 8u * (2 + 2 * NS + s); };
    auto v_empty = [&](int s) { return bar0 + 8u * (2 + 3 * NS + s); };
    auto s_full = [&](int t) { return bar0 + 8u * (2 + 4 * NS + t); };
    auto p_full = [&](int t) { return bar0 + 8u * (4 + 4 * NS + t); };
    auto o_full = [&](int t) { return bar0 + 8u * (6 + 4 * NS + t); };
    const uint32_t drain = bar0 + 8u * (8 + 4 * NS);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pair = p.causal ? (p.n_pairs - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int bh = blockIdx.y;
    const int S = p.S;

    // Query tile t covers rows [q0(t), q0(t)+128) and needs key tiles 0..jmax(t).
    auto q0 = [&](int t) { return pair * 2 * BM + t * BM; };
    auto active = [&](int t) { return q0(t) < S; };
    auto jmax = [&](int t) { return p.causal ? min(2 * pair + t, p.n_kv - 1) : p.n_kv - 1; };
    const int n_iter = (active(1) ? max(jmax(0), jmax(1)) : jmax(0)) + 1;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(q_full(t), 1);
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), BM);
            mbar_init(o_full(t), 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        mbar_init(drain, 1);
        *abort = 0;
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
            for (int t = 0; t < 2; ++t) {
                if (!active(t)) continue;
                mbar_arrive_expect_tx(q_full(t), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sb + G::Q_OFF + t * G::TILE + C::tile_off(c, BM), &p.tq[C::map_index(c)],
                                c * 64, q0(t), bh, q_full(t));
            }
            for (int j = 0; j < n_iter; ++j) {
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
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t)
            if (active(t)) ok = warp_wait(q_full(t), 0, abort, p.status);
        for (int j = 0; j <= n_iter && ok; ++j) {
            const int st = j % NS;
            const uint32_t ph = (j / NS) & 1;
            const int sp = (j + NS - 1) % NS;
            const uint32_t pph = ((j - 1) / NS) & 1;
            if (j < n_iter && !(ok = warp_wait(k_full(st), ph, abort, p.status))) break;
            bool v_ready = false;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!active(t)) continue;
                if (j >= 1 && j - 1 <= jmax(t)) {
                    if (!v_ready) {
                        if (!(ok = warp_wait(v_full(sp), pph, abort, p.status))) break;
                        v_ready = true;
                    }
                    if (!(ok = warp_wait(p_full(t), (j - 1) & 1, abort, p.status))) break;
                    tc_fence_after();
                    if (lane == 0) {
                        // O_t += P_t V_{j-1}: A = P from TMEM, B = V (MN-major, keys along K).
                        const uint32_t d_o = tmem + 256 + t * 128;
                        const uint32_t vbase = sb + G::V_OFF + sp * G::TILE;
#pragma unroll
                        for (int ks = 0; ks < BN / 16; ++ks) {
                            const uint32_t a_tm = tmem + t * 128 + ks * 8;
                            const uint32_t acc = (j - 1 > 0 || ks > 0) ? 1u : 0u;
                            if constexpr (D == 128) {
                                const uint64_t bdesc = smem_desc(vbase + ks * 16 * 128, BN * 128, 1024, SW_128B);
                                mma_ts(d_o, a_tm, bdesc, idesc_bf16(BM, 128, 0, 1), acc);
                            } else {
#pragma unroll
                                for (int c = 0; c < C::NCH; ++c) {
                                    const uint64_t bdesc = smem_desc(
                                        vbase + C::tile_off(c, BN) + ks * 16 * C::row_bytes(c), BN * 128,
                                        8 * C::row_bytes(c), C::swz(c));
                                    mma_ts(d_o + c * 64, a_tm, bdesc, idesc_bf16(BM, C::width(c), 0, 1), acc);
                                }
                            }
                        }
                        if (j - 1 == jmax(t)) mma_commit(o_full(t));
                    }
                }
                if (j < n_iter && j <= jmax(t)) {
                    if (lane == 0) {
                        // S_t = Q_t K_j^T: both operands K-major (head dim contiguous).
                        const uint32_t d_s = tmem + t * 128;
                        const uint32_t qbase = sb + G::Q_OFF + t * G::TILE;
                        const uint32_t kbase = sb + G::K_OFF + st * G::TILE;
                        int step = 0;
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
                            for (int s = 0; s < C::width(c) / 16; ++s, ++step) {
                                const uint32_t off = C::tile_off(c, BM) + s * 32;
                                const uint64_t adesc = smem_desc(qbase + off, 16, 8 * C::row_bytes(c), C::swz(c));
                                const uint64_t bdesc = smem_desc(kbase + off, 16, 8 * C::row_bytes(c), C::swz(c));
                                mma_ss(d_s, adesc, bdesc, idesc_s, step > 0 ? 1u : 0u);
                            }
                        }
                        mma_commit(s_full(t));
                    }
                }
            }
            if (!ok) break;
            if (lane == 0) {
                if (j < n_iter) mma_commit(k_empty(st));
                if (j >= 1) mma_commit(v_empty(sp));
            }
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
        const int t = warp >> 2;
        const int wq = warp & 3;
        if (active(t)) {
            const int row_local = wq * 32 + lane;
            const int row = q0(t) + row_local;
            const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
            const uint32_t tS = tmem + lane_off + t * 128;
            const uint32_t tO = tmem + lane_off + 256 + t * 128;
            const float c = p.c;
            const int key_lim = p.causal ? min(row, S - 1) : S - 1;
            float m_use = -INFINITY;
            float l_sum = 0.f;
            bool ok = true;
            for (int j = 0; j <= jmax(t); ++j) {
                if (!(ok = warp_wait(s_full(t), j & 1, abort, p.status))) break;
                tc_fence_after();
                // Pass 1: row max over the tile, 64 columns at a time (keeps
                // register use within the 168 per thread that ten warps allow).
                // Only the diagonal tile of a causal row block and a ragged
                // last tile need the per-element mask; masked scores become
                // -inf, which exp2 maps to 0 in pass 2.
                const int kbase = j * BN;
                const bool mask_tile = (p.causal && j == jmax(t)) || (kbase + BN > S);
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[64];
                    tmem_ld32(tS + 64 * h, r);
                    tmem_ld32(tS + 64 * h + 32, r + 32);
                    tmem_wait_ld();
                    reg_fence<64>(r);
                    if (mask_tile) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (kbase + 64 * h + i > key_lim) r[i] = 0xff800000u;
                    }
#pragma unroll
                    for (int i = 0; i < 64; i += 8) {
                        mx0 = max3f(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                        mx1 = max3f(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                        mx2 = max3f(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                        mx3 = max3f(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                    }
                }
                const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3));
                const float m_tile = mx * c;
                const float m_new = fmaxf(m_use, m_tile);
                if (j == 0) {
                    m_use = m_new;
                } else {
                    const bool need = m_new > m_use + RESCALE_THRESHOLD;
                    if (__any_sync(0xffffffffu, need)) {
                        const float alpha = need ? ex2(m_use - m_new) : 1.f;
                        if (need) {
                            l_sum *= alpha;
                            m_use = m_new;
                        }
                        const uint64_t a2 = f2pack(alpha, alpha);
                        // O is idle here: the PV product of the previous tile
                        // completed before this tile's S product (issue order).
#pragma unroll
                        for (int cb = 0; cb < D; cb += 64) {
                            constexpr int W = D < 64 ? D : 64;
                            const int n = (D - cb) < W ? (D - cb) : W;
                            uint32_t o[64];
#pragma unroll
                            for (int u = 0; u < W / 16; ++u)
                                if (16 * u < n) tmem_ld16(tO + cb + 16 * u, o + 16 * u);
                            tmem_wait_ld();
                            reg_fence<64>(o);
#pragma unroll
                            for (int i = 0; i < W; i += 2) {
                                if (i < n) {
                                    float lo, hi;
                                    f2unpack(mul2(f2pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), lo, hi);
                                    o[i] = __float_as_uint(lo);
                                    o[i + 1] = __float_as_uint(hi);
                                }
                            }
#pragma unroll
                            for (int u = 0; u < W / 16; ++u)
                                if (16 * u < n) tmem_st16(tO + cb + 16 * u, o + 16 * u);
                        }
                    }
                }
                const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
                const uint64_t c2 = f2pack(c, c);
                const uint64_t n2 = f2pack(neg, neg);
                // Pass 2: P = exp2(S*c - m) rounded to bf16 into the first 64
                // columns of S (columns already read), and its fp32 row sum.
                uint64_t sum_a = f2pack(0.f, 0.f), sum_b = f2pack(0.f, 0.f);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[64];
                    tmem_ld32(tS + 64 * h, r);
                    tmem_ld32(tS + 64 * h + 32, r + 32);
                    tmem_wait_ld();
                    reg_fence<64>(r);
                    if (mask_tile) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            if (kbase + 64 * h + i > key_lim) r[i] = 0xff800000u;
                    }
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
                }
                float s0, s1, s2, s3;
                f2unpack(sum_a, s0, s1);
                f2unpack(sum_b, s2, s3);
                const float sum = (s0 + s1) + (s2 + s3);
                l_sum += sum;
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_full(t));
            }
            // Epilogue (Algorithm 1 lines 15-18).
            if (ok && warp_wait(o_full(t), 0, abort, p.status)) {
                tc_fence_after();
                const float inv = 1.f / l_sum;
                __nv_bfloat16* orow = p.o + ((size_t)bh * S + row) * D;
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    uint32_t o[16];
                    tmem_ld16(tO + 16 * cc, o);
                    tmem_wait_ld();
                    reg_fence<16>(o);
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                    if (row < S) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + 16 * cc);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
                if (row < S) p.lse[(size_t)bh * S + row] = (m_use + log2f(l_sum)) * FA_LN2;
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
    p.n_pairs = (a.S + 2 * BM - 1) / (2 * BM);
    p.n_kv = (a.S + BN - 1) / BN;
    p.causal = a.causal;
    float c = fabsf(a.scale) * FA_LOG2E;
    p.c = c < 1e-30f ? 1e-30f : c;
    p.neg_a = a.scale < 0.f ? 1u : 0u;
    auto kern = fwd_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::DYN_SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_pairs, BH);
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
