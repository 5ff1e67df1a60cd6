// fa_fwd_tc.cu - bf16 FlashAttention-2 forward on the sm_103a tensor cores.
//
// Computes O = softmax(Q K^T * scale) V and L = logsumexp ("Stanford CS336
// Assignment 2 (Systems)" handout, section 4: Eq. 4-6, Eq. 12, Algorithm 1)
// with tcgen05.mma into Tensor Memory.
//
// One CTA owns two consecutive 128-row query tiles, A and B, of one
// (batch, head) and streams the 128-key K/V tiles they need through one
// TMA/mbarrier ring, so every K/V tile read from memory serves 256 query rows.
// Warp roles:
//   warps 0-3  softmax and epilogue of tile A (one query row per thread),
//   warps 4-7  softmax and epilogue of tile B,
//   warp  8    TMA producer (Q_A, Q_B once, then the K and V rings),
//   warp  9    Tensor Memory allocation and the MMA issuer (of tile A for d <= 64),
//   warp 10    the MMA issuer of tile B for d <= 64.
// The two softmax warpgroups work on different tiles, so while one of them
// turns S into P the tensor cores run the other tile's products.  One thread
// issues a tcgen05.mma only every ~80 cycles, longer than the tensor cores
// take for a 128x64x16 product, so for d <= 64 each tile has its own issuer.
//
// Tensor Memory (512 columns): S_A [0,128), S_B [128,256), then O_A, O_B.
// For d <= 64 the bf16 P of each tile has its own 64 columns after O_A, O_B:
// S_{j+1} = Q K_{j+1}^T is issued as soon as the softmax has read S_j, so a
// softmax warpgroup goes from one key tile to the next without waiting for the
// tensor cores.  For larger d the accumulators leave no room and P_j
// overwrites the first 64 columns of S_j (already in registers); S_{j+1} then
// follows the product P_j V_j.
//
// Online softmax (Algorithm 1) in base 2: scores are scaled by
// c = |scale| * log2(e).  The running max is always the exact max so far, which
// keeps the dominant probability of a sharp row at exactly 1.0 before the bf16
// rounding of P (letting the max lag by a few binades doubles the bf16 error of
// O for sharp softmax rows).  A warp rescales its rows of O only when one of
// its rows' max grew.  Fully masked causal tiles are never loaded or multiplied.
//
// Shapes: N_q query rows and N_k key rows may differ (Algorithm 1 takes Q in
// R^{N_q x d}, K, V in R^{N_k x d}); the causal mask keeps key j for query i
// when j <= i.  Q, K, V and O are [B, H, rows, d] views with any strides that
// are multiples of 8 elements (the TMA maps are 4-D over b, h, row, col).

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
constexpr int NTHREADS = 352;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;       // issues tile A's products and owns the Tensor Memory allocation
constexpr int MMA_WARP_B = 10;    // issues tile B's products
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_FLOOR = 120 * 1024;   // keeps one CTA per SM (it owns all of TMEM)

template <int D>
struct FwdTm {
    static constexpr bool PSEP = D <= 64;     // P has columns of its own
    __device__ static constexpr uint32_t s(int x) { return 128u * x; }
    __device__ static constexpr uint32_t o(int x) { return PSEP ? 256u + 64u * x : 256u + 128u * x; }
    __device__ static constexpr uint32_t pcol(int x) { return PSEP ? 384u + 64u * x : 128u * x; }
};

template <int D>
struct FwdCfg {
    static constexpr int TILE = Chunks<D>::tile_bytes(BM);
    static constexpr int NS_RAW = (222 * 1024 - 2 * TILE) / (2 * TILE);
    static constexpr int NS = NS_RAW > 4 ? 4 : NS_RAW;
    static constexpr int QA_OFF = 0;
    static constexpr int QB_OFF = TILE;
    static constexpr int K_OFF = 2 * TILE;
    static constexpr int V_OFF = K_OFF + NS * TILE;
    static constexpr int BAR_OFF = V_OFF + NS * TILE;
    // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS],
    // s_full[2], s_free[2], p_full[2], o_done[2], drain[2]
    static constexpr int NBARS = 1 + 4 * NS + 10;
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
    float* o32;       // partial attention: contiguous fp32 output (o unused)
    float* lse;       // contiguous [B*H, S]
    unsigned int* status;
    View vo;          // element strides of o
    int H;
    int S;            // query rows
    int n_units;      // 256-row query blocks per head
    int grp;          // heads per group of the grid order
    int Sk;           // key rows seen by the K/V tensor maps
    int n_kv;         // 128-key tiles in [0, Sk)
    int dshift;       // causal: key tile j is on query tile t's diagonal when j = t + dshift (<= 0)
    int causal;
    float c;          // |scale| * log2(e), at least 1e-30
    uint32_t neg_a;   // 1 when scale < 0: the S product negates Q
};

// P = exp2(S * c - m) for 32 pairs of scores r[0..63], rounded to bf16 pairs
// in pk, with the fp32 sums accumulated in sum[0..3].
__device__ __forceinline__ void exp_pairs(const uint32_t* r, uint64_t c2, uint64_t n2, uint32_t* pk, uint64_t* sum) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint64_t x = fma2(f2pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, n2);
        float x0, x1;
        f2unpack(x, x0, x1);
        const float p0 = ex2(x0);
        const float p1 = ex2(x1);
        sum[i & 3] = add2(sum[i & 3], f2pack(p0, p1));
        pk[i] = pack_bf16(p0, p1);
    }
}

// PARTIAL: attention of every query over the key window the K/V tensor maps
// start at (keys k0 + [0, Sk)), causal positions shifted by dshift tiles
// (k0 = -128 dshift); O is written normalised in fp32 and a query tile with
// no admissible key gets O = 0, L = -inf.  This is one side of the split-KV
// merge (see fa_merge_kernel).
template <int D, bool PARTIAL>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_tc_kernel(const __grid_constant__ FwdParams p) {
    using C = Chunks<D>;
    using G = FwdCfg<D>;
    using TM = FwdTm<D>;
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
    auto s_full = [&](int x) { return bar0 + 8u * (1 + 4 * NS + x); };
    auto s_free = [&](int x) { return bar0 + 8u * (3 + 4 * NS + x); };
    auto p_full = [&](int x) { return bar0 + 8u * (5 + 4 * NS + x); };
    auto o_done = [&](int x) { return bar0 + 8u * (7 + 4 * NS + x); };
    auto drain = [&](int x) { return bar0 + 8u * (9 + 4 * NS + x); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // One flat grid ordered rank-major: every head's longest causal block is
    // dispatched before any head's next one (longest job first), within head
    // groups when the heads' K and V would not stay in L2 together.
    const int BH = (int)(gridDim.x / (unsigned)p.n_units);
    int rank, bh;
    if (p.grp >= BH) {
        rank = (int)blockIdx.x / BH;
        bh = (int)blockIdx.x - rank * BH;
    } else {
        grid_unit((int)blockIdx.x, BH, p.n_units, p.grp, rank, bh);
    }
    const int bb = bh / p.H, hh = bh - bb * p.H;
    const int unit = p.causal ? (p.n_units - 1 - rank) : rank;
    const int S = p.S;
    const int qtA = 2 * unit;
    const bool hasB = (qtA + 1) * BM < S;
    // Last key tile of each query tile (inclusive, -1: none); jB >= jA.
    const int jA = p.causal ? min(qtA + p.dshift, p.n_kv - 1) : p.n_kv - 1;
    const int jB = hasB ? (p.causal ? min(qtA + 1 + p.dshift, p.n_kv - 1) : p.n_kv - 1) : jA;
    const int n_issuers = TM::PSEP ? (jA >= 0 ? 1 : 0) + ((hasB && jB >= 0) ? 1 : 0) : 1;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        // A K/V stage is free once each issuer has committed its last product
        // that reads it (the last key tile of a causal block, used by tile B
        // alone, is never refilled).
        for (int s = 0; s < NS; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), n_issuers > 0 ? n_issuers : 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), n_issuers > 0 ? n_issuers : 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(s_free(x), BM);
            mbar_init(p_full(x), BM);
            mbar_init(o_done(x), 1);
            mbar_init(drain(x), 1);
        }
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
    griddep_launch();

    if (warp == TMA_WARP) {
        // ------------------------------------------------------------ producer
        int issued_k = 0, issued_v = 0;
        if (lane == 0) {
            for (int i = 0; i < 2; ++i) {
                prefetch_tmap(&p.tq[i]);
                prefetch_tmap(&p.tk[i]);
                prefetch_tmap(&p.tv[i]);
            }
            // Q, K, V may come from the previous kernel on the stream; every
            // global access of this CTA follows these loads.
            griddep_wait();
            mbar_arrive_expect_tx(q_full, (hasB ? 2 : 1) * G::TILE);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_4d(sb + G::QA_OFF + C::tile_off(c, BM), &p.tq[C::map_index(c)], c * 64, qtA * BM, hh, bb,
                            q_full);
                if (hasB)
                    tma_load_4d(sb + G::QB_OFF + C::tile_off(c, BM), &p.tq[C::map_index(c)], c * 64, (qtA + 1) * BM,
                                hh, bb, q_full);
            }
            for (int j = 0; j <= jB; ++j) {
                const int st = j % NS;
                const uint32_t ph = (j / NS) & 1;
                if (!mbar_wait(k_empty(st), ph ^ 1, abort, p.status, WAIT_LIMIT_NS)) break;
                mbar_arrive_expect_tx(k_full(st), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(sb + G::K_OFF + st * G::TILE + C::tile_off(c, BN), &p.tk[C::map_index(c)],
                                c * 64, j * BN, hh, bb, k_full(st));
                issued_k = j + 1;
                if (!mbar_wait(v_empty(st), ph ^ 1, abort, p.status, WAIT_LIMIT_NS)) break;
                mbar_arrive_expect_tx(v_full(st), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(sb + G::V_OFF + st * G::TILE + C::tile_off(c, BN), &p.tv[C::map_index(c)],
                                c * 64, j * BN, hh, bb, v_full(st));
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
    } else if (warp == MMA_WARP || (TM::PSEP && warp == MMA_WARP_B && hasB)) {
        // ------------------------------------------------------------ MMA issuers
        const uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0) | (p.neg_a << 13);
        const uint32_t q_lo0 = desc_lo(sb + G::QA_OFF, 16);
        const uint32_t k_lo0 = desc_lo(sb + G::K_OFF, 16);
        const uint32_t v_lo0 = desc_lo(sb + G::V_OFF, BN * 128);
        // S_x(j) = Q_x K_j^T into tile x's score columns.
        auto issue_s = [&](int x, int j) {
            const uint32_t q_lo = q_lo0 + (uint32_t)x * (G::TILE >> 4);
            const uint32_t klo = k_lo0 + (uint32_t)(j % NS) * (G::TILE >> 4);
            int step = 0;
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
                for (int s = 0; s < C::width(c) / 16; ++s, ++step) {
                    const uint32_t off = (C::tile_off(c, BM) + s * 32) >> 4;
                    const uint32_t hi = desc_hi(8 * C::row_bytes(c), C::swz(c));
                    mma_ss(tmem + TM::s(x), desc_make(q_lo + off, hi), desc_make(klo + off, hi), idesc_s,
                           step > 0 ? 1u : 0u);
                }
            }
            mma_commit(s_full(x));
        };
        // O_x += P_x(j) V_j: A = P from Tensor Memory, B = V_j (MN-major, keys along K).
        auto issue_pv = [&](int x, int j) {
            const uint32_t vlo = v_lo0 + (uint32_t)(j % NS) * (G::TILE >> 4);
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks) {
                const uint32_t a_tm = tmem + TM::pcol(x) + ks * 8;
                const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
                if constexpr (C::SINGLE_N) {
                    mma_ts(tmem + TM::o(x), a_tm, desc_make(vlo + ks * 128, desc_hi(1024, SW_128B)),
                           idesc_bf16(BM, D, 0, 1), acc);
                } else {
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c) {
                        const uint32_t off = (C::tile_off(c, BN) + ks * 16 * C::row_bytes(c)) >> 4;
                        mma_ts(tmem + TM::o(x) + c * 64, a_tm,
                               desc_make(vlo + off, desc_hi(8 * C::row_bytes(c), C::swz(c))),
                               idesc_bf16(BM, C::width(c), 0, 1), acc);
                    }
                }
            }
            mma_commit(o_done(x));
        };
        // One thread runs the issuer role from start to end and waits on the
        // barriers itself: a warp-collective operation between products
        // (a shuffle or warp sync per wait) stalls the issuing path for
        // several hundred cycles, during which the tensor pipe runs dry.
        if (lane == 0) {
        auto wait = [&](uint32_t bar, uint32_t parity) {
            return mbar_wait(bar, parity, abort, p.status, WAIT_LIMIT_NS);
        };
        // Nothing to multiply when no key tile is admissible (partial attention).
        bool ok = jB >= 0 && wait(q_full, 0);
        if (ok) ok = wait(k_full(0), 0);
        if constexpr (TM::PSEP) {
            // One issuer per tile; the next scores go in as soon as the
            // softmax has read these.
            const int x = warp - MMA_WARP;
            const int jX = x ? jB : jA;
            if (jX < 0) ok = false;
            if (ok) {
                tc_fence_after();
                issue_s(x, 0);
                mma_commit(k_empty(0));
            }
            for (int j = 0; j <= jX && ok; ++j) {
                const int st1 = (j + 1) % NS;
                if (j + 1 <= jX) {
                    if (!(ok = wait(k_full(st1), ((j + 1) / NS) & 1))) break;
                    if (!(ok = wait(s_free(x), j & 1))) break;
                    tc_fence_after();
                    issue_s(x, j + 1);
                    mma_commit(k_empty(st1));
                }
                if (!(ok = wait(v_full(j % NS), (j / NS) & 1))) break;
                if (!(ok = wait(p_full(x), j & 1))) break;
                tc_fence_after();
                issue_pv(x, j);
                mma_commit(v_empty(j % NS));
            }
        } else {
            // P_j sits in S_j's columns, so S_{j+1} follows P_j V_j.  One
            // issuer alternates between the tiles: while one softmax
            // warpgroup works, the tensor cores run the other tile's products.
            auto tile_has = [&](int x, int j) { return x == 0 ? j <= jA : (hasB && j <= jB); };
            if (ok) {
                tc_fence_after();
                if (tile_has(0, 0)) issue_s(0, 0);
                if (tile_has(1, 0)) issue_s(1, 0);
                mma_commit(k_empty(0));
            }
            for (int j = 0; j <= jB && ok; ++j) {
                const bool next = j + 1 <= jB;
                const int st1 = (j + 1) % NS;
                if (!(ok = wait(v_full(j % NS), (j / NS) & 1))) break;
                if (next && !(ok = wait(k_full(st1), ((j + 1) / NS) & 1))) break;
                for (int x = 0; x < 2 && ok; ++x) {
                    if (!tile_has(x, j)) continue;
                    if (!(ok = wait(p_full(x), j & 1))) break;
                    tc_fence_after();
                    issue_pv(x, j);
                    if (tile_has(x, j + 1)) issue_s(x, j + 1);
                }
                if (!ok) break;
                mma_commit(v_empty(j % NS));
                if (next) mma_commit(k_empty(st1));
            }
        }
        if (*abort) {
            // Wait until every MMA this thread issued has finished before TMEM is freed.
            volatile int no_abort = 0;
            mma_commit(drain(warp - MMA_WARP));
            mbar_wait(drain(warp - MMA_WARP), 0, &no_abort, p.status, WAIT_LIMIT_NS);
        }
        }
        __syncwarp();
    } else if (warp < 4 || (warp < 8 && hasB)) {
        // ------------------------------------------------------------ softmax + epilogue of tile x
        const int x = warp >> 2;
        const int wq = warp & 3;                 // lane quarter of Tensor Memory
        const int row_local = wq * 32 + lane;
        const int qt = qtA + x;
        const int row = qt * BM + row_local;
        const int jX = x ? jB : jA;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + TM::s(x);
        const uint32_t tP = tmem + lane_off + TM::pcol(x);
        const uint32_t tO = tmem + lane_off + TM::o(x);
        const float c = p.c;
        const int Sk = p.Sk;
        const int key_lim = p.causal ? min(row + BM * p.dshift, Sk - 1) : Sk - 1;   // in window coordinates
        float m_use = -INFINITY;
        float l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j <= jX; ++j) {
            if (!(ok = warp_wait(s_full(x), j & 1, abort, p.status))) break;
            tc_fence_after();
            uint32_t r[128];
            tmem_ld32(tS, r);
            tmem_ld32(tS + 32, r + 32);
            tmem_ld32(tS + 64, r + 64);
            tmem_ld32(tS + 96, r + 96);
            tmem_wait_ld();
            reg_fence<128>(r);
            if constexpr (TM::PSEP) {
                tc_fence_before();
                mbar_arrive(s_free(x));          // the next scores may overwrite these columns
            }
            // Only the diagonal tile of a causal row block and a ragged last
            // tile need the per-element mask; masked scores become -inf.
            const int kbase = j * BN;
            const bool masked = (p.causal && j == qt + p.dshift) || (kbase + BN > Sk);
            if (masked) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (kbase + i > key_lim) r[i] = 0xff800000u;
            }
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 128; i += 8) {
                mx0 = max3f(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                mx1 = max3f(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                mx2 = max3f(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                mx3 = max3f(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
            }
            const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3));
            const float m_new = fmaxf(m_use, mx * c);
            const float alpha = (j == 0 || m_new == m_use) ? 1.f : ex2(m_use - m_new);
            m_use = m_new;
            const float neg = (m_use == -INFINITY) ? 0.f : -m_use;
            const uint64_t c2 = f2pack(c, c);
            const uint64_t n2 = f2pack(neg, neg);
            // P = exp2(S*c - m) rounded to bf16, and the fp32 row sum; P goes
            // to Tensor Memory in two halves of 32 columns.
            uint64_t sum[4] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
                exp_pairs(r + 64 * half, c2, n2, pk, sum);
                // The previous product P_{j-1} V_{j-1} must have finished: it
                // read the P columns and it wrote the O rescaled below.
                // d > 64: S_j's commit follows P_{j-1} V_{j-1} on the same issuer, so
                // s_full already implies it; d <= 64 issues S_j ahead of it.
                if (TM::PSEP && half == 0 && j > 0) {
                    if (!(ok = warp_wait(o_done(x), (j - 1) & 1, abort, p.status))) break;
                    tc_fence_after();
                }
                tmem_st32(tP + 32 * half, pk);
            }
            if (!ok) break;
            float s0, s1, s2, s3, s4, s5, s6, s7;
            f2unpack(sum[0], s0, s1);
            f2unpack(sum[1], s2, s3);
            f2unpack(sum[2], s4, s5);
            f2unpack(sum[3], s6, s7);
            l_sum = l_sum * alpha + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // O *= alpha, up to 64 columns per Tensor Memory round trip.
                const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
                for (int u0 = 0; u0 < D / 16; u0 += 4) {
                    constexpr int NB = 4;
                    uint32_t o[16 * NB];
#pragma unroll
                    for (int u = 0; u < NB; ++u)
                        if (u0 + u < D / 16) tmem_ld16(tO + 16 * (u0 + u), o + 16 * u);
                    tmem_wait_ld();
                    reg_fence<16 * NB>(o);
#pragma unroll
                    for (int i = 0; i < 16 * NB; i += 2) {
                        float lo, hi;
                        f2unpack(mul2(f2pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), lo, hi);
                        o[i] = __float_as_uint(lo);
                        o[i + 1] = __float_as_uint(hi);
                    }
#pragma unroll
                    for (int u = 0; u < NB; ++u)
                        if (u0 + u < D / 16) tmem_st16(tO + 16 * (u0 + u), o + 16 * u);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_full(x));
        }
        // Epilogue (the end of Algorithm 1's outer loop): O / l and L = (m + log2 l) ln 2.
        if (ok && jX < 0) {
            // No admissible key in the window (partial attention only).
            if constexpr (PARTIAL) {
                if (row < S) {
                    float4* dst = reinterpret_cast<float4*>(p.o32 + ((size_t)bh * S + row) * D);
#pragma unroll
                    for (int u = 0; u < D / 4; ++u) dst[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    p.lse[(size_t)bh * S + row] = -INFINITY;
                }
            }
        } else if (ok && warp_wait(o_done(x), jX & 1, abort, p.status)) {
            tc_fence_after();
            const float inv = 1.f / l_sum;
#pragma unroll
            for (int u = 0; u < D / 16; ++u) {
                uint32_t o[16];
                tmem_ld16(tO + 16 * u, o);
                tmem_wait_ld();
                reg_fence<16>(o);
                if (row >= S) continue;
                if constexpr (PARTIAL) {
                    float4* dst = reinterpret_cast<float4*>(p.o32 + ((size_t)bh * S + row) * D + 16 * u);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                             __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
                } else {
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(p.o + p.vo.off(bb, hh, row) + 16 * u);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
            if (row < S) p.lse[(size_t)bh * S + row] = (m_use + log2f(l_sum)) * FA_LN2;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D, bool PARTIAL>
cudaError_t fwd_tc_launch(const FwdArgs& a, int key_begin, int key_end, float* o32) {
    using C = Chunks<D>;
    using G = FwdCfg<D>;
    FwdParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    // K and V tensor maps start at the key window [key_begin, key_end) of the
    // a.Sk keys; the views' strides are unchanged.
    const int Sk = key_end - key_begin;
    const void* src[3] = {a.q, static_cast<const __nv_bfloat16*>(a.k) + (size_t)key_begin * a.vk.s,
                          static_cast<const __nv_bfloat16*>(a.v) + (size_t)key_begin * a.vv.s};
    const int rows[3] = {a.S, Sk, Sk};
    const View views[3] = {a.vq, a.vk, a.vv};
    CUtensorMap* maps[3] = {p.tq, p.tk, p.tv};
    for (int i = 0; i < 3; ++i) {
        cudaError_t e;
        if (C::N64 > 0 &&
            (e = make_tmap_bf16_4d(&maps[i][0], src[i], D, rows[i], a.H, a.B, views[i], 64, BM)) != cudaSuccess)
            return e;
        if (C::REM > 0 && !C::PAD &&
            (e = make_tmap_bf16_4d(&maps[i][1], src[i], D, rows[i], a.H, a.B, views[i], C::REM, BM)) != cudaSuccess)
            return e;
    }
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.o32 = o32;
    p.lse = a.lse;
    p.status = a.status;
    p.vo = a.vo;
    p.H = a.H;
    p.S = a.S;
    p.n_units = (a.S + 2 * BM - 1) / (2 * BM);
    // Each CTA streams its head's K and V (bf16): grouped from 128 MiB of K
    // and V, so that a group's CTAs re-read them from L2 (B4 H32 S4096 d80:
    // DRAM reads 1.11 GB -> 0.25 GB per launch, time -1 %), and only with
    // many heads (B1 H16 S32768 d128 was 7 % slower grouped).
    p.grp = head_group(BH, p.n_units, 4.0 * Sk * D, 128.0, true);
    p.Sk = Sk;
    p.n_kv = (Sk + BN - 1) / BN;
    p.dshift = -(key_begin / BN);
    p.causal = a.causal;
    float c = fabsf(a.scale) * FA_LOG2E;
    p.c = c < 1e-30f ? 1e-30f : c;
    p.neg_a = a.scale < 0.f ? 1u : 0u;
    auto kern = fwd_tc_kernel<D, PARTIAL>;
    cudaError_t e = set_smem_limit<fwd_tc_kernel<D, PARTIAL>>(G::DYN_SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.n_units * BH), dim3(NTHREADS), G::DYN_SMEM, a.stream, p);
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a) {
    switch (a.d) {
        case 16: return fwd_tc_launch<16, false>(a, 0, a.Sk, nullptr);
        case 32: return fwd_tc_launch<32, false>(a, 0, a.Sk, nullptr);
        case 64: return fwd_tc_launch<64, false>(a, 0, a.Sk, nullptr);
        case 80: return fwd_tc_launch<80, false>(a, 0, a.Sk, nullptr);
        case 96: return fwd_tc_launch<96, false>(a, 0, a.Sk, nullptr);
        case 128: return fwd_tc_launch<128, false>(a, 0, a.Sk, nullptr);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fwd_tc_partial(const FwdArgs& a, int key_begin, int key_end, float* o32) {
    switch (a.d) {
        case 16: return fwd_tc_launch<16, true>(a, key_begin, key_end, o32);
        case 32: return fwd_tc_launch<32, true>(a, key_begin, key_end, o32);
        case 64: return fwd_tc_launch<64, true>(a, key_begin, key_end, o32);
        case 80: return fwd_tc_launch<80, true>(a, key_begin, key_end, o32);
        case 96: return fwd_tc_launch<96, true>(a, key_begin, key_end, o32);
        case 128: return fwd_tc_launch<128, true>(a, key_begin, key_end, o32);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
