// fa_bwd_dq_tc.cu - query-tile-outer dQ pass of the deterministic backward,
// bf16 on the sm_103a tensor cores.
//
// "Stanford CS336 Assignment 2 (Systems)" handout, section 4, Algorithm 2 as
// it stands: dQ gets a loop of its own with the query tile outside and the
// key tiles inside, recomputing P (Eq. 13-14), dP (Eq. 16) and dS (Eq. 17)
// rather than sharing them with the dK/dV loop.  Every dQ row is then summed
// by one CTA in a fixed order (Eq. 18) with no atomics, so together with the
// dK/dV-only instance of the key-tile-outer kernel the backward is bitwise
// reproducible.  The price is a second S and dP product per tile pair.
//
// One CTA owns one 128-row query tile of one (batch, head): Q_i and dO_i stay
// in shared memory, (L, D) of its rows in registers and dQ_i in Tensor
// Memory, while the 128-key K/V tiles stream through a TMA ring.  Per key
// tile j (fp32 accumulation throughout):
//   S   = Q_i K_j^T,  dP = dO_i V_j^T
//   P   = exp2(S c - L log2 e),  dS = P * (dP - D)   (dS rounded to bf16)
//   dQ += dS K_j      (A = dS from Tensor Memory, B = K_j read MN-major)
// and at the end dq = dQ * scale rounded to bf16.
//
// Warp roles: warps 0-7 dS (one query row per thread; warps 0-3 keys 0-63,
// warps 4-7 keys 64-127) and the dq store, warp 8 TMA, warp 9 Tensor Memory
// allocation and the S/dP issuer, warp 10 the dQ issuer.  One thread issues a
// tcgen05.mma only every ~80 cycles, so two issuing threads keep the tensor
// cores busier than one.
// Shapes as in the key-tile-outer kernel: N_q queries, N_k keys, strided
// [B, H, rows, d] views (strides multiples of 8 elements), contiguous L, D.
// Tensor Memory columns: S [0,128), dP [128,256), two bf16 dS buffers
// [256,320) and [320,384), dQ [384, 384+d).  S_{j+1} and dP_{j+1} are issued
// as soon as the dS warps have read S_j and dP_j, so the products of the next
// key tile run while dS_j is formed and dQ += dS_j K_j follows them.

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

constexpr int BQ = 128;
constexpr int BK = 128;
constexpr int NTHREADS = 352;
constexpr int TMA_WARP = 8;
constexpr int SDP_WARP = 9;       // S/dP issuer, owns the Tensor Memory allocation
constexpr int DQ_WARP = 10;       // dQ issuer
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DS = 256, TM_DQ = 384;
constexpr int SMEM_BUDGET = 227 * 1024;
constexpr int SMEM_FLOOR = 120 * 1024;   // keeps one CTA per SM (it owns all of TMEM)

template <int D>
struct DqCfg {
    static constexpr int TILE = Chunks<D>::tile_bytes(128);
    static constexpr int STAGE = 2 * TILE;                  // K_j then V_j
    static constexpr int NS_RAW = (SMEM_BUDGET - 2 * TILE - 1024 - 256) / STAGE;
    static constexpr int NS = NS_RAW > 4 ? 4 : NS_RAW;
    static constexpr int Q_OFF = 0;
    static constexpr int DO_OFF = TILE;
    static constexpr int RING_OFF = 2 * TILE;
    static constexpr int BAR_OFF = RING_OFF + NS * STAGE;
    // qd_full, k_full[NS], v_full[NS], kv_empty[NS], s_full, s_free,
    // ds_full[2], ds_free[2], dq_done, drain[2]
    static constexpr int NBARS = 1 + 3 * NS + 9;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int DYN_SMEM = (BYTES + 1024) > SMEM_FLOOR ? (BYTES + 1024) : SMEM_FLOOR;
    static_assert(NS >= 2, "K/V ring needs two stages");
    static_assert(DYN_SMEM <= SMEM_BUDGET, "shared memory budget");
    static_assert(TM_DQ + D <= TMEM_COLS, "Tensor Memory budget");
};

struct DqParams {
    CUtensorMap tq[2];
    CUtensorMap tk[2];
    CUtensorMap tv[2];
    CUtensorMap tdo[2];
    const float* lse;     // contiguous [B*H, S]
    const float* Dvec;    // contiguous [B*H, S]
    __nv_bfloat16* dq;
    unsigned int* status;
    View vdq;             // element strides of dq
    int H;
    int S;                // query rows N_q
    int Sk;               // key rows N_k
    int n_q;
    int n_kv;
    int grp;              // heads per group of the grid order
    int causal;
    float c;          // |scale| * log2(e), at least 1e-30
    float scale;      // signed scale applied to dq
    uint32_t neg_a;   // 1 when scale < 0: S = -(Q K^T) so that exp uses |scale|
};

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1) bwd_dq_tc_kernel(const __grid_constant__ DqParams p) {
    using C = Chunks<D>;
    using G = DqCfg<D>;
    constexpr int NS = G::NS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (smem + G::BYTES > smem_raw + G::DYN_SMEM) {
        if (threadIdx.x == 0) set_status(p.status, FA_DEV_STATUS_BOUNDS);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + G::BAR_OFF;
    const uint32_t qd_full = bar0;
    auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto v_full = [&](int s) { return bar0 + 8u * (1 + NS + s); };
    auto kv_empty = [&](int s) { return bar0 + 8u * (1 + 2 * NS + s); };
    const uint32_t s_full = bar0 + 8u * (1 + 3 * NS);
    const uint32_t s_free = s_full + 8;
    auto ds_full = [&](int b) { return s_full + 16u + 8u * b; };
    auto ds_free = [&](int b) { return s_full + 32u + 8u * b; };
    const uint32_t dq_done = s_full + 48;
    auto drain = [&](int x) { return s_full + 56u + 8u * x; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // One flat grid ordered rank-major: under the causal mask the last query
    // tiles see the most key tiles, so every head's heaviest tile goes first
    // (within head groups when the heads' K and V would not stay in L2 together).
    const int BH = (int)(gridDim.x / (unsigned)p.n_q);
    int rank, bh;
    if (p.grp >= BH) {
        rank = (int)blockIdx.x / BH;
        bh = (int)blockIdx.x - rank * BH;
    } else {
        grid_unit((int)blockIdx.x, BH, p.n_q, p.grp, rank, bh);
    }
    const int bb = bh / p.H, hh = bh - bb * p.H;
    const int qt = p.causal ? (p.n_q - 1 - rank) : rank;
    const int S = p.S;
    const int nj = p.causal ? min(qt + 1, p.n_kv) : p.n_kv;   // key tiles at or below the diagonal

    if (threadIdx.x == 0) {
        mbar_init(qd_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(kv_empty(s), 2);       // the S/dP issuer after dP_j, the dQ issuer after dQ_j
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 256);
        for (int b = 0; b < 2; ++b) {
            mbar_init(ds_full(b), 256);
            mbar_init(ds_free(b), 1);
            mbar_init(drain(b), 1);
        }
        mbar_init(dq_done, 1);
        *abort = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == SDP_WARP) {
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
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < 2; ++i) {
                prefetch_tmap(&p.tq[i]);
                prefetch_tmap(&p.tk[i]);
                prefetch_tmap(&p.tv[i]);
                prefetch_tmap(&p.tdo[i]);
            }
            griddep_wait();
            mbar_arrive_expect_tx(qd_full, 2 * G::TILE);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_4d(sb + G::Q_OFF + C::tile_off(c, BQ), &p.tq[C::map_index(c)], c * 64, qt * BQ, hh, bb,
                            qd_full);
                tma_load_4d(sb + G::DO_OFF + C::tile_off(c, BQ), &p.tdo[C::map_index(c)], c * 64, qt * BQ, hh, bb,
                            qd_full);
            }
            for (int j = 0; j < nj; ++j) {
                const int st = j % NS;
                const uint32_t ph = (j / NS) & 1;
                if (!mbar_wait(kv_empty(st), ph ^ 1, abort, p.status, WAIT_LIMIT_NS)) break;
                const uint32_t kdst = sb + G::RING_OFF + st * G::STAGE;
                mbar_arrive_expect_tx(k_full(st), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(kdst + C::tile_off(c, BK), &p.tk[C::map_index(c)], c * 64, j * BK, hh, bb, k_full(st));
                mbar_arrive_expect_tx(v_full(st), G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(kdst + G::TILE + C::tile_off(c, BK), &p.tv[C::map_index(c)], c * 64, j * BK, hh, bb,
                                v_full(st));
                issued = j + 1;
            }
            if (*abort) {
                // Let the copies already in flight land before the CTA exits.
                volatile int no_abort = 0;
                mbar_wait(qd_full, 0, &no_abort, p.status, WAIT_LIMIT_NS);
                for (int j = max(0, issued - NS); j < issued; ++j) {
                    mbar_wait(k_full(j % NS), (j / NS) & 1, &no_abort, p.status, WAIT_LIMIT_NS);
                    mbar_wait(v_full(j % NS), (j / NS) & 1, &no_abort, p.status, WAIT_LIMIT_NS);
                }
            }
        }
        __syncwarp();
    } else if (warp == SDP_WARP) {
        // ------------------------------------------------------------ S / dP issuer
        // Both issuer roles run on one thread each and wait on the barriers
        // themselves: a warp-collective operation between products stalls
        // the issuing path while the tensor pipe runs dry.
        if (lane == 0) {
        auto wait = [&](uint32_t bar, uint32_t parity) {
            return mbar_wait(bar, parity, abort, p.status, WAIT_LIMIT_NS);
        };
        const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0) | (p.neg_a << 13);
        const uint32_t idesc_dp = idesc_bf16(128, 128, 0, 0);
        const uint32_t q_lo = desc_lo(sb + G::Q_OFF, 16), do_lo = desc_lo(sb + G::DO_OFF, 16);
        const uint32_t k_lo0 = desc_lo(sb + G::RING_OFF, 16), v_lo0 = desc_lo(sb + G::RING_OFF + G::TILE, 16);
        bool ok = wait(qd_full, 0);
        for (int j = 0; j < nj && ok; ++j) {
            const int st = j % NS;
            const uint32_t ph = (j / NS) & 1;
            const uint32_t so = (uint32_t)st * (G::STAGE >> 4);
            if (!(ok = wait(k_full(st), ph))) break;
            // The dS warps have read S_{j-1} and dP_{j-1}.
            if (j > 0 && !(ok = wait(s_free, (j - 1) & 1))) break;
            tc_fence_after();
            mma_k_is_d<D>(tmem + TM_S, q_lo, k_lo0 + so, idesc_s);      // S = Q K_j^T
            if (!(ok = wait(v_full(st), ph))) break;
            tc_fence_after();
            mma_k_is_d<D>(tmem + TM_DP, do_lo, v_lo0 + so, idesc_dp);              // dP = dO V_j^T
            mma_commit(s_full);
            mma_commit(kv_empty(st));
        }
        if (*abort) {
            volatile int no_abort = 0;
            mma_commit(drain(0));
            mbar_wait(drain(0), 0, &no_abort, p.status, WAIT_LIMIT_NS);
        }
        }
        __syncwarp();
    } else if (warp == DQ_WARP) {
        // ------------------------------------------------------------ dQ issuer
        if (lane == 0) {
        auto wait = [&](uint32_t bar, uint32_t parity) {
            return mbar_wait(bar, parity, abort, p.status, WAIT_LIMIT_NS);
        };
        const uint32_t k_mn_lo0 = desc_lo(sb + G::RING_OFF, 128 * 128);
        bool ok = true;
        for (int j = 0; j < nj && ok; ++j) {
            const int st = j % NS;
            const int b = j & 1;
            const uint32_t so = (uint32_t)st * (G::STAGE >> 4);
            // K_j cannot be refilled before this issuer's own commit below, so
            // its k_full phase is still the one of tile j.
            if (!(ok = wait(k_full(st), (j / NS) & 1))) break;
            if (!(ok = wait(ds_full(b), (j >> 1) & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)                                    // dQ += dS K_j
                mma_n_is_d<D, true>(tmem + TM_DQ, tmem + TM_DS + 64u * b + 8u * ks, 0, k_mn_lo0 + so, ks, 0,
                                    (j > 0 || ks > 0) ? 1u : 0u);
            mma_commit(ds_free(b));
            mma_commit(kv_empty(st));
        }
        if (ok) mma_commit(dq_done);
        if (*abort) {
            volatile int no_abort = 0;
            mma_commit(drain(1));
            mbar_wait(drain(1), 0, &no_abort, p.status, WAIT_LIMIT_NS);
        }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ dS and the dq store
        const int h = warp >> 2;                       // keys [64h, 64h+64) of each tile
        const int wq = warp & 3;                       // lane quarter of Tensor Memory
        const int row_local = wq * 32 + lane;
        const int row = qt * BQ + row_local;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const size_t grow = (size_t)bh * S + row;
        griddep_wait();                                // L from the forward, D from the preprocess
        const float l2 = row < S ? p.lse[grow] * FA_LOG2E : INFINITY;   // P = 0 on rows past S
        const float dd = row < S ? p.Dvec[grow] : 0.f;
        const float c = p.c;
        const uint64_t c2 = f2pack(c, c);
        const uint64_t nl2 = f2pack(-l2, -l2);
        const uint64_t ndd = f2pack(-dd, -dd);
        const int key_lim = p.causal ? min(row, p.Sk - 1) : p.Sk - 1;
        bool ok = true;
        for (int j = 0; j < nj; ++j) {
            if (!(ok = warp_wait(s_full, j & 1, abort, p.status))) break;
            tc_fence_after();
            uint32_t rs[64], rp[64];
            tmem_ld32(tmem + lane_off + TM_S + 64 * h, rs);
            tmem_ld32(tmem + lane_off + TM_S + 64 * h + 32, rs + 32);
            tmem_ld32(tmem + lane_off + TM_DP + 64 * h, rp);
            tmem_ld32(tmem + lane_off + TM_DP + 64 * h + 32, rp + 32);
            tmem_wait_ld();
            reg_fence<64>(rs);
            reg_fence<64>(rp);
            tc_fence_before();
            mbar_arrive(s_free);                       // S, dP columns may take the next key tile
            const int kbase = j * BK + 64 * h;
            // Only the diagonal tile and a ragged last tile need the per-key mask.
            const bool masked = (p.causal && j == qt) || ((j + 1) * BK > p.Sk);
            uint32_t pk[32];
            // P = exp2(S c - L2), dS = P (dP - D) in f32x2 pairs.
            auto pair = [&](int e, bool mask) {
                float p0, p1;
                f2unpack(fma2(f2pack(__uint_as_float(rs[2 * e]), __uint_as_float(rs[2 * e + 1])), c2, nl2), p0, p1);
                p0 = ex2(p0);
                p1 = ex2(p1);
                if (mask) {
                    if (kbase + 2 * e > key_lim) p0 = 0.f;
                    if (kbase + 2 * e + 1 > key_lim) p1 = 0.f;
                }
                float d0, d1;
                f2unpack(mul2(f2pack(p0, p1),
                              add2(f2pack(__uint_as_float(rp[2 * e]), __uint_as_float(rp[2 * e + 1])), ndd)), d0, d1);
                pk[e] = pack_bf16(d0, d1);
            };
            if (masked) {
#pragma unroll
                for (int e = 0; e < 32; ++e) pair(e, true);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) pair(e, false);
            }
            const int b = j & 1;
            // dQ += dS_{j-2} K_{j-2} has read this buffer.
            if (j > 1) {
                if (!(ok = warp_wait(ds_free(b), ((j >> 1) - 1) & 1, abort, p.status))) break;
                tc_fence_after();
            }
            tmem_st32(tmem + lane_off + TM_DS + 64u * b + 32u * h, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_full(b));
        }
        if (ok && warp_wait(dq_done, 0, abort, p.status)) {
            tc_fence_after();
#pragma unroll
            for (int u = h; u < D / 16; u += 2) {
                uint32_t a[16];
                tmem_ld16(tmem + lane_off + TM_DQ + 16 * u, a);
                tmem_wait_ld();
                reg_fence<16>(a);
                uint32_t v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = pack_bf16(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
                if (row < S) {
                    uint4* dst = reinterpret_cast<uint4*>(p.dq + p.vdq.off(bb, hh, row) + 16 * u);
                    dst[0] = make_uint4(v[0], v[1], v[2], v[3]);
                    dst[1] = make_uint4(v[4], v[5], v[6], v[7]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == SDP_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D>
cudaError_t bwd_dq_tc_launch(const BwdArgs& a) {
    using C = Chunks<D>;
    using G = DqCfg<D>;
    DqParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    const void* src[4] = {a.q, a.k, a.v, a.dO};
    const int rows[4] = {a.S, a.Sk, a.Sk, a.S};
    const View views[4] = {a.vq, a.vk, a.vv, a.vdo};
    CUtensorMap* maps[4] = {p.tq, p.tk, p.tv, p.tdo};
    for (int i = 0; i < 4; ++i) {
        cudaError_t e;
        if (C::N64 > 0 &&
            (e = make_tmap_bf16_4d(&maps[i][0], src[i], D, rows[i], a.H, a.B, views[i], 64, 128)) != cudaSuccess)
            return e;
        if (C::REM > 0 && !C::PAD &&
            (e = make_tmap_bf16_4d(&maps[i][1], src[i], D, rows[i], a.H, a.B, views[i], C::REM, 128)) != cudaSuccess)
            return e;
    }
    p.lse = a.lse;
    p.Dvec = a.Dvec;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.status = a.status;
    p.vdq = a.vdq;
    p.H = a.H;
    p.S = a.S;
    p.Sk = a.Sk;
    p.n_q = (a.S + BQ - 1) / BQ;
    p.n_kv = (a.Sk + BK - 1) / BK;
    // Each CTA streams its head's K and V (bf16).  Grouped from 128 MiB: at
    // B4 H32 S4096 d80 (160 MiB of K and V) grouping took this pass from 663
    // to 622 us.  As for the forward, which walks K and V the same way, only
    // with many heads.
    p.grp = head_group(a.B * a.H, p.n_q, 4.0 * a.Sk * D, 128.0, true);
    p.causal = a.causal;
    const float c = fabsf(a.scale) * FA_LOG2E;
    p.c = c < 1e-30f ? 1e-30f : c;
    p.scale = a.scale;
    p.neg_a = a.scale < 0.f ? 1u : 0u;
    auto kern = bwd_dq_tc_kernel<D>;
    cudaError_t e = set_smem_limit<bwd_dq_tc_kernel<D>>(G::DYN_SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.n_q * BH), dim3(NTHREADS), G::DYN_SMEM, a.stream, p);
}

}  // namespace

cudaError_t launch_bwd_dq_tc(const BwdArgs& a) {
    switch (a.d) {
        case 16: return bwd_dq_tc_launch<16>(a);
        case 32: return bwd_dq_tc_launch<32>(a);
        case 64: return bwd_dq_tc_launch<64>(a);
        case 80: return bwd_dq_tc_launch<80>(a);
        case 96: return bwd_dq_tc_launch<96>(a);
        case 128: return bwd_dq_tc_launch<128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
