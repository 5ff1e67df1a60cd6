// fa_bwd_tc.cu - bf16 FlashAttention-2 backward on the sm_103a tensor cores.
//
// "Stanford CS336 Assignment 2 (Systems)" handout, section 4: Eq. 13-19 with
// the key-tile-outer loop of Algorithm 2.  One CTA owns a 128-key tile of one
// (batch, head) and keeps its dK and dV accumulators in Tensor Memory while it
// walks over the 128-row query tiles at or below the diagonal.  For each
// query tile i (all products on tcgen05, fp32 accumulation):
//   S^T  = K Q_i^T                 (key-major scores, Eq. 13)
//   dP^T = V dO_i^T                (Eq. 16)
//   P^T  = exp2(S^T c - L_i log2 e),  dS^T = P^T * (dP^T - D_i)   (Eq. 14, 17)
//   dV  += P^T dO_i                (Eq. 15; P^T read from Tensor Memory)
//   dK  += dS^T Q_i                (Eq. 19; dS^T from shared memory)
//   dQ_i = dS K                    (Eq. 18; the same shared-memory dS^T tile
//                                   read as an M-major operand)
// dQ_i leaves Tensor Memory through a separate warpgroup: it stages the fp32
// tile in shared memory (for d > 64 in the slot of Q_i / dO_i, which the
// products no longer need; for d = 64 in a buffer of its own, 32 columns at a
// time) and adds it into the fp32 dQ accumulator with TMA bulk
// reduce-adds, whole 128-byte lines at a time (the stated dQ strategy: atomic
// accumulation across key tiles).  The scale of Eq. 18 is applied when the
// accumulator is converted, that of Eq. 19 when dK is written.
//
// Warp roles: warps 0-7 P^T and dS^T (one thread per key row; warps 0-3 take
// query columns 0-63, warps 4-7 columns 64-127) and the final dK/dV store,
// warps 8-11 the dQ read-out (one thread per query row), warp 12 TMA (K, V
// once; Q_i, dO_i per tile, plus L and D), warp 13 Tensor Memory allocation
// and one thread that issues the products (for d = 64 it issues S^T and dP^T
// only, and a thread of warp 14 issues dV, dK and dQ_i).
// Tensor Memory columns: dV [0,128), dK [128,256), S^T/P^T [256,384),
// dP^T [384,512), which dQ_i reuses once dS^T has been formed.  With this
// layout (d > 64) the products of tile i are issued as S^T; dP^T once dQ_{i-1}
// has been read out; dV once P^T is in; dK and dQ_i once dS^T is in.
// Shapes: N_q queries and N_k keys (Algorithm 2's Q in R^{N_q x d}, K, V in
// R^{N_k x d}), causal keeping key j for query i when j <= i; every
// [B, H, rows, d] operand is a view with strides that are multiples of 8
// elements (4-D TMA maps); L, D and the dQ accumulator are contiguous.

#include "fa_common.cuh"
#include "fa_launch.h"
#include "fa_tmap.h"
#include "sm103_ptx.cuh"
#include "fa_tc_common.cuh"

#include <cstring>
#include <type_traits>

namespace fa {
namespace {

using namespace sm103;
using namespace tc;

constexpr int BK = 128;
constexpr int BQ = 128;

constexpr int DQ_WARP0 = 8;
constexpr int TMA_WARP = 12;
constexpr int MMA_WARP = 13;
constexpr int MMA_WARP2 = 14;      // d = 64: second issuer (dV, dK, dQ_i)
// Threads per CTA: 14 warps, plus warp MMA_WARP2 where it issues (d = 64).
template <int D>
constexpr int bwd_threads() { return (D > 32 && D <= 64) ? 480 : 448; }
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 256, TM_DP = 384;
constexpr int SMEM_BUDGET = 227 * 1024;

// Tensor Memory columns.  For d <= 64 every product has its own columns
// (dV, dK, dQ_i, the bf16 P^T pairs, S^T, dP^T): S^T and dP^T of the next
// query tile are computed while the softmax warps still work on this one, and
// the dV/dK/dQ products of this tile run while they work on the next.  For
// larger d the accumulators leave no room: P^T overwrites S^T, dQ_i reuses
// dP^T, and the products of consecutive tiles follow each other.
template <int D>
struct BwdTm {
    static constexpr bool PIPE = D <= 64;
    // d <= 32: dQ_i is issued by a second thread (in the dQ read-out warps);
    // its products are the cheapest, so one issuing thread limits the most.
    static constexpr bool SPLIT_DQ = D <= 32;
    // d = 64: dQ_i is staged for the reduce-add in a 16 KB buffer of its own,
    // one 32-column chunk at a time, so that the Q_i / dO_i slot is free as
    // soon as dK has read it (the reduce-add reads ~20 bytes per clock: a
    // slot held until then kept the next loads, and so the next S^T, waiting).
    static constexpr bool DQSTAGE = PIPE && !SPLIT_DQ;
    static constexpr uint32_t DV = 0;
    static constexpr uint32_t DK = PIPE ? 64 : 128;
    static constexpr uint32_t DQ = PIPE ? 128 : TM_DP;
    static constexpr uint32_t P = PIPE ? 192 : TM_S;
    // Column of P^T for query columns [64h + 32qh, 64h + 32qh + 32) (16 pairs).
    __device__ static constexpr uint32_t p_col(int h, int qh) { return PIPE ? P + 32 * h + 16 * qh : P + 64 * h + 16 * qh; }
    // A operand (16 queries) of k-step ks of dV += P^T dO.
    __device__ static constexpr uint32_t p_kstep(int ks) { return PIPE ? P + 8 * ks : P + (ks / 4) * 64 + (ks % 4) * 8; }
};

// Head-dim layout of the K, V, Q, dO tiles.  64-column chunks pad d = 80 and
// 96 to 128 columns: the tensor cores then read (and the TMA writes) a
// 64-column remainder box for 16 or 32 columns.  d = 80 uses unpadded
// 16-column chunks instead: 20 KB tiles leave room for three [Q_i | dO_i]
// stages instead of two (each slot still takes the staged fp32 dQ_i, 40 KB).
// d = 96 uses unpadded 32-column chunks (24 KB tiles, still two stages;
// 16-column chunks of the same size measured slower).
template <int D>
using BwdChunks = std::conditional_t<D == 80, ChunksW<D, 16>, std::conditional_t<D == 96, ChunksW<D, 32>, Chunks<D>>>;

template <int D>
struct BwdCfg {
    static constexpr int TILE = BwdChunks<D>::tile_bytes(128);
    static constexpr int DS_BYTES = BK * BQ * 2;
    static constexpr int NDS = BwdTm<D>::PIPE ? 2 : 1;      // dS^T buffers
    static constexpr int LD_BYTES = BQ * 8;            // (L * log2 e, D) per query row
    static constexpr int DQS_BYTES = BwdTm<D>::DQSTAGE ? BQ * 32 * 4 : 0;   // one fp32 dQ_i chunk
    static constexpr int FIXED = 2 * TILE + NDS * DS_BYTES + DQS_BYTES;  // K, V, dS^T, dQ_i staging
    static constexpr int STAGE = 2 * TILE + LD_BYTES;  // [Q_i | dO_i], (L, D)_i
    static constexpr int NS_RAW = (SMEM_BUDGET - FIXED - 256) / STAGE;
    static constexpr int NS = NS_RAW > 3 ? 3 : NS_RAW;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = TILE;
    static constexpr int DS_OFF = 2 * TILE;
    static constexpr int QD_OFF = DS_OFF + NDS * DS_BYTES;   // stage s: Q at QD_OFF + 2*TILE*s, dO right after
    static constexpr int LD_OFF = QD_OFF + NS * 2 * TILE;
    static constexpr int DQS_OFF = LD_OFF + NS * LD_BYTES;   // 1024-byte aligned (128-byte swizzle)
    static constexpr int BAR_OFF = DQS_OFF + DQS_BYTES;
    // kv_full, q_full[NS], q_empty[NS], s_full, p_full, dq_full, dq_empty, stg, done, drain,
    // s_free, p_free, ds_free[2], drain_dq, dp_full, dst_full, stg_free
    static constexpr int NBARS = 16 + 2 * NS;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static constexpr int DYN_SMEM = (BYTES + 1024) <= SMEM_BUDGET ? (BYTES + 1024) : BYTES;
    static_assert(NS >= 2, "Q/dO ring needs two stages");
    static_assert(BYTES <= SMEM_BUDGET, "shared memory budget");
    static_assert(!BwdTm<D>::PIPE || BQ * D * 4 <= DS_BYTES, "fp32 dQ tile staged in a dS^T buffer");
};

// fp32 dQ tile [128 rows][d] staged for TMA as 32-column boxes (128-byte
// rows, 128-byte swizzle) plus one 16-column box (64-byte rows, 64-byte
// swizzle) when d is not a multiple of 32.  For d > 64 it is staged in the
// Q_i + dO_i slot (2 x 32 KB tiles for d = 128, 2 x 24 KB for d = 96,
// 2 x 20 KB for d = 80), for d <= 64 in the slot or in a dS^T buffer.
template <int D>
struct DqChunks {
    static constexpr int N32 = D / 32;
    static constexpr int NCH = N32 + (D % 32 ? 1 : 0);
    __host__ __device__ static constexpr int width(int c) { return c < N32 ? 32 : 16; }
    __host__ __device__ static constexpr int map_index(int c) { return c < N32 ? 0 : 1; }
    __host__ __device__ static constexpr int offset(int c) { return c * 128 * 128; }
    static constexpr int SPAN = offset(NCH - 1) + 128 * width(NCH - 1) * 4;
    static_assert(SPAN <= 2 * BwdCfg<D>::TILE, "staged dQ tile fits a Q_i + dO_i slot");
};

struct BwdParams {
    CUtensorMap tq[2];
    CUtensorMap tk[2];
    CUtensorMap tv[2];
    CUtensorMap tdo[2];
    CUtensorMap tdq[2];
    const float* lse;     // contiguous [B*H, S]
    const float* Dvec;    // contiguous [B*H, S]
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    unsigned int* status;
    View vdk, vdv;        // element strides of dk, dv
    uint32_t map3;        // bit i: map i of (q, k, v, dO) is 3-D over (col, row, b*H + h)
    int H;
    int grp;              // heads per group of the grid order
    int S;                // query rows N_q
    int Sk;               // key rows N_k
    int n_q;
    int n_kv;
    int causal;
    float c;          // |scale| * log2(e), at least 1e-30
    float scale;      // signed scale applied to dK
    uint32_t neg_a;   // 1 when scale < 0: S^T = -(K Q^T) so that exp uses |scale|
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// WITH_DQ = false: dK and dV only (the deterministic backward computes dQ in
// a separate query-tile-outer pass); the dQ warps then stay idle and the
// buffers the dQ read-out would release are released by the MMA issuer.
template <int D, bool WITH_DQ>
__global__ void __launch_bounds__(bwd_threads<D>(), 1) bwd_tc_kernel(const __grid_constant__ BwdParams p) {
    using C = BwdChunks<D>;
    using QC = DqChunks<D>;
    using G = BwdCfg<D>;
    constexpr int NS = G::NS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (smem + G::BYTES > smem_raw + G::DYN_SMEM) {
        // The dynamic shared window is not 1024-byte aligned and has no room to
        // align it: report and leave before touching any barrier or TMEM.
        if (threadIdx.x == 0) set_status(p.status, FA_DEV_STATUS_BOUNDS);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + G::BAR_OFF;
    const uint32_t kv_full = bar0;
    auto q_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto q_empty = [&](int s) { return bar0 + 8u * (1 + NS + s); };
    const uint32_t s_full = bar0 + 8u * (1 + 2 * NS);
    const uint32_t p_full = s_full + 8;
    const uint32_t dq_full = s_full + 16;
    const uint32_t dq_empty = s_full + 24;
    const uint32_t stg = s_full + 32;
    const uint32_t done = s_full + 40;
    const uint32_t drain = s_full + 48;
    const uint32_t s_free = s_full + 56;      // S^T and dP^T have been read (pipelined schedule)
    const uint32_t p_free = s_full + 64;      // dV has read P^T
    auto ds_free = [&](int b) { return s_full + 72u + 8u * b; };   // dS^T buffer b (holding the staged dQ) is free
    const uint32_t drain_dq = s_full + 88;    // the dQ issuer's products have finished (abort only)
    const uint32_t dp_full = s_full + 96;     // d > 64: dP^T is in Tensor Memory (s_full: S^T alone)
    const uint32_t dst_full = s_full + 104;   // d > 64: dS^T is in shared memory (p_full: P^T alone)
    const uint32_t stg_free = s_full + 112;   // d = 64: the reduce-add has read the dQ_i staging buffer
    using TM = BwdTm<D>;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::MISC_OFF);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + G::MISC_OFF + 4);
    auto q_slot = [&](int s) { return sb + G::QD_OFF + (uint32_t)(s * 2 * G::TILE); };
    auto do_slot = [&](int s) { return sb + G::QD_OFF + (uint32_t)(s * 2 * G::TILE + G::TILE); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // One flat grid ordered key-tile-major: early key tiles see the most query
    // tiles under the causal mask, so every head's heaviest tile goes first
    // (within head groups when the heads' tiles would not stay in L2 together).
    const int BH = (int)(gridDim.x / (unsigned)p.n_kv);
    int j, bh;
    if (p.grp >= BH) {
        j = (int)blockIdx.x / BH;
        bh = (int)blockIdx.x - j * BH;
    } else {
        grid_unit((int)blockIdx.x, BH, p.n_kv, p.grp, j, bh);
    }
    const int bb = bh / p.H, hh = bh - bb * p.H;
    const int S = p.S;
    const int k0 = j * BK;
    const int i0 = p.causal ? j : 0;          // query tiles above the diagonal are fully masked
    const int n_it = p.n_q - i0;              // >= 1: the grid holds no key tile past the last query tile

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(q_full(s), 33);        // TMA expect-tx arrival + 32 lanes that stage (L, D)
            // The slot is free once its last readers are done: dV and dK (the
            // MMA issuer's commit; d <= 64 and the dK/dV-only backward) or, for
            // d > 64, where dQ_i is staged in it, the dQ reduce-add's read
            // (dQ_i follows dK on the same issuer).
            mbar_init(q_empty(s), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, 2 * BK);
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, BQ);
        mbar_init(stg, BQ);
        mbar_init(done, 1);
        mbar_init(drain, 1);
        mbar_init(s_free, 2 * BK);
        mbar_init(p_free, 1);
        mbar_init(ds_free(0), 1);
        mbar_init(ds_free(1), 1);
        mbar_init(drain_dq, 1);
        mbar_init(dp_full, 1);
        mbar_init(dst_full, 2 * BK);
        mbar_init(stg_free, 1);
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
        int issued = 0;
        if (lane == 0) {
            for (int i = 0; i < 2; ++i) {
                prefetch_tmap(&p.tq[i]);
                prefetch_tmap(&p.tk[i]);
                prefetch_tmap(&p.tv[i]);
                prefetch_tmap(&p.tdo[i]);
            }
            mbar_arrive_expect_tx(kv_full, 2 * G::TILE);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_view(sb + G::K_OFF + C::tile_off(c, BK), &p.tk[C::map_index(c)], p.map3 & 2u, C::col(c), k0,
                              hh, bb, bh, kv_full);
                tma_load_view(sb + G::V_OFF + C::tile_off(c, BK), &p.tv[C::map_index(c)], p.map3 & 4u, C::col(c), k0,
                              hh, bb, bh, kv_full);
            }
        }
        const size_t rb = (size_t)bh * S;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % NS;
            const uint32_t ph = (it / NS) & 1;
            const int q0 = (i0 + it) * BQ;
            // (-L * log2 e, -D) for the 128 query rows, loaded before the
            // stage is free so that the loads overlap the wait; rows past S
            // get (-inf, 0) so that P = 0.  D (and the zeroed dQ
            // accumulator) come from the previous kernel.
            if (it == 0) griddep_wait();
            float l2[BQ / 32], dd[BQ / 32];
#pragma unroll
            for (int e = 0; e < BQ / 32; ++e) {
                const int q = q0 + e * 32 + lane;
                l2[e] = q < S ? -p.lse[rb + q] * FA_LOG2E : -INFINITY;
                dd[e] = q < S ? -p.Dvec[rb + q] : 0.f;
            }
            if (!warp_wait(q_empty(s), ph ^ 1, abort, p.status)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full(s), 2 * G::TILE);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_view(q_slot(s) + C::tile_off(c, BQ), &p.tq[C::map_index(c)], p.map3 & 1u, C::col(c), q0,
                                  hh, bb, bh, q_full(s));
                    tma_load_view(do_slot(s) + C::tile_off(c, BQ), &p.tdo[C::map_index(c)], p.map3 & 8u, C::col(c), q0,
                                  hh, bb, bh, q_full(s));
                }
            }
            // Stored per pair of rows (2r, 2r+1) as (-L2_2r, -L2_2r+1, -D_2r,
            // -D_2r+1), the operand pairs of the packed f32x2 arithmetic.
#pragma unroll
            for (int e = 0; e < BQ / 32; ++e) {
                const int r = e * 32 + lane;
                const uint32_t a = sb + G::LD_OFF + s * G::LD_BYTES + (r >> 1) * 16 + (r & 1) * 4;
                asm volatile("st.shared.f32 [%0], %1;" :: "r"(a), "f"(l2[e]) : "memory");
                asm volatile("st.shared.f32 [%0], %1;" :: "r"(a + 8), "f"(dd[e]) : "memory");
            }
            mbar_arrive(q_full(s));
            issued = it + 1;
        }
        if (*abort && lane == 0) {
            volatile int no_abort = 0;
            mbar_wait(kv_full, 0, &no_abort, p.status, WAIT_LIMIT_NS);
            for (int it = max(0, issued - NS); it < issued; ++it)
                mbar_wait(q_full(it % NS), (it / NS) & 1, &no_abort, p.status, WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else if (warp == MMA_WARP || warp == MMA_WARP2) {
        // ------------------------------------------------------------ MMA issuers
        // One thread runs this role from start to end, waiting on the
        // barriers itself: no warp-collective operation between products
        // (a shuffle or warp sync per wait measured ~300 cycles each on the
        // issuing path, about as long as the products queued ahead of it).
        constexpr bool TWO = TM::PIPE && !TM::SPLIT_DQ;
        if (lane == 0 && (warp == MMA_WARP || TWO)) {
        auto wait = [&](uint32_t bar, uint32_t parity) {
            return mbar_wait(bar, parity, abort, p.status, WAIT_LIMIT_NS);
        };
        const uint32_t idesc_s = idesc_bf16(128, 128, 0, 0) | (p.neg_a << 13);
        const uint32_t idesc_dp = idesc_bf16(128, 128, 0, 0);
        // Low descriptor words: K-major operands use LBO 16, the MN-major
        // [rows][d] tiles use the head-dim chunk stride as LBO.
        constexpr uint32_t CH = C::tile_off(1, 128);
        const uint32_t k_lo = desc_lo(sb + G::K_OFF, 16), v_lo = desc_lo(sb + G::V_OFF, 16);
        const uint32_t k_mn_lo = desc_lo(sb + G::K_OFF, CH);
        const uint32_t q_lo0 = desc_lo(sb + G::QD_OFF, 16), do_lo0 = desc_lo(sb + G::QD_OFF + G::TILE, 16);
        const uint32_t q_mn_lo0 = desc_lo(sb + G::QD_OFF, CH);
        const uint32_t do_mn_lo0 = desc_lo(sb + G::QD_OFF + G::TILE, CH);
        const uint32_t ds_k_lo = desc_lo(sb + G::DS_OFF, 16);          // dS^T as K-major A (dK)
        const uint32_t ds_m_lo = desc_lo(sb + G::DS_OFF, 16384);       // dS as M-major A (dQ)
        const uint32_t ds_hi = desc_hi(1024, SW_128B);
        bool ok = wait(kv_full, 0);
        if constexpr (TM::PIPE) {
            // S^T, dP^T of tile it+1 go in as soon as the softmax warps have
            // read those of tile it; dV, dK, dQ of tile it once P^T, dS^T exist.
            auto issue_sdp = [&](int it) {
                const uint32_t so = (uint32_t)(it % NS) * ((2 * G::TILE) >> 4);
                mma_k_is_d<D, C>(tmem + TM_S, k_lo, q_lo0 + so, idesc_s);                  // S^T = K Q^T
                mma_k_is_d<D, C>(tmem + TM_DP, v_lo, do_lo0 + so, idesc_dp);               // dP^T = V dO^T
                mma_commit(s_full);
            };
            // d = 64: S^T, dP^T on this thread (warp MMA_WARP), dV, dK, dQ_i on
            // warp MMA_WARP2's: the next scores go in as soon as the softmax
            // has read these, whatever the other products are waiting for.
            const bool do_sdp = !TWO || warp == MMA_WARP;
            const bool do_rest = !TWO || warp == MMA_WARP2;
            if (do_sdp) {
                if (ok) ok = wait(q_full(0), 0);
                if (ok) {
                    tc_fence_after();
                    issue_sdp(0);
                }
            }
            for (int it = 0; it < n_it && ok; ++it) {
                const uint32_t so = (uint32_t)(it % NS) * ((2 * G::TILE) >> 4);
                const uint32_t dso = (uint32_t)((it & 1) * G::DS_BYTES) >> 4;
                if (do_sdp && it + 1 < n_it) {
                    if (!(ok = wait(q_full((it + 1) % NS), ((it + 1) / NS) & 1))) break;
                    if (!(ok = wait(s_free, it & 1))) break;
                    tc_fence_after();
                    issue_sdp(it + 1);
                }
                if (!do_rest) continue;
                if (!(ok = wait(p_full, it & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks)                                  // dV += P^T dO
                    mma_n_is_d<D, true, C>(tmem + TM::DV, tmem + TM::p_kstep(ks), 0, do_mn_lo0 + so, ks, 0,
                                        (it > 0 || ks > 0) ? 1u : 0u);
                mma_commit(p_free);
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks) {                                  // dK += dS^T Q
                    const uint64_t adesc =
                        desc_make(ds_k_lo + dso + (((ks / 4) * 16384 + (ks % 4) * 32) >> 4), ds_hi);
                    mma_n_is_d<D, false, C>(tmem + TM::DK, 0, adesc, q_mn_lo0 + so, ks, 0,
                                         (it > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(q_empty(it % NS));       // Q_i, dO_i (and L, D) are no longer read
                if constexpr (!WITH_DQ) mma_commit(ds_free(it & 1));   // dK has read dS^T
                // (d <= 32: dQ_i = dS K is issued by a thread of the dQ read-out warps.)
                if constexpr (!WITH_DQ || TM::SPLIT_DQ) continue;
                if (it > 0 && !(ok = wait(dq_empty, (it - 1) & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < BK / 16; ++ks) {                                  // dQ_i = dS K
                    const uint64_t adesc = desc_make(ds_m_lo + dso + ks * 128, ds_hi);
                    mma_n_is_d<D, false, C>(tmem + TM::DQ, 0, adesc, k_mn_lo, ks, 1, ks > 0 ? 1u : 0u);
                }
                mma_commit(dq_full);
                mma_commit(ds_free(it & 1));        // dK and dQ_i have read dS^T
            }
        }
        if constexpr (!TM::PIPE) {
            // d > 64: dV of tile it goes in as soon as P^T is in Tensor
            // Memory, so it runs while dS^T is formed; dK and dQ_i follow
            // dS^T, and S^T of tile it+1 follows them into the columns that
            // held P^T (one thread's products run in issue order).  dP^T of
            // tile it+1 waits for the read-out of dQ_i, which shares its
            // columns; its commit also covers dK and dQ_i, which have then
            // read the one dS^T buffer.
            auto issue_s = [&](int it) {
                const uint32_t so = (uint32_t)(it % NS) * ((2 * G::TILE) >> 4);
                mma_k_is_d<D, C>(tmem + TM_S, k_lo, q_lo0 + so, idesc_s);                  // S^T = K Q^T
                mma_commit(s_full);
            };
            if (ok) ok = wait(q_full(0), 0);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int it = 0; it < n_it && ok; ++it) {
                const int s = it % NS;
                const uint32_t so = (uint32_t)s * ((2 * G::TILE) >> 4);
                if (WITH_DQ && it > 0 && !(ok = wait(dq_empty, (it - 1) & 1))) break;
                tc_fence_after();
                mma_k_is_d<D, C>(tmem + TM_DP, v_lo, do_lo0 + so, idesc_dp);                 // dP^T = V dO^T
                mma_commit(dp_full);
                if (!(ok = wait(p_full, it & 1))) break;
                tc_fence_after();
                // dV += P^T dO: P^T of query columns 64h.. sits at TMEM columns 64h.. of S^T.
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks)
                    mma_n_is_d<D, true, C>(tmem + TM::DV, tmem + TM::p_kstep(ks), 0, do_mn_lo0 + so,
                                        ks, 0, (it > 0 || ks > 0) ? 1u : 0u);
                if (!(ok = wait(dst_full, it & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < BQ / 16; ++ks) {                                      // dK += dS^T Q
                    const uint64_t adesc = desc_make(ds_k_lo + (((ks / 4) * 16384 + (ks % 4) * 32) >> 4), ds_hi);
                    mma_n_is_d<D, false, C>(tmem + TM::DK, 0, adesc, q_mn_lo0 + so, ks, 0, (it > 0 || ks > 0) ? 1u : 0u);
                }
                if constexpr (WITH_DQ) {
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {                                  // dQ_i = dS K
                        const uint64_t adesc = desc_make(ds_m_lo + ks * 128, ds_hi);
                        mma_n_is_d<D, false, C>(tmem + TM::DQ, 0, adesc, k_mn_lo, ks, 1, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(dq_full);
                } else {
                    mma_commit(q_empty(s));         // Q_i, dO_i (and L, D) are no longer read
                }
                if (it + 1 < n_it) {
                    if (!(ok = wait(q_full((it + 1) % NS), ((it + 1) / NS) & 1))) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
            }
        }
        if (ok && (!TWO || warp == MMA_WARP2)) mma_commit(done);
        if (*abort) {
            // Every product this thread issued has finished before TMEM is freed.
            volatile int no_abort = 0;
            const uint32_t dr = warp == MMA_WARP ? drain : drain_dq;
            mma_commit(dr);
            mbar_wait(dr, 0, &no_abort, p.status, WAIT_LIMIT_NS);
        }
        }
        __syncwarp();
    } else if (warp < DQ_WARP0) {
        // ------------------------------------------------------------ P^T, dS^T and the dK/dV store
        const int h = warp >> 2;                       // query columns [64h, 64h+64)
        const int wq = warp & 3;
        const int jr = wq * 32 + lane;                 // key row inside the tile
        const int key = k0 + jr;
        const bool key_ok = key < p.Sk;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + TM_S;
        const uint32_t tP = tmem + lane_off + TM_DP;
        const float c = p.c;
        const uint64_t c2 = f2pack(c, c);
        const uint32_t ds_row = sb + G::DS_OFF + jr * 128;
        const uint32_t swz = (uint32_t)(jr & 7);
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % NS;
            const uint32_t ph = (it / NS) & 1;
            const bool diag = p.causal && (i0 + it) == j;
            if (!(ok = warp_wait(q_full(s), ph, abort, p.status))) break;
            if (!(ok = warp_wait(s_full, it & 1, abort, p.status))) break;
            tc_fence_after();
            const uint32_t ldb = sb + G::LD_OFF + s * G::LD_BYTES;
            // dS^T row, queries 32qq..32qq+31 (dsp: 16 bf16 pairs): four
            // 16-byte units of the 128-byte-swizzled [key][query] tile (two
            // 64-query chunks).
            auto store_ds = [&](int qh, const uint32_t* dsp) {
                const uint32_t chunk = ds_row + (uint32_t)((it & 1) * (G::NDS - 1) * G::DS_BYTES) + (uint32_t)h * 16384;
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) {
                    const uint32_t u = (uint32_t)(qh * 4 + u4);
                    st_shared_v4(chunk + ((u ^ swz) << 4), dsp[4 * u4], dsp[4 * u4 + 1], dsp[4 * u4 + 2], dsp[4 * u4 + 3]);
                }
            };
            if constexpr (TM::PIPE) {
                // Four 16-query groups; the Tensor Memory loads of group g+1
                // are in flight while group g is computed.
                uint32_t bs[2][16], bp[2][16];
                uint32_t pk[16], dsp[16];
                tmem_ld16(tS + 64 * h, bs[0]);
                tmem_ld16(tP + 64 * h, bp[0]);
                tmem_wait_ld();
                reg_fence<16>(bs[0]);
                reg_fence<16>(bp[0]);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int cur = g & 1;
                    if (g < 3) {
                        tmem_ld16(tS + 64 * h + 16 * (g + 1), bs[cur ^ 1]);
                        tmem_ld16(tP + 64 * h + 16 * (g + 1), bp[cur ^ 1]);
                    }
                    // P = exp2(S c - L2) and dS = P (dP - D) in f32x2 pairs; only
                    // the diagonal tile and a ragged key tile need the mask.
                    auto pair = [&](int e, bool mask) {
                        const int q = 64 * h + 16 * g + 2 * e;                   // query column inside the tile
                        const float4 ld = ld_shared_f4(ldb + q * 8);           // (-L2, -D) of q and q+1
                        float p0, p1;
                        f2unpack(fma2(f2pack(__uint_as_float(bs[cur][2 * e]), __uint_as_float(bs[cur][2 * e + 1])), c2,
                                      f2pack(ld.x, ld.y)), p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        if (mask) {
                            if (!key_ok || (diag && q < jr)) p0 = 0.f;
                            if (!key_ok || (diag && q + 1 < jr)) p1 = 0.f;
                        }
                        const uint64_t p2 = f2pack(p0, p1);
                        float d0, d1;
                        f2unpack(mul2(p2, add2(f2pack(__uint_as_float(bp[cur][2 * e]), __uint_as_float(bp[cur][2 * e + 1])),
                                               f2pack(ld.z, ld.w))), d0, d1);
                        pk[8 * cur + e] = pack_bf16(p0, p1);
                        dsp[8 * cur + e] = pack_bf16(d0, d1);
                    };
                    if (diag || !key_ok) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) pair(e, true);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) pair(e, false);
                    }
                    if (g < 3) {
                        tmem_wait_ld();
                        reg_fence<16>(bs[cur ^ 1]);
                        reg_fence<16>(bp[cur ^ 1]);
                    }
                    if (g == 2) {
                        tc_fence_before();
                        mbar_arrive(s_free);                       // S^T / dP^T columns may take the next tile
                    }
                    if (cur == 1) {
                        const int qh = g >> 1;
                        if (qh == 0) {
                            // P^T and dS^T buffers of earlier tiles must have been read.
                            if (it > 0 && !(ok = warp_wait(p_free, (it - 1) & 1, abort, p.status))) break;
                            if (it > 1 && !(ok = warp_wait(ds_free(it & 1), ((it >> 1) - 1) & 1, abort, p.status))) break;
                            tc_fence_after();
                        }
                        // P^T of these 32 queries: 16 columns of bf16 pairs.
                        tmem_st16(tmem + lane_off + TM::p_col(h, qh), pk);
                        store_ds(qh, dsp);
                    }
                }
            } else {
                // d > 64, in two phases: P^T from S^T (the exponentials) as soon
                // as S^T is in, while dP^T waits for the previous dQ_i's
                // columns; p_full then lets dV read P^T while dS^T is formed
                // once dP^T is in.  P stays in fp32 registers between the phases.
                float pf[2][32];
                auto p_of = [&](int qq, const uint32_t* rs, float* pv, bool mask) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int q = 32 * qq + 2 * e;
                        const float4 ld = ld_shared_f4(ldb + q * 8);       // (-L2, -D) of q and q+1
                        float p0, p1;
                        f2unpack(fma2(f2pack(__uint_as_float(rs[2 * e]), __uint_as_float(rs[2 * e + 1])), c2,
                                      f2pack(ld.x, ld.y)), p0, p1);
                        p0 = ex2(p0);
                        p1 = ex2(p1);
                        if (mask) {
                            if (!key_ok || (diag && q < jr)) p0 = 0.f;
                            if (!key_ok || (diag && q + 1 < jr)) p1 = 0.f;
                        }
                        pv[2 * e] = p0;
                        pv[2 * e + 1] = p1;
                    }
                };
#pragma unroll
                for (int qh = 0; qh < 2; ++qh) {
                    const int qq = 2 * h + qh;
                    uint32_t rs[32];
                    tmem_ld32(tS + 32 * qq, rs);
                    tmem_wait_ld();
                    reg_fence<32>(rs);
                    if (diag || !key_ok) p_of(qq, rs, pf[qh], true);
                    else p_of(qq, rs, pf[qh], false);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(pf[qh][2 * e], pf[qh][2 * e + 1]);
                    // P^T of these 32 queries inside this half's own, already
                    // read, score columns.
                    tmem_st16(tmem + lane_off + TM::p_col(h, qh), pk);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_full);                                    // dV may read P^T
                if (!(ok = warp_wait(dp_full, it & 1, abort, p.status))) break;
                tc_fence_after();
#pragma unroll
                for (int qh = 0; qh < 2; ++qh) {
                    const int qq = 2 * h + qh;
                    uint32_t rp[32];
                    tmem_ld32(tP + 32 * qq, rp);
                    tmem_wait_ld();
                    reg_fence<32>(rp);
                    uint32_t dsp[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float4 ld = ld_shared_f4(ldb + (32 * qq + 2 * e) * 8);
                        float d0, d1;
                        f2unpack(mul2(f2pack(pf[qh][2 * e], pf[qh][2 * e + 1]),
                                      add2(f2pack(__uint_as_float(rp[2 * e]), __uint_as_float(rp[2 * e + 1])),
                                           f2pack(ld.z, ld.w))), d0, d1);
                        dsp[e] = pack_bf16(d0, d1);
                    }
                    store_ds(qh, dsp);
                }
            }
            if (!ok) break;
            if constexpr (TM::PIPE) {
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
            } else {
                fence_proxy_async_smem();
                tc_fence_before();                     // dP^T has been read: dQ_i may take its columns
                mbar_arrive(dst_full);
            }
        }
        // dK, dV rows of this key tile (16-column units split between the halves).
        if (ok && warp_wait(done, 0, abort, p.status)) {
            tc_fence_after();
#pragma unroll
            for (int u = h; u < D / 16; u += 2) {
                uint32_t a[16], b[16];
                tmem_ld16(tmem + lane_off + TM::DV + 16 * u, a);
                tmem_ld16(tmem + lane_off + TM::DK + 16 * u, b);
                tmem_wait_ld();
                reg_fence<16>(a);
                reg_fence<16>(b);
                uint32_t va[8], vb[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    va[e] = pack_bf16(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                    vb[e] = pack_bf16(__uint_as_float(b[2 * e]) * p.scale, __uint_as_float(b[2 * e + 1]) * p.scale);
                }
                if (key_ok) {
                    uint4* dvp = reinterpret_cast<uint4*>(p.dv + p.vdv.off(bb, hh, key) + 16 * u);
                    uint4* dkp = reinterpret_cast<uint4*>(p.dk + p.vdk.off(bb, hh, key) + 16 * u);
                    dvp[0] = make_uint4(va[0], va[1], va[2], va[3]);
                    dvp[1] = make_uint4(va[4], va[5], va[6], va[7]);
                    dkp[0] = make_uint4(vb[0], vb[1], vb[2], vb[3]);
                    dkp[1] = make_uint4(vb[4], vb[5], vb[6], vb[7]);
                }
            }
        }
    } else if constexpr (WITH_DQ) {
        // ------------------------------------------------------------ dQ_i read-out and reduce-add
        const int wq = warp & 3;
        const int qr = wq * 32 + lane;                 // query row inside the tile
        const uint32_t tQ = tmem + ((uint32_t)(wq * 32) << 16) + TM::DQ;
        const bool leader = threadIdx.x == DQ_WARP0 * 32;
        // d <= 32: lane 0 of the next warp issues dQ_i = dS K, beside the main
        // issuer (one thread issues a product only every ~80-100 cycles).
        const bool dq_issuer = TM::SPLIT_DQ && warp == DQ_WARP0 + 1;
        bool iss_ok = true;
        if (dq_issuer) iss_ok = warp_wait(kv_full, 0, abort, p.status);   // K is resident
        griddep_wait();                                // the dQ accumulator is zeroed by the previous kernel
        for (int it = 0; it < n_it; ++it) {
            const int s = it % NS;
            if (dq_issuer) {
                // dS^T of tile it is in shared memory and dQ_{i-1} has been read out.
                if (!(iss_ok = iss_ok && warp_wait(p_full, it & 1, abort, p.status))) break;
                if (it > 0 && !(iss_ok = warp_wait(dq_empty, (it - 1) & 1, abort, p.status))) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t dso = (uint32_t)((it & 1) * G::DS_BYTES) >> 4;
                    const uint32_t k_mn_lo = desc_lo(sb + G::K_OFF, C::tile_off(1, 128));
                    const uint32_t ds_m_lo = desc_lo(sb + G::DS_OFF, 16384);
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks) {                                  // dQ_i = dS K
                        const uint64_t adesc = desc_make(ds_m_lo + dso + ks * 128, desc_hi(1024, SW_128B));
                        mma_n_is_d<D, false, C>(tmem + TM::DQ, 0, adesc, k_mn_lo, ks, 1, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(dq_full);
                }
                __syncwarp();
            }
            if (!warp_wait(dq_full, it & 1, abort, p.status)) break;
            if constexpr (TM::DQSTAGE) {
                // All of dQ_i into registers (its columns are then free for
                // dQ_{i+1}), then chunk by chunk through the staging buffer.
                tc_fence_after();
                uint32_t r[QC::NCH][32];
#pragma unroll
                for (int cq = 0; cq < QC::NCH; ++cq) tmem_ld32(tQ + 32 * cq, r[cq]);
                tmem_wait_ld();
#pragma unroll
                for (int cq = 0; cq < QC::NCH; ++cq) reg_fence<32>(r[cq]);
                tc_fence_before();
                mbar_arrive(dq_empty);
                const uint32_t buf = sb + G::DQS_OFF;
                const int q0 = (i0 + it) * BQ;
                bool st_ok = true;
#pragma unroll
                for (int cq = 0; cq < QC::NCH; ++cq) {
                    static_assert(QC::NCH * 32 == D, "32-column dQ chunks");
                    const int k = it * QC::NCH + cq;             // staging round
                    if (k > 0 && !(st_ok = warp_wait(stg_free, (k - 1) & 1, abort, p.status))) break;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t off = (uint32_t)qr * 128 + (uint32_t)u * 16;
                        const uint32_t phys = off ^ (((off >> 7) & 7u) << 4);
                        st_shared_v4(buf + phys, r[cq][4 * u], r[cq][4 * u + 1], r[cq][4 * u + 2], r[cq][4 * u + 3]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(stg);
                    int lead_ok = 1;
                    if (leader) {
                        if (mbar_wait(stg, k & 1, abort, p.status, WAIT_LIMIT_NS)) {
                            tma_reduce_add_3d(&p.tdq[QC::map_index(cq)], buf, cq * 32, q0, bh);
                            bulk_commit();
                            bulk_wait_read();
                            mbar_arrive(stg_free);             // the buffer may take the next chunk
                        } else {
                            lead_ok = 0;
                        }
                    }
                    if ((warp == DQ_WARP0) && __shfl_sync(0xffffffffu, lead_ok, 0) == 0) {
                        st_ok = false;
                        break;
                    }
                }
                if (!st_ok) break;
                continue;
            }
            // d <= 32: dK (the other issuer's) must also have read dS^T before
            // the tile is staged over it; its commit completes q_empty.
            if (TM::SPLIT_DQ && !warp_wait(q_empty(s), (it / NS) & 1, abort, p.status)) break;
            tc_fence_after();
            // Stage this row box by box in the TMA swizzle: for d <= 32 into
            // the dS^T buffer that dK and dQ_i have just read, for d > 64 into
            // the Q_i / dO_i slot, whose readers finished before dQ_i did.
            constexpr bool IN_DS = TM::PIPE && TM::SPLIT_DQ;
            const uint32_t slot = IN_DS ? sb + G::DS_OFF + (uint32_t)((it & 1) * G::DS_BYTES) : q_slot(s);
#pragma unroll
            for (int cq = 0; cq < QC::NCH; ++cq) {
                constexpr int W32 = 32;
                const int w = QC::width(cq);
                uint32_t r[W32];
                if (w == 32) tmem_ld32(tQ + 32 * cq, r);
                else tmem_ld16(tQ + 32 * cq, r);
                tmem_wait_ld();
                reg_fence<W32>(r);
                if (cq == QC::NCH - 1) {
                    tc_fence_before();
                    mbar_arrive(dq_empty);                 // TMEM columns free for the next dP^T
                }
                const uint32_t rb = (uint32_t)w * 4;       // 128 or 64 bytes per row
                const uint32_t mask = w == 32 ? 7u : 3u;
                const uint32_t base = slot + QC::offset(cq);
#pragma unroll
                for (int u = 0; u < W32 / 4; ++u) {
                    if (u < w / 4) {
                        const uint32_t off = (uint32_t)qr * rb + (uint32_t)u * 16;
                        const uint32_t phys = off ^ (((off >> 7) & mask) << 4);
                        st_shared_v4(base + phys, r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(stg);
            int lead_ok = 1;
            if (leader) {
                if (mbar_wait(stg, it & 1, abort, p.status, WAIT_LIMIT_NS)) {
                    const int q0 = (i0 + it) * BQ;
#pragma unroll
                    for (int cq = 0; cq < QC::NCH; ++cq)
                        tma_reduce_add_3d(&p.tdq[QC::map_index(cq)], slot + QC::offset(cq), cq * 32, q0, bh);
                    bulk_commit();
                    bulk_wait_read();
                    // The buffer may take the next dS^T / the next Q, dO tile.
                    mbar_arrive(IN_DS ? ds_free(it & 1) : q_empty(s));
                } else {
                    lead_ok = 0;
                }
            }
            // The whole warp leaves together if the leader gave up.
            if ((warp == DQ_WARP0) && __shfl_sync(0xffffffffu, lead_ok, 0) == 0) break;
        }
        if (leader) bulk_wait_all();
        if (dq_issuer && *abort) {
            // Every product this thread issued has finished before TMEM is freed.
            if (lane == 0) {
                volatile int no_abort = 0;
                mma_commit(drain_dq);
                mbar_wait(drain_dq, 0, &no_abort, p.status, WAIT_LIMIT_NS);
            }
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D, bool WITH_DQ>
cudaError_t bwd_tc_launch(const BwdArgs& a) {
    using C = BwdChunks<D>;
    using G = BwdCfg<D>;
    BwdParams p;
    memset(&p, 0, sizeof(p));
    const int BH = a.B * a.H;
    const void* src[4] = {a.q, a.k, a.v, a.dO};
    const int rows[4] = {a.S, a.Sk, a.Sk, a.S};
    const View views[4] = {a.vq, a.vk, a.vv, a.vdo};
    CUtensorMap* maps[4] = {p.tq, p.tk, p.tv, p.tdo};
    for (int i = 0; i < 4; ++i) {
        cudaError_t e;
        bool r3 = false;
        if (C::MAP_W0 > 0 &&
            (e = make_tmap_bf16_view(&maps[i][0], &r3, src[i], D, rows[i], a.H, a.B, views[i], C::MAP_W0, 128)) !=
                cudaSuccess)
            return e;
        if (C::MAP_W1 > 0 &&
            (e = make_tmap_bf16_view(&maps[i][1], &r3, src[i], D, rows[i], a.H, a.B, views[i], C::MAP_W1, 128)) !=
                cudaSuccess)
            return e;
        if (r3) p.map3 |= 1u << i;
    }
    if (WITH_DQ) {
        using QC = DqChunks<D>;
        cudaError_t e;
        if (QC::N32 > 0 && (e = make_tmap_f32_3d(&p.tdq[0], a.dQacc, D, a.S, BH, 32, 128)) != cudaSuccess) return e;
        if (QC::NCH > QC::N32 && (e = make_tmap_f32_3d(&p.tdq[1], a.dQacc, D, a.S, BH, 16, 128)) != cudaSuccess) return e;
    }
    p.lse = a.lse;
    p.Dvec = a.Dvec;
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.status = a.status;
    p.vdk = a.vdk;
    p.vdv = a.vdv;
    p.H = a.H;
    p.S = a.S;
    p.Sk = a.Sk;
    p.n_q = (a.S + BQ - 1) / BQ;
    p.n_kv = (a.Sk + BK - 1) / BK;
    // Causal: key tiles past the last query tile are attended by no query;
    // their zero gradients are written by a separate launch.
    if (a.causal) p.n_kv = std::min(p.n_kv, p.n_q);
    // Each CTA streams its head's Q, dO (bf16) and, with dQ, the fp32 dQ rows.
    p.grp = head_group(BH, p.n_kv, (4.0 + (WITH_DQ ? 4.0 : 0.0)) * a.S * D, WITH_DQ ? 160.0 : 128.0);
    p.causal = a.causal;
    const float c = fabsf(a.scale) * FA_LOG2E;
    p.c = c < 1e-30f ? 1e-30f : c;
    p.scale = a.scale;
    p.neg_a = a.scale < 0.f ? 1u : 0u;
    auto kern = bwd_tc_kernel<D, WITH_DQ>;
    cudaError_t e = set_smem_limit<bwd_tc_kernel<D, WITH_DQ>>(G::DYN_SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.n_kv * BH), dim3(bwd_threads<D>()), G::DYN_SMEM, a.stream, p);
}

template <bool WITH_DQ>
cudaError_t bwd_tc_dispatch(const BwdArgs& a) {
    switch (a.d) {
        case 16: return bwd_tc_launch<16, WITH_DQ>(a);
        case 32: return bwd_tc_launch<32, WITH_DQ>(a);
        case 64: return bwd_tc_launch<64, WITH_DQ>(a);
        case 80: return bwd_tc_launch<80, WITH_DQ>(a);
        case 96: return bwd_tc_launch<96, WITH_DQ>(a);
        case 128: return bwd_tc_launch<128, WITH_DQ>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs& a) { return bwd_tc_dispatch<true>(a); }

cudaError_t launch_bwd_tc_dkdv(const BwdArgs& a) { return bwd_tc_dispatch<false>(a); }

}  // namespace fa
