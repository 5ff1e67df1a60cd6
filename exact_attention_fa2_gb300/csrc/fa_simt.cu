// fa_simt.cu - FlashAttention-2 forward and backward on the FMA pipes.
//
// This is the fp32 path: every product and sum in fp32 FFMA, no tensor cores,
// for tight checking against the fp64 oracle.  The same templates also run
// with bf16 storage (inputs widened to fp32 in shared memory, P and dS rounded
// to bf16 before their products, as the tensor-core path does).
//
// Forward ("Stanford CS336 Assignment 2 (Systems)" handout, section 4,
// Algorithm 1): one CTA per (64-row query tile, batch*head); loop over 64-key
// tiles with the running max m, running sum l and an fp32 output accumulator.
// Scores are kept in base-2 units (scale*log2(e) folded in) and L is converted
// back to the natural log at the end.  Fully masked causal tiles are skipped.
//
// Backward (same handout, Eq. 13-19 and Algorithm 2, key-tile-outer part):
// one CTA per (64-key tile, batch*head) accumulates dK and dV in registers
// over all query tiles at or below the diagonal; dQ contributions of every
// key tile are added with fp32 atomics into the dQ accumulator, or, for the
// deterministic backward, summed by a separate query-tile-outer pass.

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int BQ = 64;
constexpr int BK = 64;
constexpr int NT = 256;
constexpr int LDP = BK + 1;

// Load rows [row0, row0+64) of one [rows, D] slice (row stride rs elements,
// 16-byte aligned rows) into shared memory as fp32 with leading dimension ld;
// rows at or beyond S are zero.
template <typename T, int D>
__device__ __forceinline__ void load_tile(float* dst, int ld, const T* src, long long rs, int row0, int S) {
    constexpr int VN = Vec16<T>::N;
    constexpr int CPR = D / VN;
    for (int idx = threadIdx.x; idx < 64 * CPR; idx += NT) {
        const int r = idx / CPR;
        const int c = (idx % CPR) * VN;
        float tmp[VN];
        if (row0 + r < S) {
            Vec16<T>::load(src + (row0 + r) * rs + c, tmp);
        } else {
#pragma unroll
            for (int i = 0; i < VN; ++i) tmp[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < VN; ++i) dst[r * ld + c + i] = tmp[i];
    }
}

template <int D>
constexpr size_t fwd_smem_bytes() {
    return sizeof(float) * (size_t)(64 * (D + 1) * 2 + 64 * D + 64 * LDP + 3 * 64);
}

template <int D>
constexpr size_t bwd_smem_bytes() {
    return sizeof(float) * (size_t)(64 * (D + 1) * 4 + 2 * 64 * LDP + 2 * 64);
}

template <typename T, int D>
__global__ void __launch_bounds__(NT)
fwd_simt_kernel(const T* __restrict__ q, View vq, const T* __restrict__ k, View vk, const T* __restrict__ v,
                View vv, T* __restrict__ o, View vo, float* __restrict__ lse, int S, int H, int n_qtiles,
                int causal, float scale_log2, int kb, int ke) {
    // Keys [kb, ke) only (the whole row for the plain forward); a row with no
    // admissible key gets O = 0 and L = -inf (partial attention).
    extern __shared__ float smem[];
    constexpr int LDQ = D + 1, LDK = D + 1, LDV = D;
    constexpr int NC = D / 16;
    float* Qs = smem;
    float* Ks = Qs + 64 * LDQ;
    float* Vs = Ks + 64 * LDK;
    float* Ps = Vs + 64 * LDV;
    float* m_s = Ps + 64 * LDP;
    float* l_s = m_s + 64;
    float* a_s = l_s + 64;

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int qt = n_qtiles - 1 - (int)blockIdx.x;   // long causal rows start first
    const int q0 = qt * BQ;
    const int bb = (int)blockIdx.y / H, hh = (int)blockIdx.y - bb * H;
    const T* qb = q + vq.off(bb, hh, 0);
    const T* kbp = k + vk.off(bb, hh, 0);
    const T* vbp = v + vv.off(bb, hh, 0);

    load_tile<T, D>(Qs, LDQ, qb, vq.s, q0, S);
    if (tid < 64) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }

    float acc[4][NC];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;

    int n_k = (ke - kb + BK - 1) / BK;
    if (causal) n_k = min(n_k, q0 + BQ - 1 >= kb ? (q0 + BQ - 1 - kb) / BK + 1 : 0);   // fully masked tiles skipped

    for (int kt = 0; kt < n_k; ++kt) {
        __syncthreads();
        load_tile<T, D>(Ks, LDK, kbp, vk.s, kb + kt * BK, ke);
        load_tile<T, D>(Vs, LDV, vbp, vv.s, kb + kt * BK, ke);
        __syncthreads();

        // S tile (the score block of Algorithm 1), rows ty*4+r, columns tx+16c.
        float s[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
#pragma unroll 8
        for (int kk = 0; kk < D; ++kk) {
            float qa[4], kb[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) qa[r] = Qs[(ty * 4 + r) * LDQ + kk];
#pragma unroll
            for (int c = 0; c < 4; ++c) kb[c] = Ks[(tx + 16 * c) * LDK + kk];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) s[r][c] = fmaf(qa[r], kb[c], s[r][c]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = q0 + ty * 4 + r;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = kb + kt * BK + tx + 16 * c;
                const bool keep = col < ke && (!causal || col <= row);
                Ps[(ty * 4 + r) * LDP + tx + 16 * c] = keep ? s[r][c] * scale_log2 : -INFINITY;
            }
        }
        __syncthreads();

        // Online softmax (Algorithm 1's running max and sum): four threads per row, 16 columns each.
        {
            const int row = tid / 4, part = tid % 4;
            float* prow = Ps + row * LDP + part * 16;
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 16; ++i) mx = fmaxf(mx, prow[i]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_old = m_s[row];
            const float m_new = fmaxf(m_old, mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float p = exp2f(prow[i] - m_use);
                sum += p;
                prow[i] = round_to<T>(p);   // P cast to V's dtype before PV
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            __syncwarp();
            if (part == 0) {
                const float alpha = exp2f(m_old - m_use);
                a_s[row] = alpha;
                l_s[row] = l_s[row] * alpha + sum;
                m_s[row] = m_new;
            }
        }
        __syncthreads();

        // O = diag(alpha) O + P V (Algorithm 1's rescaled accumulator).
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float al = a_s[ty * 4 + r];
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[r][c] *= al;
        }
#pragma unroll 4
        for (int kk = 0; kk < BK; ++kk) {
            float pa[4], vb[NC];
#pragma unroll
            for (int r = 0; r < 4; ++r) pa[r] = Ps[(ty * 4 + r) * LDP + kk];
#pragma unroll
            for (int c = 0; c < NC; ++c) vb[c] = Vs[kk * LDV + tx + 16 * c];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[r][c] = fmaf(pa[r], vb[c], acc[r][c]);
        }
    }
    __syncthreads();

    // Epilogue (the end of Algorithm 1's outer loop): O / l, L = (m + log2 l) * ln 2.
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int lr = ty * 4 + r;
        const int row = q0 + lr;
        if (row < S) {
            const float inv = l_s[lr] > 0.f ? 1.f / l_s[lr] : 0.f;
#pragma unroll
            for (int c = 0; c < NC; ++c)
                o[vo.off(bb, hh, row) + tx + 16 * c] = from_f32<T>(acc[r][c] * inv);
        }
    }
    if (tid < 64 && q0 + tid < S)
        lse[(size_t)blockIdx.y * S + q0 + tid] = l_s[tid] > 0.f ? (m_s[tid] + log2f(l_s[tid])) * FA_LN2 : -INFINITY;
}

template <typename T, int D>
__global__ void __launch_bounds__(NT)
bwd_simt_kernel(const T* __restrict__ q, View vq, const T* __restrict__ k, View vk, const T* __restrict__ v,
                View vv, const T* __restrict__ dO, View vdo, const float* __restrict__ lse,
                const float* __restrict__ Dvec, float* __restrict__ dQacc,
                T* __restrict__ dk, View vdk, T* __restrict__ dv, View vdv, int S, int Sk, int H, int causal,
                float scale, float scale_log2) {
    extern __shared__ float smem[];
    constexpr int LD = D + 1;
    constexpr int NC = D / 16;
    float* Ks = smem;
    float* Vs = Ks + 64 * LD;
    float* Qs = Vs + 64 * LD;
    float* dOs = Qs + 64 * LD;
    float* Ps = dOs + 64 * LD;
    float* dSs = Ps + 64 * LDP;
    float* L2s = dSs + 64 * LDP;
    float* Ds = L2s + 64;

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int kt = blockIdx.x;            // early key tiles see the most query tiles
    const int k0 = kt * BK;
    const size_t bh = blockIdx.y;
    const int bb = (int)bh / H, hh = (int)bh - bb * H;
    const size_t base = bh * S * D;       // of the contiguous dQ accumulator
    const T* qb = q + vq.off(bb, hh, 0);
    const T* dob = dO + vdo.off(bb, hh, 0);

    load_tile<T, D>(Ks, LD, k + vk.off(bb, hh, 0), vk.s, k0, Sk);
    load_tile<T, D>(Vs, LD, v + vv.off(bb, hh, 0), vv.s, k0, Sk);

    float dk_acc[4][NC], dv_acc[4][NC];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) { dk_acc[r][c] = 0.f; dv_acc[r][c] = 0.f; }

    const int n_q = (S + BQ - 1) / BQ;
    for (int qt = causal ? kt : 0; qt < n_q; ++qt) {
        const int q0 = qt * BQ;
        __syncthreads();
        load_tile<T, D>(Qs, LD, qb, vq.s, q0, S);
        load_tile<T, D>(dOs, LD, dob, vdo.s, q0, S);
        if (tid < 64) {
            const int row = q0 + tid;
            L2s[tid] = row < S ? lse[bh * S + row] * FA_LOG2E : INFINITY;
            Ds[tid] = row < S ? Dvec[bh * S + row] : 0.f;
        }
        __syncthreads();

        // Recompute S and P (Eq. 13-14), dP (Eq. 16), dS (Eq. 17): rows are
        // queries ty*4+r, columns keys tx+16c.
        float s[4][4], dp[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) { s[r][c] = 0.f; dp[r][c] = 0.f; }
#pragma unroll 4
        for (int kk = 0; kk < D; ++kk) {
            float qa[4], da[4], kb[4], vb[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) { qa[r] = Qs[(ty * 4 + r) * LD + kk]; da[r] = dOs[(ty * 4 + r) * LD + kk]; }
#pragma unroll
            for (int c = 0; c < 4; ++c) { kb[c] = Ks[(tx + 16 * c) * LD + kk]; vb[c] = Vs[(tx + 16 * c) * LD + kk]; }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s[r][c] = fmaf(qa[r], kb[c], s[r][c]);
                    dp[r][c] = fmaf(da[r], vb[c], dp[r][c]);
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int lr = ty * 4 + r;
            const int row = q0 + lr;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = k0 + tx + 16 * c;
                const bool keep = col < Sk && row < S && (!causal || col <= row);
                const float p = keep ? exp2f(fmaf(s[r][c], scale_log2, -L2s[lr])) : 0.f;
                const float ds = p * (dp[r][c] - Ds[lr]);
                Ps[lr * LDP + tx + 16 * c] = round_to<T>(p);
                dSs[lr * LDP + tx + 16 * c] = round_to<T>(ds);
            }
        }
        __syncthreads();

        // dV += P^T dO (Eq. 15), dK += dS^T Q (Eq. 19, scale applied at the end);
        // rows are keys ty*4+r.
#pragma unroll 4
        for (int qq = 0; qq < BQ; ++qq) {
            float pa[4], sa[4], db[NC], qb[NC];
#pragma unroll
            for (int r = 0; r < 4; ++r) { pa[r] = Ps[qq * LDP + ty * 4 + r]; sa[r] = dSs[qq * LDP + ty * 4 + r]; }
#pragma unroll
            for (int c = 0; c < NC; ++c) { db[c] = dOs[qq * LD + tx + 16 * c]; qb[c] = Qs[qq * LD + tx + 16 * c]; }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    dv_acc[r][c] = fmaf(pa[r], db[c], dv_acc[r][c]);
                    dk_acc[r][c] = fmaf(sa[r], qb[c], dk_acc[r][c]);
                }
        }

        // dQ_i += dS K (Eq. 18, scale applied when dQacc is converted); the
        // deterministic backward (no dQacc) sums dQ in its own pass instead.
        if (dQacc == nullptr) continue;
        float dq[4][NC];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < NC; ++c) dq[r][c] = 0.f;
#pragma unroll 4
        for (int kk = 0; kk < BK; ++kk) {
            float sa[4], kb[NC];
#pragma unroll
            for (int r = 0; r < 4; ++r) sa[r] = dSs[(ty * 4 + r) * LDP + kk];
#pragma unroll
            for (int c = 0; c < NC; ++c) kb[c] = Ks[kk * LD + tx + 16 * c];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < NC; ++c) dq[r][c] = fmaf(sa[r], kb[c], dq[r][c]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = q0 + ty * 4 + r;
            if (row < S) {
#pragma unroll
                for (int c = 0; c < NC; ++c)
                    atomicAdd(dQacc + base + (size_t)row * D + tx + 16 * c, dq[r][c]);
            }
        }
    }

#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int row = k0 + ty * 4 + r;
        if (row < Sk) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                dk[vdk.off(bb, hh, row) + tx + 16 * c] = from_f32<T>(dk_acc[r][c] * scale);
                dv[vdv.off(bb, hh, row) + tx + 16 * c] = from_f32<T>(dv_acc[r][c]);
            }
        }
    }
}

// Deterministic dQ pass (Algorithm 2's separate query-tile-outer loop): one
// CTA per (64-row query tile, batch*head) recomputes S, P, dP and dS for every
// key tile at or below the diagonal and sums dQ = dS K in registers in key
// order, so every dQ element has one fixed summation order and no atomics.
template <typename T, int D>
__global__ void __launch_bounds__(NT)
bwd_dq_simt_kernel(const T* __restrict__ q, View vq, const T* __restrict__ k, View vk, const T* __restrict__ v,
                   View vv, const T* __restrict__ dO, View vdo, const float* __restrict__ lse,
                   const float* __restrict__ Dvec, T* __restrict__ dq, View vdq, int S, int Sk, int H, int causal,
                   float scale, float scale_log2) {
    extern __shared__ float smem[];
    constexpr int LD = D + 1;
    constexpr int NC = D / 16;
    float* Ks = smem;
    float* Vs = Ks + 64 * LD;
    float* Qs = Vs + 64 * LD;
    float* dOs = Qs + 64 * LD;
    float* dSs = dOs + 64 * LD;          // [query][key]
    float* L2s = dSs + 64 * LDP;
    float* Ds = L2s + 64;

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int n_q = (S + BQ - 1) / BQ;
    const int qt = causal ? n_q - 1 - (int)blockIdx.x : (int)blockIdx.x;   // longest rows first
    const int q0 = qt * BQ;
    const size_t bh = blockIdx.y;
    const int bb = (int)bh / H, hh = (int)bh - bb * H;
    const T* kb_ = k + vk.off(bb, hh, 0);
    const T* vb_ = v + vv.off(bb, hh, 0);

    load_tile<T, D>(Qs, LD, q + vq.off(bb, hh, 0), vq.s, q0, S);
    load_tile<T, D>(dOs, LD, dO + vdo.off(bb, hh, 0), vdo.s, q0, S);
    if (tid < 64) {
        const int row = q0 + tid;
        L2s[tid] = row < S ? lse[bh * S + row] * FA_LOG2E : INFINITY;
        Ds[tid] = row < S ? Dvec[bh * S + row] : 0.f;
    }
    float acc[4][NC];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[r][c] = 0.f;

    const int n_kall = (Sk + BK - 1) / BK;
    const int n_k = causal ? min(qt + 1, n_kall) : n_kall;
    for (int kt = 0; kt < n_k; ++kt) {
        const int k0 = kt * BK;
        __syncthreads();
        load_tile<T, D>(Ks, LD, kb_, vk.s, k0, Sk);
        load_tile<T, D>(Vs, LD, vb_, vv.s, k0, Sk);
        __syncthreads();
        // S, dP (Eq. 13, 16): rows queries ty*4+r, columns keys tx+16c.
        float s[4][4], dp[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) { s[r][c] = 0.f; dp[r][c] = 0.f; }
#pragma unroll 4
        for (int kk = 0; kk < D; ++kk) {
            float qa[4], da[4], kb[4], vb[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) { qa[r] = Qs[(ty * 4 + r) * LD + kk]; da[r] = dOs[(ty * 4 + r) * LD + kk]; }
#pragma unroll
            for (int c = 0; c < 4; ++c) { kb[c] = Ks[(tx + 16 * c) * LD + kk]; vb[c] = Vs[(tx + 16 * c) * LD + kk]; }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s[r][c] = fmaf(qa[r], kb[c], s[r][c]);
                    dp[r][c] = fmaf(da[r], vb[c], dp[r][c]);
                }
        }
        // P, dS (Eq. 14, 17).
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int lr = ty * 4 + r;
            const int row = q0 + lr;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = k0 + tx + 16 * c;
                const bool keep = col < Sk && row < S && (!causal || col <= row);
                const float pr = keep ? exp2f(fmaf(s[r][c], scale_log2, -L2s[lr])) : 0.f;
                dSs[lr * LDP + tx + 16 * c] = round_to<T>(pr * (dp[r][c] - Ds[lr]));
            }
        }
        __syncthreads();
        // dQ_i += dS K_j (Eq. 18): rows queries ty*4+r, columns d tx+16c.
#pragma unroll 4
        for (int kk = 0; kk < BK; ++kk) {
            float sa[4], kb[NC];
#pragma unroll
            for (int r = 0; r < 4; ++r) sa[r] = dSs[(ty * 4 + r) * LDP + kk];
#pragma unroll
            for (int c = 0; c < NC; ++c) kb[c] = Ks[kk * LD + tx + 16 * c];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[r][c] = fmaf(sa[r], kb[c], acc[r][c]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int row = q0 + ty * 4 + r;
        if (row < S) {
#pragma unroll
            for (int c = 0; c < NC; ++c) dq[vdq.off(bb, hh, row) + tx + 16 * c] = from_f32<T>(acc[r][c] * scale);
        }
    }
}

template <typename T, int D>
cudaError_t fwd_simt_launch(const FwdArgs& a, int kb, int ke, T* o, View vo) {
    constexpr size_t smem = fwd_smem_bytes<D>();
    auto kern = fwd_simt_kernel<T, D>;
    cudaError_t e = set_smem_limit<fwd_simt_kernel<T, D>>((int)smem);
    if (e != cudaSuccess) return e;
    const int n_qtiles = (a.S + BQ - 1) / BQ;
    dim3 grid(n_qtiles, a.B * a.H);
    kern<<<grid, NT, smem, a.stream>>>((const T*)a.q, a.vq, (const T*)a.k, a.vk, (const T*)a.v, a.vv, o, vo,
                                       a.lse, a.S, a.H, n_qtiles, a.causal, a.scale * FA_LOG2E, kb, ke);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_simt_launch(const BwdArgs& a) {
    constexpr size_t smem = bwd_smem_bytes<D>();
    auto kern = bwd_simt_kernel<T, D>;
    cudaError_t e = set_smem_limit<bwd_simt_kernel<T, D>>((int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.Sk + BK - 1) / BK, a.B * a.H);
    kern<<<grid, NT, smem, a.stream>>>((const T*)a.q, a.vq, (const T*)a.k, a.vk, (const T*)a.v, a.vv,
                                       (const T*)a.dO, a.vdo, a.lse, a.Dvec, a.dQacc, (T*)a.dk, a.vdk, (T*)a.dv,
                                       a.vdv, a.S, a.Sk, a.H, a.causal, a.scale, a.scale * FA_LOG2E);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_dq_simt_launch(const BwdArgs& a) {
    constexpr size_t smem = sizeof(float) * (size_t)(64 * (D + 1) * 4 + 64 * LDP + 2 * 64);
    auto kern = bwd_dq_simt_kernel<T, D>;
    cudaError_t e = set_smem_limit<bwd_dq_simt_kernel<T, D>>((int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.S + BQ - 1) / BQ, a.B * a.H);
    kern<<<grid, NT, smem, a.stream>>>((const T*)a.q, a.vq, (const T*)a.k, a.vk, (const T*)a.v, a.vv,
                                       (const T*)a.dO, a.vdo, a.lse, a.Dvec, (T*)a.dq, a.vdq, a.S, a.Sk, a.H,
                                       a.causal, a.scale, a.scale * FA_LOG2E);
    return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_dq_simt_dispatch(const BwdArgs& a) {
    switch (a.d) {
        case 16: return bwd_dq_simt_launch<T, 16>(a);
        case 32: return bwd_dq_simt_launch<T, 32>(a);
        case 64: return bwd_dq_simt_launch<T, 64>(a);
        case 80: return bwd_dq_simt_launch<T, 80>(a);
        case 96: return bwd_dq_simt_launch<T, 96>(a);
        case 128: return bwd_dq_simt_launch<T, 128>(a);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t fwd_simt_dispatch(const FwdArgs& a, int kb, int ke, T* o, View vo) {
    switch (a.d) {
        case 16: return fwd_simt_launch<T, 16>(a, kb, ke, o, vo);
        case 32: return fwd_simt_launch<T, 32>(a, kb, ke, o, vo);
        case 64: return fwd_simt_launch<T, 64>(a, kb, ke, o, vo);
        case 80: return fwd_simt_launch<T, 80>(a, kb, ke, o, vo);
        case 96: return fwd_simt_launch<T, 96>(a, kb, ke, o, vo);
        case 128: return fwd_simt_launch<T, 128>(a, kb, ke, o, vo);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t bwd_simt_dispatch(const BwdArgs& a) {
    switch (a.d) {
        case 16: return bwd_simt_launch<T, 16>(a);
        case 32: return bwd_simt_launch<T, 32>(a);
        case 64: return bwd_simt_launch<T, 64>(a);
        case 80: return bwd_simt_launch<T, 80>(a);
        case 96: return bwd_simt_launch<T, 96>(a);
        case 128: return bwd_simt_launch<T, 128>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a) {
    return a.dtype == DT_FP32 ? fwd_simt_dispatch<float>(a, 0, a.Sk, (float*)a.o, a.vo)
                              : fwd_simt_dispatch<__nv_bfloat16>(a, 0, a.Sk, (__nv_bfloat16*)a.o, a.vo);
}

cudaError_t launch_fwd_simt_partial(const FwdArgs& a, int key_begin, int key_end, float* o32) {
    // fp32 storage only: the partial output is fp32 like the inputs.
    if (a.dtype != DT_FP32) return cudaErrorInvalidValue;
    return fwd_simt_dispatch<float>(a, key_begin, key_end, o32, contiguous_view(a.H, a.S, a.d));
}

cudaError_t launch_bwd_simt(const BwdArgs& a) {
    return a.dtype == DT_FP32 ? bwd_simt_dispatch<float>(a) : bwd_simt_dispatch<__nv_bfloat16>(a);
}

cudaError_t launch_bwd_dq_simt(const BwdArgs& a) {
    return a.dtype == DT_FP32 ? bwd_dq_simt_dispatch<float>(a) : bwd_dq_simt_dispatch<__nv_bfloat16>(a);
}

}  // namespace fa
