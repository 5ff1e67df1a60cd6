"""Plain fp64 attention: forward, standard backward, D, and the two-half merge.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports this module, and this module imports nothing from the library.

Layout: every 4-D array is [B, H, N, d] (float64) with N = N_q for Q, O, dO
and N = N_k for K, V (Algorithms 1 and 2 of the handout take Q in R^{N_q x d}
and K, V in R^{N_k x d}); L and D are [B, H, N_q].  Under the causal mask key j
is kept for query i when j <= i, whatever N_q and N_k are.  Inputs are widened
exactly to float64 by the caller from the values the GPU sees (bf16- or
fp32-rounded).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "scores", "causal_keep", "attention_fwd", "attention_fwd_rows", "attention_bwd",
    "attention_bwd_from_output", "attention_bwd_query_rows", "attention_bwd_key_rows", "rowsum_o_do",
    "round_to_storage", "partial_attention", "merge_two_halves",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def causal_keep(n_q: int, n_k: int) -> np.ndarray:
    """Boolean [n_q, n_k]: True where key j may be attended by query i (j <= i).

    "CS336 Assignment 2: Systems" (blog), FlashAttention-2 Triton kernel: an
    entry is masked when the query index is smaller than the key index.  The
    handout's ``flash_forward`` (c) adds -1e6 to masked scores; here masked
    entries are excluded outright (-inf), which gives the same softmax because
    the diagonal is always kept.
    """
    i = np.arange(n_q)[:, None]
    j = np.arange(n_k)[None, :]
    return j <= i


def scores(q_bh: np.ndarray, k_bh: np.ndarray, scale: float) -> np.ndarray:
    """S = Q K^T * scale for one (batch, head): handout Eq. 4 (scale = 1/sqrt(d) there)."""
    return (_f64(q_bh) @ _f64(k_bh).T) * float(scale)


def _softmax_and_lse(S: np.ndarray, keep):
    """Row softmax P (handout Eq. 5) and logsumexp L (Eq. 12) of one score matrix.

    L_i = log sum_j exp(S_ij) over the kept j, evaluated in the stable form
    m_i + log sum_j exp(S_ij - m_i) with m_i the row maximum.
    """
    if keep is not None:
        S = np.where(keep, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    e = np.exp(S - m)                      # excluded entries give exp(-inf) = 0
    l = e.sum(axis=1, keepdims=True)
    P = e / l
    L = m[:, 0] + np.log(l[:, 0])
    return P, L


def attention_fwd(q, k, v, causal: bool, scale: float):
    """O = softmax(Q K^T * scale) V and L = logsumexp of the scaled scores.

    Handout Eq. 4-6 and Eq. 12, one (b, h) slice at a time, full N_q x N_k
    matrix.  Returns (O [B,H,N_q,d], L [B,H,N_q]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    keep = causal_keep(Nq, k.shape[2]) if causal else None
    O = np.empty_like(q)
    L = np.empty((B, H, Nq))
    for b in range(B):
        for h in range(H):
            P, Lbh = _softmax_and_lse(scores(q[b, h], k[b, h], scale), keep)
            O[b, h] = P @ v[b, h]
            L[b, h] = Lbh
    return O, L


def attention_fwd_rows(q_bh, k_bh, v_bh, rows, causal: bool, scale: float):
    """The same definition for a chosen set of query rows of one (b, h) slice.

    Each output row depends only on its own query row and on all of K, V
    (handout Eq. 4-6), so sampled rows of a large problem are computed exactly
    without forming the whole score matrix.  Returns (O_rows [r,d], L_rows [r]).
    """
    q_bh, k_bh, v_bh = _f64(q_bh), _f64(k_bh), _f64(v_bh)
    rows = np.asarray(rows, dtype=np.int64)
    S = scores(q_bh[rows], k_bh, scale)                  # [r, S]
    keep = (np.arange(k_bh.shape[0])[None, :] <= rows[:, None]) if causal else None
    P, L = _softmax_and_lse(S, keep)
    return P @ v_bh, L


def attention_bwd(q, k, v, do, causal: bool, scale: float):
    """dQ, dK, dV by the standard backward pass, handout Eq. 7-11.

    P is recomputed by the plain forward definition, then
      dV = P^T dO                              (Eq. 7)
      dP = dO V^T                              (Eq. 8)
      dS_i = (diag(P_i) - P_i P_i^T) dP_i      (Eq. 9), i.e. P_i*dP_i - P_i (P_i . dP_i)
      dQ = dS K * scale                        (Eq. 10)
      dK = dS^T Q * scale                      (Eq. 11)
    The D shortcut of Eq. 13-19 is deliberately not used here; the pins check
    separately that P_i . dP_i equals D_i = rowsum(O * dO)_i.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, Nq, d = q.shape
    keep = causal_keep(Nq, k.shape[2]) if causal else None
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for b in range(B):
        for h in range(H):
            P, _ = _softmax_and_lse(scores(q[b, h], k[b, h], scale), keep)
            dv[b, h] = P.T @ do[b, h]
            dP = do[b, h] @ v[b, h].T
            dS = P * dP - P * np.sum(P * dP, axis=1, keepdims=True)
            dq[b, h] = (dS @ k[b, h]) * scale
            dk[b, h] = (dS.T @ q[b, h]) * scale
    return dq, dk, dv


def attention_bwd_from_output(q, k, v, o, do, L, causal: bool, scale: float):
    """dQ, dK, dV by the backward pass with recomputation, handout Eq. 13-19.

    Algorithm 2 of the handout takes the forward's output O and logsumexp L as
    inputs next to Q, K, V and dO; D = rowsum(O * dO) is formed from that O.
    With the exact O and L this equals ``attention_bwd`` (the D identity);
    with O as the forward stores it (rounded to the storage dtype, handout
    flash_forward (b): cast O to the input dtype before writing) it is the
    exact result of the method's backward on the method's own stored output.
      S = Q K^T * scale (Eq. 13),  P_ij = exp(S_ij - L_i) (Eq. 14),
      dV = P^T dO (Eq. 15),  dP = dO V^T (Eq. 16),  dS_ij = P_ij (dP_ij - D_i) (Eq. 17),
      dQ = dS K * scale (Eq. 18),  dK = dS^T Q * scale (Eq. 19).
    """
    q, k, v, o, do, L = _f64(q), _f64(k), _f64(v), _f64(o), _f64(do), _f64(L)
    B, H, Nq, d = q.shape
    keep = causal_keep(Nq, k.shape[2]) if causal else None
    D = rowsum_o_do(o, do)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for b in range(B):
        for h in range(H):
            Sm = scores(q[b, h], k[b, h], scale)
            P = np.exp(Sm - L[b, h][:, None])
            if keep is not None:
                P = np.where(keep, P, 0.0)
            dv[b, h] = P.T @ do[b, h]
            dP = do[b, h] @ v[b, h].T
            dS = P * (dP - D[b, h][:, None])
            dq[b, h] = (dS @ k[b, h]) * scale
            dk[b, h] = (dS.T @ q[b, h]) * scale
    return dq, dk, dv


def attention_bwd_query_rows(q_bh, k_bh, v_bh, o_rows, do_rows, L_rows, rows, causal: bool, scale: float):
    """dQ for chosen query rows of one (b, h) slice: handout Eq. 13-18 read one
    query row at a time.

    Row i of dQ involves row i of the score matrix and nothing else:
      S_ij  = scale * Q_i . K_j            (Eq. 13)
      P_ij  = exp(S_ij - L_i)              (Eq. 14; 0 for keys the mask drops)
      dP_ij = dO_i . V_j                   (Eq. 16)
      D_i   = dO_i . O_i                   (rowsum(O * dO))
      dQ_i  = scale * sum_j P_ij (dP_ij - D_i) K_j     (Eq. 17-18)
    so sampled rows of a long sequence are exact without the other rows.
    ``o_rows``, ``do_rows`` and ``L_rows`` are those rows' O (as the forward
    stored it), dO and L.  Returns dQ rows [r, d].
    """
    q_bh, k_bh, v_bh = _f64(q_bh), _f64(k_bh), _f64(v_bh)
    o_rows, do_rows, L_rows = _f64(o_rows), _f64(do_rows), _f64(L_rows)
    rows = np.asarray(rows, dtype=np.int64)
    S_rows = scores(q_bh[rows], k_bh, scale)                       # [r, N_k]
    P_rows = np.exp(S_rows - L_rows[:, None])
    if causal:
        P_rows = np.where(np.arange(k_bh.shape[0])[None, :] <= rows[:, None], P_rows, 0.0)
    dP_rows = do_rows @ v_bh.T
    D_rows = np.sum(o_rows * do_rows, axis=1)
    dS_rows = P_rows * (dP_rows - D_rows[:, None])
    return (dS_rows @ k_bh) * scale


def attention_bwd_key_rows(q_bh, k_bh, v_bh, o_bh, do_bh, L_bh, keys, causal: bool, scale: float):
    """dK and dV for chosen key rows of one (b, h) slice: handout Eq. 13-17,
    15 and 19 read one key (one column of the score matrix) at a time.

    Key j's gradients involve column j of P and of dS, hence every query row's
    L_i and D_i:
      P_ij  = exp(scale * Q_i . K_j - L_i) (Eq. 13-14; 0 for queries the mask drops)
      dV_j  = sum_i P_ij dO_i              (Eq. 15)
      dS_ij = P_ij (dO_i . V_j - D_i)      (Eq. 16-17), D_i = dO_i . O_i
      dK_j  = scale * sum_i dS_ij Q_i      (Eq. 19)
    ``o_bh``, ``do_bh``, ``L_bh`` hold every query row.  Returns
    (dK rows [c, d], dV rows [c, d]).
    """
    q_bh, k_bh, v_bh = _f64(q_bh), _f64(k_bh), _f64(v_bh)
    o_bh, do_bh, L_bh = _f64(o_bh), _f64(do_bh), _f64(L_bh)
    keys = np.asarray(keys, dtype=np.int64)
    n_q = q_bh.shape[0]
    S_cols = scores(q_bh, k_bh[keys], scale)                       # [N_q, c]: columns of S
    P_cols = np.exp(S_cols - L_bh[:, None])
    if causal:
        P_cols = np.where(keys[None, :] <= np.arange(n_q)[:, None], P_cols, 0.0)
    dP_cols = do_bh @ v_bh[keys].T
    D = np.sum(o_bh * do_bh, axis=1)
    dS_cols = P_cols * (dP_cols - D[:, None])
    return (dS_cols.T @ q_bh) * scale, P_cols.T @ do_bh


def round_to_storage(x, dtype: str) -> np.ndarray:
    """Round values to the storage dtype and widen back to float64.

    "fp32": round to the nearest float32.  "bf16": round to float32, then to
    the nearest bfloat16 (8 significant bits, ties to even), the rounding a
    store of an fp32 result to bfloat16 performs.  Finite inputs only.
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "fp32":
        return x32.astype(np.float64)
    if dtype != "bf16":
        raise ValueError(dtype)
    u = x32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1                      # ties go to the even 16-bit result
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def rowsum_o_do(o, do) -> np.ndarray:
    """D = rowsum(O * dO), handout section 4 "Backward pass with recomputation"
    (computed once before the backward loops, Algorithm 2, before its loops)."""
    return np.sum(_f64(o) * _f64(do), axis=-1)


def partial_attention(q_bh, k_bh, v_bh, key_idx, causal: bool, scale: float):
    """Softmax pieces of one key subset, in the notation of the two-half merge.

    "[Attention] FlashAttention/Ring-Attention/...统一原理": for the keys in
    ``key_idx`` take x = the scaled scores, m = their row maximum, the
    numerators A = exp(x - m), the denominator B = sum A, and the partial
    output o = (A . v) / B.  A row with no admissible key in the subset
    (possible under the causal mask) gets m = -inf, B = 0 and o = 0.
    Returns (o [S,d], m [S], B [S]).
    """
    q_bh, k_bh, v_bh = _f64(q_bh), _f64(k_bh), _f64(v_bh)
    key_idx = np.asarray(key_idx, dtype=np.int64)
    n = q_bh.shape[0]
    x = scores(q_bh, k_bh[key_idx], scale)               # [S, |subset|]
    if causal:
        x = np.where(key_idx[None, :] <= np.arange(n)[:, None], x, -np.inf)
    m = x.max(axis=1)
    o = np.zeros((n, v_bh.shape[1]))
    Bsum = np.zeros(n)
    ok = np.isfinite(m)
    A = np.exp(x[ok] - m[ok][:, None])
    Bsum[ok] = A.sum(axis=1)
    o[ok] = (A @ v_bh[key_idx]) / Bsum[ok][:, None]
    return o, m, Bsum


def merge_two_halves(o_l, m_l, B_l, o_r, m_r, B_r):
    """Merge two partial attentions over disjoint key sets.

    Same page as ``partial_attention``: with m = max(m_l, m_r),
      B = e^(m_l - m) B_l + e^(m_r - m) B_r
      o = (B_l e^(m_l - m) o_l + B_r e^(m_r - m) o_r) / B
    The merged logsumexp is L = m + log B.  Returns (o, m, B, L).
    """
    m = np.maximum(m_l, m_r)
    wl = np.where(np.isfinite(m_l), np.exp(m_l - m), 0.0) * B_l
    wr = np.where(np.isfinite(m_r), np.exp(m_r - m), 0.0) * B_r
    Bm = wl + wr
    o = (wl[:, None] * o_l + wr[:, None] * o_r) / Bm[:, None]
    return o, m, Bm, m + np.log(Bm)
