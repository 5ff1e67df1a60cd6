"""Shared test helpers: tolerances, fp64 widening and element-wise comparison."""
import numpy as np
import torch

import oracle

# Tolerances |x - ref| <= atol + rtol*|ref| per element.
TOL = {
    "fp32": {"o": (1e-4, 1e-4), "lse": (1e-5, 0.0), "grad": (1e-4, 1e-4), "D": (1e-4, 1e-4)},
    "bf16": {"o": (2e-2, 2e-2), "lse": (1e-3, 0.0), "grad": (5e-2, 5e-2), "D": (1e-4, 1e-4)},
}


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def assert_close(name, got, ref, atol, rtol):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{name}: non-finite values in the GPU result"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())}/{bad.size} elements out of tolerance (atol={atol}, rtol={rtol}); "
            f"worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}; max abs err {err.max():.3e}")


def oracle_head(q, k, v, do, b, h, causal, scale, dtype):
    """Oracle results for one (b, h) slice of [B,H,S,d] tensors.

    Returns O, L (exact forward), O_st (O rounded to the storage dtype, the
    tensor the method's forward hands to its backward), L_st (L as fp32) and
    the gradients of the backward with recomputation (Eq. 13-19) applied to
    O_st and L_st, plus D = rowsum(O_st * dO), and the exact gradient
    (Eq. 7-11 on the exact forward) as dq_exact, dk_exact, dv_exact.
    """
    sl = lambda t: f64(t[b:b + 1, h:h + 1])
    O, L = oracle.attention_fwd(sl(q), sl(k), sl(v), causal, scale)
    O_st = oracle.round_to_storage(O, dtype)
    L_st = oracle.round_to_storage(L, "fp32")
    dq, dk, dv = oracle.attention_bwd_from_output(sl(q), sl(k), sl(v), O_st, sl(do), L_st, causal, scale)
    D = oracle.rowsum_o_do(O_st, sl(do))
    ex = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), causal, scale)
    return dict(O=O[0, 0], L=L[0, 0], O_st=O_st[0, 0], L_st=L_st[0, 0], dq=dq[0, 0], dk=dk[0, 0],
                dv=dv[0, 0], D=D[0, 0], dq_exact=ex[0][0, 0], dk_exact=ex[1][0, 0], dv_exact=ex[2][0, 0])


def oracle_forward_all_rows(q_bh, k_bh, v_bh, causal, scale, block=1024):
    """O and L of every query row of one (b, h) slice, a block of rows at a
    time (each row of the forward is independent of the others), so that no
    S x S matrix is held at long S.  Causal: a block's rows see only keys up
    to its last row, so only those keys are passed."""
    q_bh, k_bh, v_bh = f64(q_bh), f64(k_bh), f64(v_bh)
    n = q_bh.shape[0]
    O = np.empty((n, v_bh.shape[1]))
    L = np.empty(n)
    for r0 in range(0, n, block):
        rows = np.arange(r0, min(n, r0 + block))
        kend = int(rows[-1]) + 1 if causal else k_bh.shape[0]
        O[rows], L[rows] = oracle.attention_fwd_rows(q_bh, k_bh[:kend], v_bh[:kend], rows, causal, scale)
    return O, L


def oracle_sampled_grads(q, k, v, do, b, h, rows, keys, causal, scale, dtype):
    """Oracle gradients of one (b, h) slice on sampled query rows (dQ) and
    key rows (dK, dV), at any length.

    ``dq``/``dk``/``dv``: the backward with recomputation (Eq. 13-19) on O as
    the forward stores it (the exact O rounded to the storage dtype) and L as
    fp32, the same reading as ``oracle_head``.  ``*_exact``: the same rows of
    the true gradient (exact O and L).  Also returns the exact O, L rows."""
    Q, K, V, dO = (f64(t[b, h]) for t in (q, k, v, do))
    O, L = oracle_forward_all_rows(Q, K, V, causal, scale)
    O_st = oracle.round_to_storage(O, dtype)
    L_st = oracle.round_to_storage(L, "fp32")
    out = dict(O=O[rows], L=L[rows])
    for tag, Ou, Lu in (("", O_st, L_st), ("_exact", O, L)):
        out["dq" + tag] = oracle.attention_bwd_query_rows(Q, K, V, Ou[rows], dO[rows], Lu[rows], rows, causal, scale)
        out["dk" + tag], out["dv" + tag] = oracle.attention_bwd_key_rows(Q, K, V, Ou, dO, Lu, keys, causal, scale)
    return out


def sample_positions(S, seed, extra=8):
    """Sorted row indices of a length-S sequence: both ends of the first two
    128-row tiles, the middle, the last two tiles (the last tile is ragged
    unless 128 divides S) and `extra` seeded random rows."""
    base = {0, 1, 63, 64, 127, 128, 129, 255, 256, S // 2 - 1, S // 2, S - 129, S - 128, S - 127, S - 2, S - 1}
    rnd = np.random.default_rng(seed).choice(S, size=min(extra, S), replace=False)
    return np.array(sorted(p for p in base | set(int(x) for x in rnd) if 0 <= p < S), dtype=np.int64)
