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
    O_st and L_st, plus D = rowsum(O_st * dO).
    """
    sl = lambda t: f64(t[b:b + 1, h:h + 1])
    O, L = oracle.attention_fwd(sl(q), sl(k), sl(v), causal, scale)
    O_st = oracle.round_to_storage(O, dtype)
    L_st = oracle.round_to_storage(L, "fp32")
    dq, dk, dv = oracle.attention_bwd_from_output(sl(q), sl(k), sl(v), O_st, sl(do), L_st, causal, scale)
    D = oracle.rowsum_o_do(O_st, sl(do))
    return dict(O=O[0, 0], L=L[0, 0], O_st=O_st[0, 0], L_st=L_st[0, 0], dq=dq[0, 0], dk=dk[0, 0],
                dv=dv[0, 0], D=D[0, 0])
