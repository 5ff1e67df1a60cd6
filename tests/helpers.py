"""Shared test helpers: tolerances, fp64 widening and element-wise comparison."""
import numpy as np
import torch

import oracle

# Tolerances |x - ref| <= atol + rtol*|ref| per element.
TOL = {
    "fp32": {"o": (1e-4, 1e-4), "lse": (1e-5, 0.0), "grad": (1e-4, 1e-4), "D": (1e-4, 1e-4)},
    "bf16": {"o": (2e-2, 2e-2), "lse": (1e-3, 0.0), "grad": (5e-2, 5e-2), "D": (1e-3, 1e-3)},
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


def oracle_head(q, k, v, do, b, h, causal, scale):
    """Oracle forward and backward for one (b, h) slice of [B,H,S,d] tensors."""
    sl = lambda t: f64(t[b:b + 1, h:h + 1])
    O, L = oracle.attention_fwd(sl(q), sl(k), sl(v), causal, scale)
    dq, dk, dv = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), causal, scale)
    return O[0, 0], L[0, 0], dq[0, 0], dk[0, 0], dv[0, 0]
