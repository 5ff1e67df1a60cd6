"""Randomised checks of the oracle over many small shapes (CPU only).

The fixed-shape pins in test_oracle_pins.py are repeated here over shapes and
scales drawn by hypothesis, including the extremes a fixed list can miss
(one query or one key, N_q < N_k and N_q > N_k under the causal mask):
the forward against plain Python loops over the definition, and the
gradients against central finite differences of a weighted loss.
"""
import math

import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

shapes = st.tuples(st.integers(1, 5), st.integers(1, 5), st.integers(1, 4), st.booleans(),
                   st.floats(0.1, 2.0), st.integers(0, 2 ** 31 - 1))


def _draw(nq, nk, d, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((1, 1, nq, d)), r.standard_normal((1, 1, nk, d)),
            r.standard_normal((1, 1, nk, d)), r.standard_normal((1, 1, nq, d)))


def _loops(q, k, v, causal, scale):
    """O and L by the definition, one scalar at a time."""
    nq, d = q.shape[2], q.shape[3]
    nk = k.shape[2]
    O = np.zeros((nq, d))
    L = np.zeros(nq)
    for i in range(nq):
        keys = [j for j in range(nk) if not causal or j <= i]
        s = [scale * sum(q[0, 0, i, t] * k[0, 0, j, t] for t in range(d)) for j in keys]
        m = max(s)
        z = sum(math.exp(x - m) for x in s)
        L[i] = m + math.log(z)
        for t in range(d):
            O[i, t] = sum(math.exp(x - L[i]) * v[0, 0, j, t] for x, j in zip(s, keys))
    return O, L


@settings(max_examples=60, deadline=None)
@given(shapes)
def test_forward_equals_loops_on_random_shapes(sh):
    nq, nk, d, causal, scale, seed = sh
    q, k, v, _ = _draw(nq, nk, d, seed)     # causal with nq > nk: the last queries see every key
    O, L = oracle.attention_fwd(q, k, v, causal, scale)
    Ow, Lw = _loops(q, k, v, causal, scale)
    np.testing.assert_allclose(O[0, 0], Ow, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L[0, 0], Lw, rtol=1e-12, atol=1e-12)


@settings(max_examples=30, deadline=None)
@given(shapes)
def test_gradients_equal_finite_differences_on_random_shapes(sh):
    nq, nk, d, causal, scale, seed = sh
    q, k, v, do = _draw(nq, nk, d, seed)

    def loss(q_, k_, v_):
        return float(np.sum(oracle.attention_fwd(q_, k_, v_, causal, scale)[0] * do))

    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, scale)
    O, L = oracle.attention_fwd(q, k, v, causal, scale)
    dq2, dk2, dv2 = oracle.attention_bwd_from_output(q, k, v, O, do, L, causal, scale)
    h = 1e-6
    for x, g, g2, which in ((q, dq, dq2, 0), (k, dk, dk2, 1), (v, dv, dv2, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7)
        np.testing.assert_allclose(g2, g, rtol=1e-10, atol=1e-12)
