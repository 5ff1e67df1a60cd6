"""Pins that tie the fp64 oracle to facts other than itself (CPU only).

Each test checks the oracle against a hand-worked example, a closed form, an
invariant of exact softmax attention, finite differences or an independent
brute-force evaluation in plain Python.  Together they catch a dropped term,
a wrong sign, a transposed operand, a wrong mask direction or a misplaced
scale anywhere in the oracle.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- hand-worked example
@pytest.mark.parametrize("causal", [False, True])
def test_hand_worked_two_rows(causal):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_2x1.json")))
    p = g["params"]
    env = dict(c=p["c"], a=p["a"], b=p["b"], E1=math.exp(p["c"]), E2=math.exp(2 * p["c"]),
               log=math.log)
    ev = lambda xs: np.array([eval(x, {"__builtins__": {}}, env) if isinstance(x, str) else x
                              for x in xs])
    q = np.array(g["Q"])[None, None]
    k = np.array(g["K"])[None, None]
    v = np.array(g["V"])[None, None]
    do = ev(g["dO"]).reshape(1, 1, 2, 1)
    exp = g["causal" if causal else "noncausal"]
    O, L = oracle.attention_fwd(q, k, v, causal, p["c"])
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, p["c"])
    np.testing.assert_allclose(O[0, 0, :, 0], ev(exp["O"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], ev(exp["L"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0, :, 0], ev(exp["dV"]), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dq[0, 0, :, 0], ev(exp["dQ"]), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk[0, 0, :, 0], ev(exp["dK"]), rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_single_key_gives_v(causal):
    """S = 1: the only weight is 1, so O = V, L = q.k*scale, dV = dO, dQ = dK = 0."""
    q, k, v, do = (rnd(s, 2, 3, 1, 8) for s in range(4))
    sc = 0.37
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    np.testing.assert_allclose(O, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L, sc * np.sum(q * k, -1), rtol=1e-14, atol=1e-15)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, sc)
    np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15


def test_zero_queries_causal_prefix_mean():
    """Q = 0, causal: P_ij = 1/(i+1) for j <= i, so O_i is the prefix mean of V,
    L_i = log(i+1), dK = 0, dV_j = sum_{i>=j} dO_i/(i+1), and
    dQ_i = scale * sum_{j<=i} (dO_i.V_j - dO_i.O_i) K_j / (i+1)."""
    S, d, sc = 9, 5, 0.41
    q = np.zeros((1, 1, S, d))
    k, v, do = rnd(10, 1, 1, S, d), rnd(11, 1, 1, S, d), rnd(12, 1, 1, S, d)
    O, L = oracle.attention_fwd(q, k, v, True, sc)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, sc)
    V, K, dO = v[0, 0], k[0, 0], do[0, 0]
    for i in range(S):
        mean = sum(V[j] for j in range(i + 1)) / (i + 1)
        np.testing.assert_allclose(O[0, 0, i], mean, rtol=1e-14, atol=1e-14)
        assert abs(L[0, 0, i] - math.log(i + 1)) < 1e-14
        dqi = sum((dO[i] @ V[j] - dO[i] @ mean) * K[j] for j in range(i + 1)) * sc / (i + 1)
        np.testing.assert_allclose(dq[0, 0, i], dqi, rtol=1e-12, atol=1e-13)
    for j in range(S):
        dvj = sum(dO[i] / (i + 1) for i in range(j, S))
        np.testing.assert_allclose(dv[0, 0, j], dvj, rtol=1e-13, atol=1e-14)
    assert np.abs(dk).max() == 0.0


def test_zero_queries_noncausal_mean():
    S, d = 7, 3
    q = np.zeros((1, 2, S, d))
    k, v, do = rnd(20, 1, 2, S, d), rnd(21, 1, 2, S, d), rnd(22, 1, 2, S, d)
    O, L = oracle.attention_fwd(q, k, v, False, 0.9)
    np.testing.assert_allclose(O, np.broadcast_to(v.mean(2, keepdims=True), O.shape), atol=1e-14)
    np.testing.assert_allclose(L, math.log(S), atol=1e-14)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, False, 0.9)
    np.testing.assert_allclose(dv, np.broadcast_to(do.sum(2, keepdims=True) / S, dv.shape),
                               atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_value_rows(causal):
    """V_j = v for every j: O = v and dP_ij = dO_i.v = D_i, so dS = 0 and dQ = dK = 0."""
    S, d = 8, 4
    q, k, do = rnd(30, 1, 1, S, d), rnd(31, 1, 1, S, d), rnd(32, 1, 1, S, d)
    v = np.broadcast_to(rnd(33, d), (1, 1, S, d)).copy()
    O, _ = oracle.attention_fwd(q, k, v, causal, 0.5)
    np.testing.assert_allclose(O, v, atol=1e-14)
    dq, dk, _ = oracle.attention_bwd(q, k, v, do, causal, 0.5)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


# ---------------------------------------------------------------- brute force
def _brute_fwd(Q, K, V, causal, sc):
    S, d = len(Q), len(Q[0])
    O, L = [], []
    for i in range(S):
        js = [j for j in range(S) if (j <= i or not causal)]
        s = {j: sc * sum(Q[i][t] * K[j][t] for t in range(d)) for j in js}
        den = sum(math.exp(s[j]) for j in js)
        O.append([sum(math.exp(s[j]) / den * V[j][t] for j in js) for t in range(d)])
        L.append(math.log(den))
    return np.array(O), np.array(L)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_brute_force_loops(causal):
    S, d, sc = 6, 3, 0.7
    q, k, v = rnd(40, 1, 1, S, d), rnd(41, 1, 1, S, d), rnd(42, 1, 1, S, d)
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    Ob, Lb = _brute_fwd(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), causal, sc)
    np.testing.assert_allclose(O[0, 0], Ob, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], Lb, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_dsoftmax_jacobian_brute_force(causal):
    """Eq. 9 with the Jacobian diag(P_i) - P_i P_i^T built explicitly per row."""
    S, d, sc = 5, 3, 0.8
    q, k, v, do = (rnd(50 + s, 1, 1, S, d) for s in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, sc)
    Q, K, V, dO = q[0, 0], k[0, 0], v[0, 0], do[0, 0]
    Sm = sc * Q @ K.T
    if causal:
        Sm = np.where(np.tril(np.ones((S, S), bool)), Sm, -np.inf)
    P = np.exp(Sm - Sm.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    dP = dO @ V.T
    dS = np.stack([(np.diag(P[i]) - np.outer(P[i], P[i])) @ dP[i] for i in range(S)])
    np.testing.assert_allclose(dq[0, 0], sc * dS @ K, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dk[0, 0], sc * dS.T @ Q, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0], P.T @ dO, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    """Central differences of loss = sum(W * O) w.r.t. Q, K, V (fp64, h = 1e-6)."""
    S, d, sc, h = 5, 3, 0.6, 1e-6
    q, k, v, w = (rnd(60 + s, 1, 1, S, d) for s in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, w, causal, sc)

    def loss(q_, k_, v_):
        return float(np.sum(w * oracle.attention_fwd(q_, k_, v_, causal, sc)[0]))

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros((S, d))
        for i in range(S):
            for t in range(d):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][0, 0, i, t] += h
                args_m[which][0, 0, i, t] -= h
                num[i, t] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad[0, 0], num, rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """K_j += u for all j adds scale*Q_i.u to every score of row i: P, O, dQ, dK, dV
    are unchanged and L_i moves by scale*Q_i.u."""
    S, d, sc = 8, 4, 0.45
    q, k, v, do = (rnd(70 + s, 1, 2, S, d) for s in range(4))
    u = rnd(74, d)
    O1, L1 = oracle.attention_fwd(q, k, v, causal, sc)
    O2, L2 = oracle.attention_fwd(q, k + u, v, causal, sc)
    np.testing.assert_allclose(O2, O1, atol=1e-13)
    np.testing.assert_allclose(L2 - L1, sc * q @ u, atol=1e-13)
    g1 = oracle.attention_bwd(q, k, v, do, causal, sc)
    g2 = oracle.attention_bwd(q, k + u, v, do, causal, sc)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_key_permutation_invariance_noncausal():
    S, d = 8, 4
    q, k, v, do = (rnd(80 + s, 1, 1, S, d) for s in range(4))
    perm = np.random.default_rng(84).permutation(S)
    O1, L1 = oracle.attention_fwd(q, k, v, False, 0.5)
    O2, L2 = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm], False, 0.5)
    np.testing.assert_allclose(O2, O1, atol=1e-14)
    np.testing.assert_allclose(L2, L1, atol=1e-14)
    _, dk1, dv1 = oracle.attention_bwd(q, k, v, do, False, 0.5)
    _, dk2, dv2 = oracle.attention_bwd(q, k[:, :, perm], v[:, :, perm], do, False, 0.5)
    np.testing.assert_allclose(dk2, dk1[:, :, perm], atol=1e-13)
    np.testing.assert_allclose(dv2, dv1[:, :, perm], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sums_and_d_identity(causal):
    """Rows of dS sum to 0, hence sum_j dK_j = 0; and D = rowsum(O*dO) equals
    rowsum(P*dP) (handout, backward pass with recomputation)."""
    S, d, sc = 10, 6, 0.3
    q, k, v, do = (rnd(90 + s, 1, 1, S, d) for s in range(4))
    O, _ = oracle.attention_fwd(q, k, v, causal, sc)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, sc)
    np.testing.assert_allclose(dk.sum(2), 0.0, atol=1e-13)
    D = oracle.rowsum_o_do(O, do)[0, 0]
    Q, K, V, dO = q[0, 0], k[0, 0], v[0, 0], do[0, 0]
    for i in range(S):
        js = range(i + 1) if causal else range(S)
        s = [sc * (Q[i] @ K[j]) for j in js]
        den = sum(math.exp(x) for x in s)
        val = sum(math.exp(x) / den * (dO[i] @ V[j]) for x, j in zip(s, js))
        assert abs(val - D[i]) < 1e-12


# ---------------------------------------------------------------- two-half merge
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("split", [1, 4, 7])
def test_two_half_merge_equals_full(causal, split):
    S, d, sc = 8, 4, 0.55
    q, k, v = (rnd(100 + s, 1, 1, S, d)[0, 0] for s in range(3))
    O, L = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], causal, sc)
    ol, ml, bl = oracle.partial_attention(q, k, v, np.arange(split), causal, sc)
    orr, mr, br = oracle.partial_attention(q, k, v, np.arange(split, S), causal, sc)
    om, m, Bm, Lm = oracle.merge_two_halves(ol, ml, bl, orr, mr, br)
    np.testing.assert_allclose(om, O[0, 0], atol=1e-14)
    np.testing.assert_allclose(Lm, L[0, 0], atol=1e-14)


def test_merge_is_symmetric_associative_and_has_an_identity():
    """The merge of the partial softmax pieces is the exact combination of
    two key sets, so its result cannot depend on the order of the sets or on
    how three sets are grouped, and a set with no admissible key (m = -inf,
    B = 0) leaves the other unchanged.  A partial over a single key is that
    key's value row with logsumexp equal to its score."""
    S, d, sc = 9, 3, 0.8
    q, k, v = (rnd(120 + s, 1, 1, S, d)[0, 0] for s in range(3))
    a = oracle.partial_attention(q, k, v, np.array([0, 1, 2]), False, sc)
    b = oracle.partial_attention(q, k, v, np.array([3, 4]), False, sc)
    c = oracle.partial_attention(q, k, v, np.array([5, 6, 7, 8]), False, sc)
    ab = oracle.merge_two_halves(*a, *b)
    ba = oracle.merge_two_halves(*b, *a)
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-15)
    np.testing.assert_allclose(ab[3], ba[3], atol=1e-15)
    ab_c = oracle.merge_two_halves(*ab[:3], *c)
    bc = oracle.merge_two_halves(*b, *c)
    a_bc = oracle.merge_two_halves(*a, *bc[:3])
    np.testing.assert_allclose(ab_c[0], a_bc[0], atol=1e-14)
    np.testing.assert_allclose(ab_c[3], a_bc[3], atol=1e-14)
    O, L = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], False, sc)
    np.testing.assert_allclose(ab_c[0], O[0, 0], atol=1e-14)
    # Causal: keys 5..8 are admissible only for queries 5..8; rows 0..4 get
    # an empty set, which the merge must ignore.
    e = oracle.partial_attention(q, k, v, np.array([5, 6, 7, 8]), True, sc)
    assert np.all(np.isneginf(e[1][:5])) and np.all(e[2][:5] == 0) and np.all(e[0][:5] == 0)
    f = oracle.partial_attention(q, k, v, np.arange(5), True, sc)
    ef = oracle.merge_two_halves(*f, *e)
    Oc, Lc = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], True, sc)
    np.testing.assert_allclose(ef[0], Oc[0, 0], atol=1e-14)
    np.testing.assert_allclose(ef[3], Lc[0, 0], atol=1e-14)
    np.testing.assert_array_equal(ef[0][:5], f[0][:5])
    # One key: the output is that key's value row, the logsumexp its score.
    o1, m1, b1 = oracle.partial_attention(q, k, v, np.array([4]), False, sc)
    np.testing.assert_allclose(o1, np.broadcast_to(v[4], o1.shape), atol=1e-15)
    np.testing.assert_allclose(m1, sc * q @ k[4], atol=1e-15)
    np.testing.assert_allclose(b1, 1.0, atol=0)


def test_sampled_rows_match_full():
    S, d = 12, 4
    q, k, v = (rnd(110 + s, 1, 1, S, d) for s in range(3))
    for causal in (False, True):
        O, L = oracle.attention_fwd(q, k, v, causal, 0.5)
        rows = [0, 5, 11]
        Or, Lr = oracle.attention_fwd_rows(q[0, 0], k[0, 0], v[0, 0], rows, causal, 0.5)
        np.testing.assert_allclose(Or, O[0, 0, rows], atol=1e-15)
        np.testing.assert_allclose(Lr, L[0, 0, rows], atol=1e-15)


# ---------------------------------------------------------------- library cross-check (extra)
@pytest.mark.parametrize("causal", [False, True])
def test_torch_sdpa_fp64_cross_check(causal):
    torch = pytest.importorskip("torch")
    S, d, sc = 16, 8, 0.25
    q, k, v, do = (rnd(120 + s, 2, 2, S, d) for s in range(4))
    O, _ = oracle.attention_fwd(q, k, v, causal, sc)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, sc)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=sc)
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(O, to.detach().numpy(), atol=1e-12)
    for a, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-12)


# ---------------------------------------------------------------- recompute backward and storage rounding
@pytest.mark.parametrize("causal", [False, True])
def test_recompute_backward_equals_standard_with_exact_output(causal):
    """Eq. 13-19 with the exact O and L give the same gradients as Eq. 7-11."""
    S, d, sc = 11, 5, 0.45
    q, k, v, do = (rnd(130 + s, 2, 2, S, d) for s in range(4))
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    g1 = oracle.attention_bwd(q, k, v, do, causal, sc)
    g2 = oracle.attention_bwd_from_output(q, k, v, O, do, L, causal, sc)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(b, a, rtol=1e-11, atol=1e-13)


def test_recompute_backward_uses_the_given_output():
    """Perturbing O by e in one row moves D_i by e.dO_i, hence dQ_i by
    -scale * (e.dO_i) * sum_j P_ij K_j and dK_j by -scale * (e.dO_i) P_ij Q_i."""
    S, d, sc = 6, 3, 0.5
    q, k, v, do = (rnd(140 + s, 1, 1, S, d) for s in range(4))
    O, L = oracle.attention_fwd(q, k, v, False, sc)
    e = rnd(144, d) * 1e-3
    O2 = O.copy()
    O2[0, 0, 2] += e
    dq1, dk1, _ = oracle.attention_bwd_from_output(q, k, v, O, do, L, False, sc)
    dq2, dk2, _ = oracle.attention_bwd_from_output(q, k, v, O2, do, L, False, sc)
    dD = float(e @ do[0, 0, 2])
    P = np.exp(sc * q[0, 0] @ k[0, 0].T - L[0, 0][:, None])
    np.testing.assert_allclose(dq2[0, 0, 2] - dq1[0, 0, 2], -sc * dD * (P[2] @ k[0, 0]), atol=1e-14)
    np.testing.assert_allclose(dk2[0, 0] - dk1[0, 0], -sc * dD * np.outer(P[2], q[0, 0, 2]), atol=1e-14)


def test_round_to_bf16_closed_cases():
    x = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-7, -3.0 - 2**-7, 2.0**-130, 65504.0, 0.0])
    want = np.array([1.0, 1.0, 1 + 2**-6, 1 + 2**-7, -3.0, 2.0**-130, 65536.0, 0.0])
    np.testing.assert_array_equal(oracle.round_to_storage(x, "bf16"), want)
    np.testing.assert_array_equal(oracle.round_to_storage(np.array([1 + 2**-30]), "fp32"), [1.0])


def test_round_to_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = rnd(150, 100000) * np.exp(rnd(151, 100000) * 5)
    ref = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_to_storage(x, "bf16"), ref)


# ---------------------------------------------------------------- N_q != N_k (Algorithms 1 and 2: Q has N_q rows, K, V have N_k)
def _brute_fwd_rect(Q, K, V, causal, sc):
    """Plain loops over N_q query rows and N_k keys; causal keeps key j <= i."""
    O, L = [], []
    for i in range(len(Q)):
        js = [j for j in range(len(K)) if (j <= i or not causal)]
        s = {j: sc * sum(a * b for a, b in zip(Q[i], K[j])) for j in js}
        den = sum(math.exp(s[j]) for j in js)
        O.append([sum(math.exp(s[j]) / den * V[j][t] for j in js) for t in range(len(V[0]))])
        L.append(math.log(den))
    return np.array(O), np.array(L)


@pytest.mark.parametrize("nq,nk", [(3, 7), (7, 3), (5, 5)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_forward_matches_brute_force_loops(nq, nk, causal):
    d, sc = 3, 0.65
    q, k, v = rnd(300 + nq, 1, 1, nq, d), rnd(310 + nk, 1, 1, nk, d), rnd(320 + nk, 1, 1, nk, d)
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    assert O.shape == (1, 1, nq, d) and L.shape == (1, 1, nq)
    Ob, Lb = _brute_fwd_rect(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), causal, sc)
    np.testing.assert_allclose(O[0, 0], Ob, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(L[0, 0], Lb, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("nq,nk", [(3, 6), (6, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_gradients_finite_differences(nq, nk, causal):
    """Both backward forms against central differences of sum(W * O) for N_q != N_k."""
    d, sc, hh = 3, 0.55, 1e-6
    q, w = rnd(330, 1, 1, nq, d), rnd(331, 1, 1, nq, d)
    k, v = rnd(332, 1, 1, nk, d), rnd(333, 1, 1, nk, d)
    g_std = oracle.attention_bwd(q, k, v, w, causal, sc)
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    g_rec = oracle.attention_bwd_from_output(q, k, v, O, w, L, causal, sc)

    def loss(q_, k_, v_):
        return float(np.sum(w * oracle.attention_fwd(q_, k_, v_, causal, sc)[0]))

    for which, n in ((0, nq), (1, nk), (2, nk)):
        num = np.zeros((n, d))
        for i in range(n):
            for t in range(d):
                ap = [q.copy(), k.copy(), v.copy()]
                am = [q.copy(), k.copy(), v.copy()]
                ap[which][0, 0, i, t] += hh
                am[which][0, 0, i, t] -= hh
                num[i, t] = (loss(*ap) - loss(*am)) / (2 * hh)
        np.testing.assert_allclose(g_std[which][0, 0], num, rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(g_rec[which][0, 0], num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("nq,nk", [(9, 20), (20, 9)])
@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_torch_sdpa_fp64_cross_check(nq, nk, causal):
    """PyTorch's scaled_dot_product_attention aligns is_causal top-left
    (keep j <= i) for N_q != N_k, the reading taken here."""
    torch = pytest.importorskip("torch")
    d, sc = 8, 0.3
    q, do = rnd(340, 2, 2, nq, d), rnd(341, 2, 2, nq, d)
    k, v = rnd(342, 2, 2, nk, d), rnd(343, 2, 2, nk, d)
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    dq, dk, dv = oracle.attention_bwd_from_output(q, k, v, O, do, L, causal, sc)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=sc)
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(O, to.detach().numpy(), atol=1e-12)
    for a, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-12)


def test_rectangular_causal_keys_past_the_last_query_get_no_gradient():
    """Top-left causal with N_k > N_q: keys j >= N_q are never attended, so
    their dK and dV are exactly zero and removing them changes nothing."""
    nq, nk, d, sc = 4, 9, 3, 0.5
    q, do = rnd(350, 1, 1, nq, d), rnd(351, 1, 1, nq, d)
    k, v = rnd(352, 1, 1, nk, d), rnd(353, 1, 1, nk, d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, sc)
    assert np.all(dk[0, 0, nq:] == 0) and np.all(dv[0, 0, nq:] == 0)
    O, L = oracle.attention_fwd(q, k, v, True, sc)
    O2, L2 = oracle.attention_fwd(q, k[:, :, :nq], v[:, :, :nq], True, sc)
    np.testing.assert_allclose(O, O2, atol=1e-15)
    np.testing.assert_allclose(L, L2, atol=1e-15)
    dq2, dk2, dv2 = oracle.attention_bwd(q, k[:, :, :nq], v[:, :, :nq], do, True, sc)
    np.testing.assert_allclose(dq, dq2, atol=1e-15)
    np.testing.assert_allclose(dk[:, :, :nq], dk2, atol=1e-15)


# ---------------------------------------------------------------- backward on chosen query rows and key rows
@pytest.mark.parametrize("nq,nk", [(7, 7), (5, 9), (9, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_row_and_key_backward_match_the_whole_backward(nq, nk, causal):
    """dQ on chosen query rows and dK, dV on chosen key rows equal the whole
    matrices of Eq. 13-19, for the exact O and for a perturbed stored O."""
    d, sc = 4, 0.6
    q, do = rnd(400 + nq, 1, 1, nq, d), rnd(401, 1, 1, nq, d)
    k, v = rnd(402 + nk, 1, 1, nk, d), rnd(403, 1, 1, nk, d)
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    rows = [0, nq // 2, nq - 1]
    keys = [0, nk // 3, nk - 1]
    for Ost in (O, O + 1e-3 * rnd(404, 1, 1, nq, d)):
        dq, dk, dv = oracle.attention_bwd_from_output(q, k, v, Ost, do, L, causal, sc)
        dq_r = oracle.attention_bwd_query_rows(q[0, 0], k[0, 0], v[0, 0], Ost[0, 0, rows], do[0, 0, rows],
                                               L[0, 0, rows], rows, causal, sc)
        dk_c, dv_c = oracle.attention_bwd_key_rows(q[0, 0], k[0, 0], v[0, 0], Ost[0, 0], do[0, 0], L[0, 0],
                                                   keys, causal, sc)
        np.testing.assert_allclose(dq_r, dq[0, 0, rows], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dk_c, dk[0, 0, keys], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dv_c, dv[0, 0, keys], rtol=1e-12, atol=1e-14)


def test_row_and_key_backward_zero_queries_closed_form():
    """Q = 0, causal, with O and L given by their closed forms (prefix mean of
    V, log(i+1)): dK_j = 0, dV_j = sum_{i>=j} dO_i/(i+1) and
    dQ_i = scale * sum_{j<=i} (dO_i.V_j - dO_i.O_i) K_j / (i+1)."""
    S, d, sc = 11, 4, 0.7
    q = np.zeros((S, d))
    k, v, do = rnd(410, S, d), rnd(411, S, d), rnd(412, S, d)
    n = np.arange(1, S + 1, dtype=np.float64)
    O = np.cumsum(v, axis=0) / n[:, None]
    L = np.log(n)
    rows, keys = [0, 4, 10], [0, 6, 10]
    dq_r = oracle.attention_bwd_query_rows(q, k, v, O[rows], do[rows], L[rows], rows, True, sc)
    dk_c, dv_c = oracle.attention_bwd_key_rows(q, k, v, O, do, L, keys, True, sc)
    for a, i in enumerate(rows):
        want = sc * sum((do[i] @ v[j] - do[i] @ O[i]) * k[j] for j in range(i + 1)) / (i + 1)
        np.testing.assert_allclose(dq_r[a], want, rtol=1e-12, atol=1e-14)
    for a, j in enumerate(keys):
        np.testing.assert_allclose(dv_c[a], sum(do[i] / (i + 1) for i in range(j, S)), rtol=1e-13, atol=1e-14)
    assert np.abs(dk_c).max() == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_row_and_key_backward_finite_differences(causal):
    """Central differences of loss = sum(W * O) w.r.t. single rows of Q and
    single rows of K and V, against the row and key backward fed with the
    exact O and L (fp64, h = 1e-6)."""
    S, d, sc, h = 6, 3, 0.55, 1e-6
    q, k, v, w = (rnd(420 + s, 1, 1, S, d) for s in range(4))
    O, L = oracle.attention_fwd(q, k, v, causal, sc)
    rows, keys = [0, 3, 5], [0, 2, 5]
    dq_r = oracle.attention_bwd_query_rows(q[0, 0], k[0, 0], v[0, 0], O[0, 0, rows], w[0, 0, rows], L[0, 0, rows],
                                           rows, causal, sc)
    dk_c, dv_c = oracle.attention_bwd_key_rows(q[0, 0], k[0, 0], v[0, 0], O[0, 0], w[0, 0], L[0, 0], keys, causal, sc)

    def loss(q_, k_, v_):
        return float(np.sum(w * oracle.attention_fwd(q_, k_, v_, causal, sc)[0]))

    for which, idx, got in ((0, rows, dq_r), (1, keys, dk_c), (2, keys, dv_c)):
        num = np.zeros((len(idx), d))
        for a, i in enumerate(idx):
            for t in range(d):
                ap = [q.copy(), k.copy(), v.copy()]
                am = [q.copy(), k.copy(), v.copy()]
                ap[which][0, 0, i, t] += h
                am[which][0, 0, i, t] -= h
                num[a, t] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(got, num, rtol=1e-6, atol=1e-8)
