"""GPU parity: the CUDA library (called through its C ABI) against the fp64 oracle.

Inputs are the seeded synthetic tensors of ``seeded_inputs``; the oracle sees
the same values widened exactly to float64.  Small problems are compared
element by element in full; full-size workloads are compared on sampled
(batch, head) slices, each computed exactly by the oracle.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_fa2_gb300 as fa
import oracle
from seeded_inputs import WORKLOADS, make_inputs, make_workload_inputs, sweep_points
from tests.helpers import TOL, assert_close, f64, oracle_head, oracle_sampled_grads, sample_positions

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from exact_attention_fa2_gb300 import build
    build.build()
    fa.load_library()


def run_gpu(q, k, v, do, causal, scale, o_in=None, lse_in=None):
    """fwd then bwd as a user calls them; with o_in/lse_in given, the backward
    runs on those (host-made) tensors instead of the forward's outputs."""
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal, scale)
    if o_in is not None:
        o, lse = o_in.to(DEV), lse_in.to(DEV)
    B, H, S, d = q.shape
    ws = torch.empty(fa.bwd_workspace_size(B, H, S, d, q.dtype), device=DEV, dtype=torch.uint8)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, causal, scale, workspace=ws)
    fa.check_status()
    rows = B * H * S
    D = ws[: rows * 4].view(torch.float32).view(B, H, S)
    return [t.cpu() for t in (o, lse, dq, dk, dv, D)]


def check_heads(q, k, v, do, causal, scale, dtype, heads, exact_grad=True):
    """Compare sampled (b, h) slices with the oracle, twice:
    (1) forward then backward on the forward's own outputs, as a user runs it;
    (2) the backward alone on the oracle's stored O and L (fed from the host),
        which also checks D = rowsum(O * dO) exactly on a known input.
    With ``exact_grad`` the gradients of (1) must also lie within the same
    tolerance of the exact gradient (Eq. 7-11 on the exact forward), not only
    of the recompute backward applied to the stored O."""
    tol = TOL[dtype]
    refs = {(b, h): oracle_head(q, k, v, do, b, h, causal, scale, dtype) for (b, h) in heads}
    o, lse, dq, dk, dv, _ = run_gpu(q, k, v, do, causal, scale)
    B, H, S, d = q.shape
    o_in = torch.zeros_like(q)
    lse_in = torch.full((B, H, S), 1e4, dtype=torch.float32)   # P = 0 in unsampled heads
    for (b, h), r in refs.items():
        o_in[b, h] = torch.from_numpy(r["O_st"]).to(q.dtype)
        lse_in[b, h] = torch.from_numpy(r["L_st"]).float()
    _, _, dq2, dk2, dv2, D2 = run_gpu(q, k, v, do, causal, scale, o_in, lse_in)
    for (b, h), r in refs.items():
        tag = f"[b={b},h={h},causal={causal}]"
        assert_close("O" + tag, o[b, h], r["O"], *tol["o"])
        assert_close("L" + tag, lse[b, h], r["L"], *tol["lse"])
        for name, g in (("dQ", dq), ("dK", dk), ("dV", dv)):
            assert_close(name + tag, g[b, h], r[name.lower()], *tol["grad"])
        for name, g in (("dQ", dq2), ("dK", dk2), ("dV", dv2)):
            assert_close(name + " (bwd alone)" + tag, g[b, h], r[name.lower()], *tol["grad"])
        assert_close("D" + tag, D2[b, h], r["D"], *tol["D"])
        if exact_grad:
            for name, g in (("dQ", dq), ("dK", dk), ("dV", dv)):
                assert_close(name + " vs exact gradient" + tag, g[b, h], r[name.lower() + "_exact"], *tol["grad"])


def all_heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


# ------------------------------------------------------------------ workloads
@pytest.mark.parametrize("causal", [True, False])
def test_c1_fp32_full(causal):
    w = WORKLOADS["c1"]
    q, k, v, do = make_workload_inputs(w)
    check_heads(q, k, v, do, causal, w.scale, w.dtype, all_heads(w.B, w.H))


def test_c2_bf16_causal_sampled_heads():
    w = WORKLOADS["c2"]
    q, k, v, do = make_workload_inputs(w)
    check_heads(q, k, v, do, True, w.scale, w.dtype, [(0, 0), (1, 7), (3, 11)])


@pytest.mark.parametrize("causal", [True, False])
def test_c3_bf16_sampled_heads(causal):
    w = WORKLOADS["c3"]
    q, k, v, do = make_workload_inputs(w)
    check_heads(q, k, v, do, causal, w.scale, w.dtype, [(0, 3), (3, 15)])


def test_c4_bf16_d80_sampled_heads():
    # The sharp softmax of the x2 inputs: the bf16 rounding of the stored O
    # alone moves some gradients past the tolerance of the exact gradient;
    # the distance is measured in test_c4_distance_to_the_exact_gradient.
    w = WORKLOADS["c4"]
    q, k, v, do = make_workload_inputs(w)
    check_heads(q, k, v, do, True, w.scale, w.dtype, [(0, 0), (2, 31)], exact_grad=False)


_C4 = {}


def _c4_run():
    """c4 inputs and one fwd + bwd on the GPU, shared by the c4 tests."""
    if not _C4:
        w = WORKLOADS["c4"]
        q, k, v, do = make_workload_inputs(w)
        _C4.update(w=w, inputs=(q, k, v, do), out=run_gpu(q, k, v, do, True, w.scale))
    return _C4


def test_c4_every_head_forward_rows_and_every_head_group_backward():
    """c4 (B4 H32 S4096 d80, x2 inputs): the forward on sampled rows of all
    128 heads, and dQ rows, dK and dV key rows of 15 heads spread so that
    every run of 10 consecutive heads holds one, including the last heads
    (the backward orders its grid in groups of heads at this size, the last
    group shorter than the others)."""
    c = _c4_run()
    w = c["w"]
    q, k, v, do = c["inputs"]
    o, lse, dq, dk, dv, _ = c["out"]
    tol = TOL["bf16"]
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    for b in range(w.B):
        for h in range(w.H):
            rows = sample_positions(w.S, 9000 + 32 * b + h, extra=2)[::3]
            Or, Lr = oracle.attention_fwd_rows(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), rows, True, w.scale)
            tag = f"[b={b},h={h}]"
            assert_close("O rows" + tag, o[b, h, rows], Or, *tol["o"])
            assert_close("L rows" + tag, lse[b, h, rows], Lr, *tol["lse"])
    for bh in list(range(0, w.B * w.H, 9)) + [w.B * w.H - 1]:
        b, h = divmod(bh, w.H)
        rows = sample_positions(w.S, 9500 + bh)
        keys = sample_positions(w.S, 9700 + bh)
        r = oracle_sampled_grads(q, k, v, do, b, h, rows, keys, True, w.scale, "bf16")
        tag = f"[b={b},h={h}]"
        assert_close("dQ rows" + tag, dq[b, h, rows], r["dq"], *tol["grad"])
        assert_close("dK keys" + tag, dk[b, h, keys], r["dk"], *tol["grad"])
        assert_close("dV keys" + tag, dv[b, h, keys], r["dv"], *tol["grad"])


def test_c4_distance_to_the_exact_gradient():
    """At c4 the gradients are compared with the recompute backward applied
    to O as stored in bf16 (the method's own input to its backward).  This
    measures, and bounds, how far they sit from the exact gradient of the
    exact forward on two heads; the figures are printed for the record."""
    c = _c4_run()
    w = c["w"]
    q, k, v, do = c["inputs"]
    _, _, dq, dk, dv, _ = c["out"]
    atol, rtol = TOL["bf16"]["grad"]
    for (b, h) in [(0, 0), (3, 31)]:
        r = oracle_head(q, k, v, do, b, h, True, w.scale, "bf16")
        for name, g in (("dq", dq), ("dk", dk), ("dv", dv)):
            got = f64(g[b, h])
            err = np.abs(got - r[name + "_exact"])
            excess = err - (atol + rtol * np.abs(r[name + "_exact"]))
            print(f"c4 [b={b},h={h}] {name}: max |gpu - exact| = {err.max():.4f}, "
                  f"{int((excess > 0).sum())}/{err.size} beyond the tolerance, "
                  f"max |gpu - stored-O reference| = {np.abs(got - r[name]).max():.4f}")
            assert err.max() < 0.25, f"{name} [b={b},h={h}] far from the exact gradient"
            assert (excess > 0).mean() < 1e-3


LONG = [(16384, 64, 1.0), (16384, 64, 2.0), (16384, 128, 1.0), (16384, 128, 2.0),
        (32768, 64, 1.0), (32768, 128, 2.0)]


@pytest.mark.parametrize("S,d,qkv_scale", LONG, ids=[f"S{s}_d{d}_x{int(x)}" for s, d, x in LONG])
def test_long_sequence_gradients_on_sampled_rows_and_keys(S, d, qkv_scale):
    """The backward at the lengths the throughput figures are quoted on:
    dQ on sampled query rows and dK, dV on sampled key rows (first, middle
    and last tiles and random rows) of one head, element by element against
    the oracle, whose rows are exact at any length; the forward rows too."""
    B, H = 1, 2
    q, k, v, do = make_inputs(B, H, S, d, "bf16", seed=9900 + S // 128 + d, qkv_scale=qkv_scale)
    scale = 1 / math.sqrt(d)
    o, lse, dq, dk, dv, _ = run_gpu(q, k, v, do, True, scale)
    tol = TOL["bf16"]
    b, h = 0, 1
    rows = sample_positions(S, 9910 + d)
    keys = sample_positions(S, 9920 + d)
    r = oracle_sampled_grads(q, k, v, do, b, h, rows, keys, True, scale, "bf16")
    assert_close("O rows", o[b, h, rows], r["O"], *tol["o"])
    assert_close("L rows", lse[b, h, rows], r["L"], *tol["lse"])
    assert_close("dQ rows", dq[b, h, rows], r["dq"], *tol["grad"])
    assert_close("dK keys", dk[b, h, keys], r["dk"], *tol["grad"])
    assert_close("dV keys", dv[b, h, keys], r["dv"], *tol["grad"])
    if qkv_scale == 1.0:
        for name, g in (("dq", dq[b, h, rows]), ("dk", dk[b, h, keys]), ("dv", dv[b, h, keys])):
            assert_close(name + " vs exact gradient", g, r[name + "_exact"], *tol["grad"])
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


SWEEP = [p for p in sweep_points(4096)]


@pytest.mark.parametrize("w", SWEEP, ids=[p.name for p in SWEEP])
def test_c5_sweep_point(w):
    q, k, v, do = make_workload_inputs(w)
    heads = [(0, 5)] if w.S >= 2048 else [(0, 0), (0, 15)]
    check_heads(q, k, v, do, True, w.scale, w.dtype, heads)


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 80, 96, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths_every_head_dim(dtype, d, causal):
    # 333 = 2*128 + 77: several tiles and a ragged tail.
    q, k, v, do = make_inputs(2, 2, 333, d, dtype, seed=7000 + d)
    check_heads(q, k, v, do, causal, 1.0 / math.sqrt(d), dtype, all_heads(2, 2))


@pytest.mark.parametrize("S", [1, 2, 17, 127, 128, 129, 255, 257])
def test_short_and_boundary_lengths(S):
    q, k, v, do = make_inputs(1, 3, S, 64, "bf16", seed=7100 + S)
    check_heads(q, k, v, do, True, 0.125, "bf16", all_heads(1, 3))
    q, k, v, do = make_inputs(1, 1, S, 64, "fp32", seed=7200 + S)
    check_heads(q, k, v, do, False, 0.125, "fp32", all_heads(1, 1))


@pytest.mark.parametrize("S", [512, 640, 896, 1152])
@pytest.mark.parametrize("d", [64, 128])
def test_causal_tile_pairings(S, d):
    # Few heads: the forward runs its heaviest query tiles alone and pairs the
    # light ones (odd and even tile counts, ragged and whole last tiles).
    q, k, v, do = make_inputs(1, 2, S, d, "bf16", seed=7900 + S + d)
    check_heads(q, k, v, do, True, 1.0 / math.sqrt(d), "bf16", all_heads(1, 2))


def test_single_key_closed_form():
    q, k, v, do = make_inputs(2, 4, 1, 128, "bf16", seed=7300)
    o, lse, dq, dk, dv, _ = run_gpu(q, k, v, do, True, 0.1)
    assert torch.equal(o, v)                       # the only weight is exactly 1
    assert torch.equal(dv, do)
    # dS = P (dP - D) is a difference of two fp32 sums of the same products.
    assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-3
    np.testing.assert_allclose(f64(lse), 0.1 * np.sum(f64(q) * f64(k), -1), atol=1e-3)


def test_empty_problem():
    z = torch.empty((2, 3, 0, 64), device=DEV, dtype=torch.bfloat16)
    o, lse = fa.fwd(z, z, z, True)
    assert o.shape == z.shape and lse.shape == (2, 3, 0)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_custom_scale(dtype):
    q, k, v, do = make_inputs(1, 2, 200, 32, dtype, seed=7400)
    check_heads(q, k, v, do, True, 0.37, dtype, all_heads(1, 2))


def test_zero_queries_large_causal_closed_form():
    """Q = 0 at a length the oracle cannot materialise: P_ij = 1/(i+1), so
    O_i is the prefix mean of V, L_i = log(i+1), dK = 0 and
    dV_j = sum_{i>=j} dO_i/(i+1)."""
    B, H, S, d = 1, 2, 16384, 64
    _, k, v, do = make_inputs(B, H, S, d, "bf16", seed=7500)
    q = torch.zeros_like(k)
    o, lse, dq, dk, dv, _ = run_gpu(q, k, v, do, True, 0.125)
    V, dO = f64(v), f64(do)
    n = np.arange(1, S + 1, dtype=np.float64)[:, None]
    prefix_mean = np.cumsum(V, axis=2) / n
    assert_close("O", o, prefix_mean, 2e-2, 2e-2)
    assert_close("L", lse, np.broadcast_to(np.log(n[:, 0]), (B, H, S)), 1e-3, 0)
    assert dk.abs().max().item() == 0.0
    dv_ref = np.cumsum((dO / n)[:, :, ::-1], axis=2)[:, :, ::-1]
    assert_close("dV", dv, dv_ref, 5e-2, 5e-2)


def test_long_sequence_sampled_rows():
    """Forward rows are independent: sampled rows of an S = 32768 problem are
    exact in the oracle without the full score matrix."""
    B, H, S, d = 1, 1, 32768, 128
    q, k, v, _ = make_inputs(B, H, S, d, "bf16", seed=7600)
    o, lse = fa.fwd(q.to(DEV), k.to(DEV), v.to(DEV), True)
    fa.check_status()
    rows = [0, 1, 127, 128, 4095, 20000, S - 1]
    Or, Lr = oracle.attention_fwd_rows(f64(q[0, 0]), f64(k[0, 0]), f64(v[0, 0]), rows, True, 1 / math.sqrt(d))
    assert_close("O rows", o[0, 0, rows].cpu(), Or, 2e-2, 2e-2)
    assert_close("L rows", lse[0, 0, rows].cpu(), Lr, 1e-3, 0)


def test_repeat_runs_deterministic_where_promised():
    """O, L, dK, dV come out bit-identical on repeated runs; dQ (fp32 atomics)
    may differ only in its last bits."""
    q, k, v, do = make_inputs(2, 4, 1024, 64, "bf16", seed=7700)
    r1 = run_gpu(q, k, v, do, True, 0.125)
    r2 = run_gpu(q, k, v, do, True, 0.125)
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), r1, r2):
        if name == "dq":
            assert_close("dq repeat", a, b, 1e-2, 1e-2)
        else:
            assert torch.equal(a, b), name


def test_autograd_function_matches_oracle():
    q, k, v, do = make_inputs(1, 2, 256, 64, "bf16", seed=7800)
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    out = fa.attention(qd, kd, vd, causal=True)
    out.backward(do.to(DEV))
    for b, h in all_heads(1, 2):
        r = oracle_head(q, k, v, do, b, h, True, 0.125, "bf16")
        assert_close("O", out[b, h].detach().cpu(), r["O"], *TOL["bf16"]["o"])
        assert_close("dQ", qd.grad[b, h].cpu(), r["dq"], *TOL["bf16"]["grad"])
        assert_close("dK", kd.grad[b, h].cpu(), r["dk"], *TOL["bf16"]["grad"])
        assert_close("dV", vd.grad[b, h].cpu(), r["dv"], *TOL["bf16"]["grad"])


def test_device_errors_are_reported_not_raised_on_device():
    x = torch.zeros((1, 1, 128, 64), device=DEV, dtype=torch.bfloat16)
    bad = torch.zeros(128 * 64 + 1, device=DEV, dtype=torch.bfloat16)[1:].view(1, 1, 128, 64)
    with pytest.raises(fa.FAError) as e:
        fa.fwd(bad, x, x, True)
    assert e.value.code == -3
    fa.check_status()


# ------------------------------------------------------------------ host-buffer step
def _host_step(q, k, v, do, causal, scale, stream=None):
    B, H, S, d = q.shape
    hq, hk, hv, hdo = (t.contiguous().pin_memory() for t in (q, k, v, do))
    outs = (torch.empty_like(hq).pin_memory(), torch.empty((B, H, S), dtype=torch.float32).pin_memory(),
            torch.empty_like(hq).pin_memory(), torch.empty_like(hq).pin_memory(), torch.empty_like(hq).pin_memory())
    buf = torch.empty(fa.fwd_bwd_host_buffer_size(B, H, S, d, q.dtype), device=DEV, dtype=torch.uint8)
    fa.fwd_bwd_host(hq, hk, hv, hdo, outs, buf, causal, scale, stream=stream)
    return outs, buf


@pytest.mark.parametrize("dtype,S,d,causal", [("bf16", 333, 64, True), ("fp32", 200, 32, False),
                                              ("bf16", 1024, 128, True), ("bf16", 640, 80, False)])
def test_host_buffer_step_matches_device_path_and_oracle(dtype, S, d, causal):
    """fa_fwd_bwd_host (host in, host out) gives the device path's results
    (the same kernels: O, L, dK, dV bit for bit, dQ up to its atomics) and
    the oracle's."""
    q, k, v, do = make_inputs(2, 2, S, d, dtype, seed=8100 + S + d)
    scale = 1.0 / math.sqrt(d)
    outs, _ = _host_step(q, k, v, do, causal, scale)
    torch.cuda.synchronize()
    fa.check_status()
    o, lse, dq, dk, dv = outs
    ref = run_gpu(q, k, v, do, causal, scale)
    for name, a, b in (("o", o, ref[0]), ("lse", lse, ref[1]), ("dk", dk, ref[3]), ("dv", dv, ref[4])):
        assert torch.equal(a, b), name
    assert_close("dq vs device path", dq, ref[2], *TOL[dtype]["grad"])
    tol = TOL[dtype]
    for (b, h) in [(0, 0), (1, 1)]:
        r = oracle_head(q, k, v, do, b, h, causal, scale, dtype)
        assert_close("O", o[b, h], r["O"], *tol["o"])
        assert_close("L", lse[b, h], r["L"], *tol["lse"])
        for name, g in (("dQ", dq), ("dK", dk), ("dV", dv)):
            assert_close(name, g[b, h], r[name.lower()], *tol["grad"])


def test_host_buffer_steps_on_concurrent_streams():
    """Steps on different streams with their own buffers overlap and stay correct."""
    cases = [make_inputs(1, 4, 512, 64, "bf16", seed=8200 + i) for i in range(3)]
    streams = [torch.cuda.Stream(device=DEV) for _ in cases]
    runs = [_host_step(*c, True, 0.125, stream=st) for c, st in zip(cases, streams)]
    torch.cuda.synchronize()
    fa.check_status()
    for (q, k, v, do), (outs, _) in zip(cases, runs):
        ref = run_gpu(q, k, v, do, True, 0.125)
        assert torch.equal(outs[0], ref[0]) and torch.equal(outs[3], ref[3]) and torch.equal(outs[4], ref[4])
        assert_close("dq", outs[2], ref[2], *TOL["bf16"]["grad"])


def test_kernels_see_the_writes_of_earlier_kernels_on_the_stream():
    """Every kernel is launched as a programmatic dependent of the one before
    it; an in-place PyTorch kernel right before each call must still be seen
    (x2 and x0.5 are exact in bf16)."""
    q, k, v, do = make_inputs(1, 2, 512, 64, "bf16", seed=8300)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    ws = torch.empty(fa.bwd_workspace_size(1, 2, 512, 64, qd.dtype), device=DEV, dtype=torch.uint8)
    for _ in range(3):
        qd.mul_(2)
        o, lse = fa.fwd(qd, kd, vd, True, 0.125)
        dod.mul_(0.5)
        dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, True, 0.125, workspace=ws)
    fa.check_status()
    q8, do8 = q * 8, do * 0.125
    for b, h in all_heads(1, 2):
        r = oracle_head(q8, k, v, do8, b, h, True, 0.125, "bf16")
        assert_close("O", o[b, h].cpu(), r["O"], *TOL["bf16"]["o"])
        assert_close("dQ", dq[b, h].cpu(), r["dq"], *TOL["bf16"]["grad"])
        assert_close("dK", dk[b, h].cpu(), r["dk"], *TOL["bf16"]["grad"])
        assert_close("dV", dv[b, h].cpu(), r["dv"], *TOL["bf16"]["grad"])


def test_peak_memory_far_below_materialised():
    """The score matrix is never written: fwd+bwd needs O(S*d) device memory
    (outputs and the fp32 workspace) where the materialised computation holds
    S x S score tensors."""
    B, H, S, d = 1, 16, 2048, 64
    q, k, v, do = (t.to(DEV) for t in make_inputs(B, H, S, d, "bf16", seed=8400))
    o, lse = fa.fwd(q, k, v, True)
    fa.bwd(q, k, v, o, do, lse, True)
    del o, lse
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    o, lse = fa.fwd(q, k, v, True)
    fa.bwd(q, k, v, o, do, lse, True)
    torch.cuda.synchronize()
    ours = torch.cuda.max_memory_allocated() - base
    fa.check_status()
    elt_bytes = B * H * S * d * 2
    # o, dq, dk, dv (bf16), lse, and the fp32 workspace (D + dQacc): about 6.1x one input.
    assert ours <= 7 * elt_bytes, ours
    assert ours * 4 < B * H * S * S * 2          # under a quarter of ONE bf16 S x S score tensor


# ------------------------------------------------------------------ split-KV and merge
def _oracle_partial(q, k, v, b, h, keys, causal, scale):
    o, m, Bsum = oracle.partial_attention(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), keys, causal, scale)
    with np.errstate(divide="ignore"):
        L = np.where(np.isfinite(m), m + np.log(np.where(Bsum > 0, Bsum, 1.0)), -np.inf)
    return o, L


def _check_partial(o, lse, ref_o, ref_L, tol):
    o, lse = f64(o), f64(lse)
    empty = ~np.isfinite(ref_L)
    assert np.all(np.isneginf(lse[empty])), "rows without keys must carry L = -inf"
    assert np.all(o[empty] == 0.0), "rows without keys must carry O = 0"
    ok = ~empty
    assert_close("O part", o[ok], ref_o[ok], *tol["o"])
    assert_close("L part", lse[ok], ref_L[ok], *tol["lse"])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("causal", [True, False])
def test_partial_windows_match_oracle(dtype, causal):
    """Attention over one key window equals the oracle's partial softmax over
    the same keys (queries before the window: O = 0, L = -inf when causal)."""
    B, H, S, d = 1, 2, 333, 64
    q, k, v, _ = make_inputs(B, H, S, d, dtype, seed=8500 + causal)
    scale = 1.0 / math.sqrt(d)
    tol = TOL[dtype]
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    for kb, ke in [(0, 128), (128, 333), (256, 300), (0, 333)]:
        o, lse = fa.fwd_partial(qd, kd, vd, kb, ke, causal, scale)
        fa.check_status()
        o, lse = o.cpu(), lse.cpu()
        for b, h in all_heads(B, H):
            ref_o, ref_L = _oracle_partial(q, k, v, b, h, np.arange(kb, ke), causal, scale)
            _check_partial(o[b, h], lse[b, h], ref_o, ref_L, tol)


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("bf16", 80), ("fp32", 32)])
def test_split_kv_merge_equals_full_attention(dtype, d):
    """Partials over windows that tile the keys, merged pairwise (the chain
    keeps fp32 in between), give the full attention: against fa_fwd and the
    oracle's two-half merge."""
    B, H, S = 1, 3, 640
    q, k, v, _ = make_inputs(B, H, S, d, dtype, seed=8600 + d)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    edges = [0, 256, 384, S]
    parts = [fa.fwd_partial(qd, kd, vd, a, b, True, scale) for a, b in zip(edges[:-1], edges[1:])]
    o_acc, l_acc = parts[0]
    for o_p, l_p in parts[1:-1]:
        o_acc, l_acc = fa.merge(o_acc, l_acc, o_p, l_p, torch.float32)
    o, lse = fa.merge(o_acc, l_acc, parts[-1][0], parts[-1][1], qd.dtype)
    o_full, lse_full = fa.fwd(qd, kd, vd, True, scale)
    fa.check_status()
    tol = TOL[dtype]
    assert_close("O merged vs fa_fwd", o.cpu(), f64(o_full.cpu()), *tol["o"])
    assert_close("L merged vs fa_fwd", lse.cpu(), f64(lse_full.cpu()), *tol["lse"])
    for b, h in all_heads(B, H):
        oa, ma, Ba = oracle.partial_attention(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), np.arange(0, 256), True, scale)
        ob, mb, Bb = oracle.partial_attention(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), np.arange(256, S), True, scale)
        ref_o, _, _, ref_L = oracle.merge_two_halves(oa, ma, Ba, ob, mb, Bb)
        assert_close("O merged vs oracle", o[b, h].cpu(), ref_o, *tol["o"])
        assert_close("L merged vs oracle", lse[b, h].cpu(), ref_L, *tol["lse"])


def _bwd_both(q, k, v, do, causal, scale):
    """Forward once, then the atomic backward once and the deterministic
    backward twice (the second on a fresh, garbage-filled workspace)."""
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal, scale)
    atomic = fa.bwd(qd, kd, vd, o, dod, lse, causal, scale)
    dets = []
    for fill in (0, 0x7F):
        B, H, S, d = q.shape
        ws = torch.full((B * H * S * 4,), fill, device=DEV, dtype=torch.uint8)
        dets.append(fa.bwd(qd, kd, vd, o, dod, lse, causal, scale, workspace=ws, deterministic=True))
    fa.check_status()
    cpu = lambda ts: [t.cpu() for t in ts]
    return cpu(atomic), cpu(dets[0]), cpu(dets[1])


@pytest.mark.parametrize("dtype,d,S,causal,scale", [
    ("bf16", 64, 333, True, None), ("bf16", 128, 640, False, None), ("bf16", 80, 300, True, None),
    ("bf16", 96, 257, False, None), ("bf16", 16, 200, True, None), ("bf16", 32, 129, False, -0.3),
    ("bf16", 128, 1, True, None), ("fp32", 32, 200, True, None), ("fp32", 64, 129, False, 0.05),
])
def test_deterministic_backward_matches_oracle_and_repeats_bitwise(dtype, d, S, causal, scale):
    """Algorithm 2's separate dQ loop: every gradient within the tolerance of
    the oracle, dK and dV bitwise equal to the atomic backward's (the same
    key-tile-outer arithmetic), and all three bitwise equal across runs."""
    q, k, v, do = make_inputs(2, 2, S, d, dtype, seed=8100 + d + S)
    scale = 1 / math.sqrt(d) if scale is None else scale
    atomic, det1, det2 = _bwd_both(q, k, v, do, causal, scale)
    for name, a, b in zip(("dq", "dk", "dv"), det1, det2):
        assert torch.equal(a, b), f"{name} differs between deterministic runs"
    assert torch.equal(det1[1], atomic[1]), "dk differs from the atomic backward"
    assert torch.equal(det1[2], atomic[2]), "dv differs from the atomic backward"
    tol = TOL[dtype]
    assert_close("dq vs atomic backward", det1[0], f64(atomic[0]), *tol["grad"])
    for (b, h) in all_heads(2, 2):
        r = oracle_head(q, k, v, do, b, h, causal, scale, dtype)
        for name, g in zip(("dq", "dk", "dv"), det1):
            assert_close(f"{name} deterministic [b={b},h={h}]", g[b, h], r[name], *tol["grad"])


def test_deterministic_backward_c2_sampled_heads():
    """The deterministic backward at the full c2 workload size (4x12x1024,
    d=64, causal), sampled heads against the oracle, and repeat-exact."""
    w = WORKLOADS["c2"]
    q, k, v, do = make_workload_inputs(w)
    scale = 1 / math.sqrt(w.d)
    atomic, det1, det2 = _bwd_both(q, k, v, do, True, scale)
    for a, b in zip(det1, det2):
        assert torch.equal(a, b)
    assert torch.equal(det1[1], atomic[1]) and torch.equal(det1[2], atomic[2])
    for (b, h) in [(0, 0), (1, 5), (3, 11)]:
        r = oracle_head(q, k, v, do, b, h, True, scale, "bf16")
        for name, g in zip(("dq", "dk", "dv"), det1):
            assert_close(f"{name} deterministic [b={b},h={h}]", g[b, h], r[name], *TOL["bf16"]["grad"])


def test_deterministic_backward_c4_every_head_group():
    """The deterministic backward at c4 (B4 H32 S4096 d80, x2 inputs), where
    its dQ pass orders the grid in groups of heads: repeat-exact, dK and dV
    bit-identical to the atomic backward, and dQ on sampled rows of 15 heads
    spread so that every run of 10 consecutive heads holds one (the last,
    shorter group included) against the oracle."""
    w = WORKLOADS["c4"]
    q, k, v, do = make_workload_inputs(w)
    atomic, det1, det2 = _bwd_both(q, k, v, do, True, w.scale)
    for a, b in zip(det1, det2):
        assert torch.equal(a, b)
    assert torch.equal(det1[1], atomic[1]) and torch.equal(det1[2], atomic[2])
    assert torch.isfinite(det1[0]).all()
    for bh in list(range(0, w.B * w.H, 9)) + [w.B * w.H - 1]:
        b, h = divmod(bh, w.H)
        rows = sample_positions(w.S, 9600 + bh)
        keys = sample_positions(w.S, 9800 + bh)[:4]
        r = oracle_sampled_grads(q, k, v, do, b, h, rows, keys, True, w.scale, "bf16")
        assert_close(f"dQ rows deterministic [b={b},h={h}]", det1[0][b, h, rows], r["dq"], *TOL["bf16"]["grad"])


def test_deterministic_autograd_matches_atomic():
    q, k, v, do = make_inputs(1, 2, 384, 64, "bf16", seed=8200)
    grads = []
    for det in (False, True):
        qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
        out = fa.attention(qd, kd, vd, True, None, deterministic=det)
        out.backward(do.to(DEV))
        grads.append([t.grad.cpu() for t in (qd, kd, vd)])
    assert torch.equal(grads[0][1], grads[1][1]) and torch.equal(grads[0][2], grads[1][2])
    assert_close("dq", grads[1][0], f64(grads[0][0]), *TOL["bf16"]["grad"])


# ---------------------------------------------------------------- general shapes: N_q != N_k, strided views
from seeded_inputs import make_inputs_rect  # noqa: E402


def _run_rect(q, k, v, do, causal, scale, deterministic=False):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, causal, scale, deterministic=deterministic)
    fa.check_status()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 128), ("bf16", 80), ("bf16", 32), ("bf16", 16),
                                     ("fp32", 32)])
@pytest.mark.parametrize("Sq,Sk", [(200, 333), (333, 200), (128, 640), (640, 128), (1, 300), (300, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_rectangular_lengths_match_oracle(dtype, d, Sq, Sk, causal):
    """N_q != N_k (Algorithms 1 and 2 as stated), causal top-left, both
    backward forms, every head against the oracle."""
    q, k, v, do = make_inputs_rect(1, 2, Sq, Sk, d, dtype, seed=8300 + Sq + 7 * Sk + d)
    scale = 1 / math.sqrt(d)
    tol = TOL[dtype]
    res = _run_rect(q, k, v, do, causal, scale)
    det = _run_rect(q, k, v, do, causal, scale, deterministic=True)
    for h in range(2):
        r = oracle_head(q, k, v, do, 0, h, causal, scale, dtype)
        tag = f"[h={h},Sq={Sq},Sk={Sk},causal={causal}]"
        assert_close("O" + tag, res[0][0, h], r["O"], *tol["o"])
        assert_close("L" + tag, res[1][0, h], r["L"], *tol["lse"])
        for name, i in (("dq", 2), ("dk", 3), ("dv", 4)):
            assert_close(name + tag, res[i][0, h], r[name], *tol["grad"])
            assert_close(name + " deterministic" + tag, det[i][0, h], r[name], *tol["grad"])
    if causal and Sk > Sq:
        # Keys past the last query are never attended: exactly zero gradients.
        assert torch.count_nonzero(res[3][:, :, Sq:]) == 0 and torch.count_nonzero(res[4][:, :, Sq:]) == 0


def _layout(t, kind):
    """The same values as contiguous t [B, H, S, d] in another memory layout."""
    B, H, S, d = t.shape
    if kind == "bshd":            # [B, S, H, d] storage, viewed as [B, H, S, d]
        return t.transpose(1, 2).contiguous().transpose(1, 2)
    if kind == "padded":          # rows of d + 16 elements, the first d used
        buf = torch.zeros((B, H, S, d + 16), dtype=t.dtype, device=t.device)
        buf[..., :d] = t
        return buf[..., :d]
    if kind == "hbsd":            # [H, B, S, d] storage
        return t.transpose(0, 1).contiguous().transpose(0, 1)
    raise ValueError(kind)


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("bf16", 96), ("fp32", 64)])
@pytest.mark.parametrize("kind", ["bshd", "padded", "hbsd"])
def test_strided_views_give_bitwise_the_contiguous_results(dtype, d, kind):
    """Strides change only the addressing: O, L, dK, dV and the deterministic
    dQ must equal the contiguous call's bit for bit; the outputs are written
    into views of the same layout."""
    B, H, Sq, Sk = 2, 3, 257, 190
    q, k, v, do = (t.to(DEV) for t in make_inputs_rect(B, H, Sq, Sk, d, dtype, seed=8400 + d))
    scale = 1 / math.sqrt(d)
    ref_o, ref_l = fa.fwd(q, k, v, True, scale)
    ref_g = fa.bwd(q, k, v, ref_o, do, ref_l, True, scale, deterministic=True)
    ref_ga = fa.bwd(q, k, v, ref_o, do, ref_l, True, scale)
    qs, ks, vs, dos = (_layout(t, kind) for t in (q, k, v, do))
    assert not qs.is_contiguous()
    o_s = _layout(torch.zeros_like(q), kind)
    o, l = fa.fwd(qs, ks, vs, True, scale, out=o_s)
    grads_out = tuple(_layout(torch.zeros_like(t), kind) for t in (q, k, v))
    g = fa.bwd(qs, ks, vs, o, dos, l, True, scale, out=grads_out, deterministic=True)
    ga = fa.bwd(qs, ks, vs, o, dos, l, True, scale, out=tuple(_layout(torch.zeros_like(t), kind) for t in (q, k, v)))
    fa.check_status()
    assert o.data_ptr() == o_s.data_ptr()
    assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
    for name, a, b in zip(("dq", "dk", "dv"), g, ref_g):
        assert torch.equal(a, b), f"{name} ({kind}) differs from the contiguous call"
    assert torch.equal(ga[1], ref_ga[1]) and torch.equal(ga[2], ref_ga[2])
    assert_close("dq atomic strided", ga[0].cpu(), f64(ref_ga[0].cpu()), *TOL[dtype]["grad"])
    if kind == "padded":
        # The padding columns of the output views were not touched.
        assert torch.count_nonzero(o_s.as_strided((B, H, Sq, 16), o_s.stride(), d)) == 0


def test_backward_with_no_queries_zeroes_dk_dv():
    k, v = (torch.randn(1, 2, 200, 64, device=DEV).to(torch.bfloat16) for _ in range(2))
    q = torch.empty(1, 2, 0, 64, device=DEV, dtype=torch.bfloat16)
    o, lse = fa.fwd(q, k, v, False)
    dq, dk, dv = fa.bwd(q, k, v, o, torch.empty_like(q), lse, False,
                        out=(torch.empty_like(q), torch.full_like(k, 7.0), torch.full_like(v, 7.0)))
    fa.check_status()
    assert o.shape == (1, 2, 0, 64) and torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_misaligned_stride_is_refused():
    """A row stride of 68 bf16 elements (136 bytes) cannot be a TMA stride: the
    call is refused on the host with FA_ERR_MISALIGNED, nothing is launched."""
    base = torch.randn(1, 2, 64, 68 + 4, device=DEV).to(torch.bfloat16)
    qv = base.as_strided((1, 2, 16, 64), (2 * 64 * 72, 64 * 72, 68, 1))   # row stride 68: 136 bytes
    with pytest.raises(fa.FAError):
        fa.fwd(qv, qv, qv, False)


def test_bounded_wait_runs_out_and_is_reported_then_the_context_works():
    """Failure detection on the device: a wait that can never complete gives
    up after its limit, the kernel returns, the host reads
    FA_ERR_DEVICE_TIMEOUT, and the next calls run normally."""
    import ctypes
    lib = fa.load_library()
    assert lib.fa_selftest_bounded_wait(ctypes.c_ulonglong(20_000_000), None) == 0
    with pytest.raises(fa.FAError) as e:
        fa.check_status()
    assert e.value.code == -6 and "bounded wait" in str(e.value)
    fa.check_status()                                      # the word was cleared
    q, k, v, do = make_inputs(1, 2, 256, 64, "bf16", seed=8500)
    o, lse, dq, dk, dv, _ = run_gpu(q, k, v, do, True, 0.125)
    r = oracle_head(q, k, v, do, 0, 1, True, 0.125, "bf16")
    assert_close("O after the timeout", o[0, 1], r["O"], *TOL["bf16"]["o"])
    assert_close("dQ after the timeout", dq[0, 1], r["dq"], *TOL["bf16"]["grad"])
