"""The seeded input generators shared by the oracle side and the CUDA side
(CPU only): reproducible draws in the stated order, exact rounding to the
working dtype, the workloads' shapes, scales and seeds, and no attention
arithmetic in the module."""
import inspect
import re

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si


def test_same_seed_same_tensors_bitwise():
    a = si.make_inputs(1, 2, 130, 64, "bf16", seed=11)
    b = si.make_inputs(1, 2, 130, 64, "bf16", seed=11)
    c = si.make_inputs(1, 2, 130, 64, "bf16", seed=12)
    for x, y, z in zip(a, b, c):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        assert not torch.equal(x, z)


def test_draw_order_q_k_v_do():
    """Q, K, V, dO are consecutive N(0,1) draws of one generator: Q drawn with
    a shorter dO must not change, and the fp32 draws come out in that order."""
    q, k, v, do = si.make_inputs(1, 1, 8, 16, "fp32", seed=5)
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    draws = [torch.randn((1, 1, 8, 16), generator=g, dtype=torch.float32) for _ in range(4)]
    for got, want in zip((q, k, v, do), draws):
        assert torch.equal(got, want)
    q2, k2, v2, do2 = si.make_inputs_rect(1, 1, 8, 3, 16, "fp32", seed=5)
    assert torch.equal(q2, q)                    # the first draw is the same whatever comes after
    assert k2.shape == (1, 1, 3, 16) and do2.shape == (1, 1, 8, 16)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_values_are_the_fp32_draws_rounded_to_nearest_even(dtype):
    q, k, v, do = si.make_inputs(2, 1, 40, 32, dtype, seed=9, qkv_scale=2.0)
    g = torch.Generator(device="cpu")
    g.manual_seed(9)
    for i, t in enumerate((q, k, v, do)):
        raw = torch.randn((2, 1, 40, 32), generator=g, dtype=torch.float32) * (2.0 if i < 3 else 1.0)
        want = oracle.round_to_storage(raw.numpy(), dtype)
        assert t.dtype == si.torch_dtype(dtype) and t.is_contiguous()
        np.testing.assert_array_equal(t.to(torch.float64).numpy(), want)


def test_value_scale_of_the_sharp_workload():
    w = si.WORKLOADS["c4"]
    q, k, v, do = si.make_inputs(1, 2, 512, w.d, w.dtype, w.seed, w.qkv_scale)
    for t in (q, k, v):
        assert abs(t.float().std().item() - 2.0) < 0.05
    assert abs(do.float().std().item() - 1.0) < 0.03
    assert abs(q.float().mean().item()) < 0.05


def test_workload_table():
    W = si.WORKLOADS
    assert (W["c1"].B, W["c1"].H, W["c1"].S, W["c1"].d, W["c1"].dtype, W["c1"].causal) == (1, 2, 128, 64, "fp32", (True, False))
    assert (W["c2"].B, W["c2"].H, W["c2"].S, W["c2"].d, W["c2"].dtype, W["c2"].causal) == (4, 12, 1024, 64, "bf16", (True,))
    assert (W["c3"].B, W["c3"].H, W["c3"].S, W["c3"].d, W["c3"].dtype, W["c3"].causal) == (4, 16, 2048, 64, "bf16", (True, False))
    assert (W["c4"].B, W["c4"].H, W["c4"].S, W["c4"].d, W["c4"].dtype, W["c4"].qkv_scale) == (4, 32, 4096, 80, "bf16", 2.0)
    assert W["c4"].scale == pytest.approx(1 / np.sqrt(80))
    assert len({w.seed for w in W.values()}) == len(W)


def test_sweep_points():
    pts = si.sweep_points()
    assert len(pts) == 2 * 4 * 10                 # {bf16, fp32} x d in {16,32,64,128} x S = 2^7..2^16
    assert {p.S for p in pts} == {2 ** e for e in range(7, 17)}
    assert {p.d for p in pts} == {16, 32, 64, 128}
    assert all((p.B, p.H, p.causal) == (1, 16, (True,)) for p in pts)
    assert len({p.seed for p in pts}) == len(pts)
    assert len(si.sweep_points(max_S=1024)) == 2 * 4 * 4


def test_module_holds_no_attention_arithmetic():
    src = inspect.getsource(si)
    code = re.sub(r'""".*?"""', "", src, flags=re.S)            # docstrings may describe it
    for banned in ("softmax", "exp(", "matmul", "einsum", " @ ", "logsumexp", "bmm("):
        assert banned not in code, banned
