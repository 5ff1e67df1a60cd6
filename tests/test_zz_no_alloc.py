"""fa_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers of this library cannot allocate device memory when they run the
backward pass (code inside an allocator's callbacks, runtimes that forbid
allocation during a step, plugins whose host owns all device memory).
fa_bwd_noalloc serves them with a workspace compiled into the library.  This
test calls it through the C ABI and checks that two calls in a row give the
same gradients as fa_bwd with a caller-allocated workspace.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_fa2_gb300 as fa
from seeded_inputs import make_inputs
from tests.helpers import TOL, assert_close

DEV = "cuda:0"


def _lib():
    from exact_attention_fa2_gb300 import build
    build.build()
    lib = fa.load_library()
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc_scratch_bytes.argtypes = []
    lib.fa_bwd_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return lib


def _noalloc_bwd(lib, q, k, v, o, do, lse, causal, scale, out=None):
    B, H, S, d = q.shape
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = fa.FA_BF16 if q.dtype == torch.bfloat16 else fa.FA_FP32
    rc = lib.fa_bwd_noalloc(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv),
                            B, H, S, d, int(causal), float(scale), code, stream)
    assert rc == 0, lib.fa_get_last_error()
    fa.check_status()
    return dq, dk, dv


def _check_case(lib, shape, dtype, causal, seed):
    B, H, S, d = shape
    q, k, v, do = (t.to(DEV) for t in make_inputs(B, H, S, d, dtype, seed=seed))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, causal, scale)
    ref = fa.bwd(q, k, v, o, do, lse, causal, scale)
    outs = [tuple(torch.empty_like(t) for t in (q, k, v)) for _ in range(2)]
    # The first call on the device looks up the scratch's address; from then
    # on a call changes neither PyTorch's allocations nor the device's free
    # memory.
    _noalloc_bwd(lib, q, k, v, o, do, lse, causal, scale, out=outs[0])
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    _noalloc_bwd(lib, q, k, v, o, do, lse, causal, scale, out=outs[1])
    torch.cuda.synchronize()
    assert (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]) == before
    # dK and dV come from the same deterministic kernels on both calls.
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])
    for call, got in enumerate(outs):
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert_close(f"{name} {dtype} (call {call + 1})", a.cpu(), b.cpu(), *TOL[dtype]["grad"])


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    lib = _lib()
    _check_case(lib, (2, 4, 1024, 64), "bf16", True, 9001)
    _check_case(lib, (1, 2, 333, 80), "fp32", False, 9002)


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib()
    cap = lib.fa_bwd_noalloc_scratch_bytes()
    B, H, S, d = 8, 16, 8192, 128                     # ~70 MB of workspace
    assert fa.bwd_workspace_size(B, H, S, d, fa.FA_BF16) > cap
    x = torch.zeros(16, device=DEV, dtype=torch.bfloat16)
    p = ctypes.c_void_p(x.data_ptr())
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, S, d, 1, 0.1, fa.FA_BF16, None)
    assert rc == -4
    assert b"built-in scratch" in lib.fa_get_last_error()
    # An oversized call that also breaks another rule gets that rule's code.
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, None, p, p, p, B, H, S, d, 1, 0.1, fa.FA_BF16, None)
    assert rc == -1 and b"lse is null" in lib.fa_get_last_error()
