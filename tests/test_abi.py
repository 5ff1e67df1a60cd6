"""The C-ABI library builds, loads and exports every declared symbol; the host
side of the argument checks works without a GPU (no kernel is launched)."""
import ctypes
import os
import re

import pytest

import exact_attention_fa2_gb300 as fa
from exact_attention_fa2_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_get_last_error",
                 "fa_check_status", "fa_version"):
        assert must in names


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_version(lib):
    assert lib.fa_version() >= 100


def test_workspace_size(lib):
    n = fa.bwd_workspace_size(2, 3, 100, 64, fa.FA_BF16)
    rows = 2 * 3 * 100
    assert n == ((rows * 4 + 255) // 256) * 256 + rows * 64 * 4
    assert fa.bwd_workspace_size(0, 3, 100, 64, fa.FA_BF16) == 0
    assert fa.bwd_workspace_size(1, 1, 1, 48, fa.FA_BF16) == 0


A = 1 << 20   # a fake, 16-byte aligned, never dereferenced address


def call_fwd(B=1, H=1, S=128, d=64, causal=0, scale=0.125, dtype=0, q=A, k=A, v=A, o=A, lse=A):
    return fa.fa_fwd(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v), ctypes.c_void_p(o),
                     ctypes.c_void_p(lse), B, H, S, d, causal, scale, dtype, None)


def test_argument_errors_need_no_gpu(lib):
    assert call_fwd(B=-1) == -1
    assert call_fwd(d=48) == -2
    assert call_fwd(dtype=7) == -2
    assert call_fwd(scale=float("nan")) == -1
    assert call_fwd(q=0) == -1
    assert call_fwd(k=A + 8) == -3
    assert b"16-byte" in lib.fa_get_last_error()
    assert call_fwd(B=1 << 12, H=1 << 12, S=1 << 10, d=128) == -2   # too many elements
    # Empty problems are valid and launch nothing.
    assert call_fwd(S=0, q=0, k=0, v=0, o=0, lse=0) == 0
    assert call_fwd(B=0) == 0


def test_bwd_workspace_errors_need_no_gpu(lib):
    P = ctypes.c_void_p(A)
    rc = fa.fa_bwd(P, P, P, P, P, P, P, P, P, P, 16, 1, 1, 128, 64, 1, 0.125, 0, None)
    assert rc == -4 and b"workspace" in lib.fa_get_last_error()
    rc = fa.fa_bwd(P, P, P, P, P, P, P, P, P, ctypes.c_void_p(A + 16), 1 << 30, 1, 1, 128, 64, 1,
                   0.125, 0, None)
    assert rc == -3


def test_host_step_buffer_size_and_errors_need_no_gpu(lib):
    B, H, S, d = 2, 3, 100, 64
    rows = B * H * S
    up = lambda x: (x + 255) // 256 * 256
    want = 8 * up(rows * d * 2) + up(rows * 4) + fa.bwd_workspace_size(B, H, S, d, fa.FA_BF16)
    assert fa.fwd_bwd_host_buffer_size(B, H, S, d, fa.FA_BF16) == want
    assert fa.fwd_bwd_host_buffer_size(B, H, S, 48, fa.FA_BF16) == 0
    P = ctypes.c_void_p(A)
    call = lambda buf, nbytes, **kw: lib.fa_fwd_bwd_host(
        P, P, P, kw.get("dO", P), P, P, P, P, P, buf, nbytes, B, H, S, d, 1, 0.125, fa.FA_BF16, None)
    assert call(ctypes.c_void_p(A), 16) == -4 and b"device buffer" in lib.fa_get_last_error()
    assert call(ctypes.c_void_p(A + 16), 1 << 30) == -3
    assert call(ctypes.c_void_p(A), 1 << 30, dO=ctypes.c_void_p(0)) == -1


def test_partial_and_merge_argument_errors_need_no_gpu(lib):
    P = ctypes.c_void_p(A)
    part = lambda kb, ke, **kw: lib.fa_fwd_partial(P, P, P, P, P, 1, 2, 512, 64, kb, ke, 1, 0.125,
                                                   kw.get("dtype", fa.FA_BF16), None)
    assert part(64, 512) == -2 and b"multiple of 128" in lib.fa_get_last_error()
    assert part(256, 256) == -1
    assert part(0, 600) == -1
    assert part(-128, 256) == -1
    mrg = lambda **kw: lib.fa_merge(P, P, kw.get("o_b", P), P, P, P, 1, 2, 512, kw.get("d", 64), fa.FA_BF16, None)
    assert mrg(o_b=ctypes.c_void_p(0)) == -1
    assert mrg(d=48) == -2


def test_deterministic_bwd_workspace_rules_need_no_gpu(lib):
    """The deterministic backward needs only D (B*H*S fp32) as workspace and
    checks it, and the pointers, before launching anything."""
    P = ctypes.c_void_p(A)
    B, H, S, d = 1, 2, 128, 64
    det = lambda ws, nbytes, **kw: fa.fa_bwd_deterministic(P, P, P, P, P, P, kw.get("dq", P), P, P, ws, nbytes,
                                                          B, H, S, kw.get("d", d), 1, 0.125, 0, None)
    assert det(P, B * H * S * 4 - 1) == -4 and b"need 1024" in lib.fa_get_last_error()
    assert det(ctypes.c_void_p(A + 16), B * H * S * 4) == -3
    assert det(P, B * H * S * 4, dq=ctypes.c_void_p(0)) == -1
    assert det(P, B * H * S * 4, d=48) == -2
    assert fa.fa_bwd_deterministic(None, None, None, None, None, None, None, None, None, None, 0,
                                   0, 2, 128, 64, 1, 0.125, 0, None) == 0


def test_strided_and_rectangular_argument_errors_need_no_gpu(lib):
    """fa_fwd_strided / fa_bwd_strided check strides and N_k before any launch."""
    P = ctypes.c_void_p(A)
    st = lambda *x: (ctypes.c_longlong * 3)(*x)
    good = st(2 * 64 * 128, 64 * 128, 64)
    fwd = lambda qs=good, ks=good, Sq=128, Sk=128, B=2, H=2, dtype=0: lib.fa_fwd_strided(
        P, qs, P, ks, P, good, P, good, P, B, H, Sq, Sk, 64, 1, 0.125, dtype, None)
    assert fwd(ks=st(0, 64 * 128, 64)) == -1 and b"not positive" in lib.fa_get_last_error()
    assert fwd(qs=st(2 * 64 * 128, 64 * 128, 68)) == -3 and b"16 bytes" in lib.fa_get_last_error()
    assert fwd(Sk=0) == -1 and b"no key rows" in lib.fa_get_last_error()
    assert fwd(Sq=0) == 0                                  # nothing to compute
    # A stride of a dimension with one index is never used, so it is not checked.
    assert fwd(qs=st(0, 0, 64), B=1, H=1, Sk=0) == -1     # fails on Sk, not on the strides
    ws = ctypes.c_void_p(A)
    bwd = lambda Sq, Sk, ws_bytes=1 << 30, dk=P: lib.fa_bwd_strided(
        P, None, P, None, P, None, P, None, P, None, P, P, None, dk, None, P, None, ws, ws_bytes,
        1, 2, Sq, Sk, 64, 1, 0.125, 0, 0, None)
    assert bwd(128, 0) == -1
    assert bwd(128, 256, ws_bytes=16) == -4
    assert bwd(0, 256, dk=ctypes.c_void_p(0)) == -1       # no queries: dk, dv still written, so checked
    assert bwd(0, 0) == 0


def test_selftest_limit_checked_without_launch(lib):
    assert lib.fa_selftest_bounded_wait(ctypes.c_ulonglong(0), None) == -1
    assert lib.fa_selftest_bounded_wait(ctypes.c_ulonglong(20_000_000_000), None) == -1


def test_noalloc_limits_need_no_gpu(lib):
    """fa_bwd_noalloc refuses a problem whose workspace exceeds its built-in
    scratch before touching the device, naming both sizes; empty problems
    and unsupported head dims are answered as fa_bwd answers them."""
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc_scratch_bytes.restype = ctypes.c_size_t
    scratch = lib.fa_bwd_noalloc_scratch_bytes()
    assert scratch == 32 << 20
    P = ctypes.c_void_p(A)
    call = lambda B, H, S, d: lib.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, B, H, S, d, 1, 0.125, fa.FA_BF16, None)
    need = fa.bwd_workspace_size(1, 16, 8192, 128, fa.FA_BF16)
    assert need > scratch
    assert call(1, 16, 8192, 128) == -4
    msg = lib.fa_get_last_error()
    assert str(need).encode() in msg and str(scratch).encode() in msg
    assert call(0, 16, 8192, 128) == 0          # empty: nothing to do
    assert call(1, 2, 128, 48) == -2            # unsupported head dim
