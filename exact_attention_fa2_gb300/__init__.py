"""Python binding of the GB300 exact-attention library (``libfa_gb300.so``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/fa_gb300.h``.  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: if the
library has not been built, or the tensors are not on a CUDA device, the calls
raise.

Layout: q, k, v, o, dO, dq, dk, dv are contiguous [B, H, S, d] tensors
(bfloat16 or float32); lse is [B, H, S] float32 (natural log).

The autograd contract follows the "CS336 Assignment 2: Systems" FlashAttention-2
section and the handout's problem flash_forward: forward(Q, K, V, is_causal)
returns O and saves L, Q, K, V, O; backward(dO) returns dQ, dK, dV.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = [
    "FAError", "library_path", "load_library", "fa_fwd", "fa_bwd", "fa_bwd_deterministic", "fwd", "bwd",
    "bwd_workspace_size", "check_status", "attention", "FlashAttention", "version",
    "FA_BF16", "FA_FP32", "profile_enable", "profile_read",
]

FA_BF16 = 0
FA_FP32 = 1
FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", -1: "FA_ERR_INVALID_ARG", -2: "FA_ERR_UNSUPPORTED", -3: "FA_ERR_MISALIGNED",
    -4: "FA_ERR_WORKSPACE", -5: "FA_ERR_CUDA", -6: "FA_ERR_DEVICE_TIMEOUT", -7: "FA_ERR_DEVICE_BOUNDS",
}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_FILE = os.path.join(_PKG, "libfa_gb300.so")
_lib = None
_lock = threading.Lock()


class FAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_FILE


def load_library():
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_FILE):
            raise RuntimeError(
                f"{_LIB_FILE} is missing: build it with `python -m exact_attention_fa2_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(_LIB_FILE)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_deterministic.argtypes = lib.fa_bwd.argtypes
        lib.fa_bwd_deterministic.restype = i
        lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_get_last_error.argtypes = []
        lib.fa_get_last_error.restype = ctypes.c_char_p
        lib.fa_check_status.argtypes = [vp]
        lib.fa_check_status.restype = i
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i
        lib.fa_profile_enable.argtypes = [i]
        lib.fa_profile_enable.restype = i
        lib.fa_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
        lib.fa_profile_read.restype = i
        lib.fa_fwd_partial.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_partial.restype = i
        lib.fa_merge.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
        lib.fa_merge.restype = i
        lib.fa_fwd_bwd_host_buffer_size.argtypes = [i, i, i, i, i]
        lib.fa_fwd_bwd_host_buffer_size.restype = sz
        lib.fa_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_bwd_host.restype = i
        lib.fa_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, vp]
        lib.fa_selftest_bounded_wait.restype = i
        lib.fa_fwd_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_strided.restype = i
        lib.fa_bwd_strided.argtypes = ([vp] * 17 + [vp, sz] + [i, i, i, i, i, i, f, i, i, vp])
        lib.fa_bwd_strided.restype = i
        _lib = lib
    return _lib


def _check(rc: int):
    if rc != FA_OK:
        raise FAError(rc, load_library().fa_get_last_error().decode(errors="replace"))


def version() -> int:
    return load_library().fa_version()


PROFILE_KINDS = ("fwd", "bwd_preprocess", "bwd_main", "dq_convert", "dq_pass")


def profile_enable(on: bool = True):
    """Start or stop per-kernel CUDA-event timing inside the library."""
    _check(load_library().fa_profile_enable(1 if on else 0))


def profile_read():
    """{kind: (total_ms, launches)} for the kernels timed since the last read."""
    ms = (ctypes.c_double * len(PROFILE_KINDS))()
    n = (ctypes.c_int * len(PROFILE_KINDS))()
    _check(load_library().fa_profile_read(ms, n))
    return {k: (ms[i], n[i]) for i, k in enumerate(PROFILE_KINDS)}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device_index=None) -> int:
    """cudaStream_t of `stream` (a torch stream or an int); None = the current
    stream of `device_index` (default: the current device)."""
    if stream is None:
        if device_index is None:
            device_index = torch.cuda.current_device()
        if _raw_stream is not None:
            return int(_raw_stream(device_index))
        stream = torch.cuda.current_stream(device_index)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_qkv(*ts):
    """q, k, v (then o, dO): [B, H, N, d] CUDA tensors of one dtype and device
    with a contiguous head dimension; q (o, dO) share N_q, k and v share N_k.
    Other strides are passed to the library, which checks their alignment.
    Returns the device index."""
    q = ts[0]
    dev = q.get_device()
    if dev < 0:
        raise ValueError("tensors must be on a CUDA device (there is no CPU fallback)")
    qs, ks = q.shape, ts[1].shape
    if len(qs) != 4 or len(ks) != 4 or ks[0] != qs[0] or ks[1] != qs[1] or ks[3] != qs[3]:
        raise ValueError("q, o, dO must be [B, H, N_q, d] and k, v [B, H, N_k, d]")
    dt = q.dtype
    for i, t in enumerate(ts):
        if t.dtype is not dt or t.get_device() != dev:
            raise ValueError("q, k, v (and o, dO) must share dtype and CUDA device")
        if t.shape != (ks if i in (1, 2) else qs):
            raise ValueError("q, o, dO must be [B, H, N_q, d] and k, v [B, H, N_k, d]")
        if t.stride(-1) != 1:
            raise ValueError("the head dimension (last) must be contiguous")
    return dev


def _plain(*ts):
    """True when the plain (contiguous, N_q = N_k) entry points apply."""
    return all(t.is_contiguous() for t in ts) and ts[0].shape == ts[1].shape


def _strides(t):
    return (ctypes.c_longlong * 3)(t.stride(0), t.stride(1), t.stride(2))


def fa_fwd(q, k, v, o, lse, B, H, S, d, causal, scale, dtype, stream) -> int:
    """Raw C-ABI call on device pointers (ints or ctypes pointers); returns the status."""
    return load_library().fa_fwd(q, k, v, o, lse, B, H, S, d, int(causal), float(scale), dtype, stream)


def fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, ws, ws_bytes, B, H, S, d, causal, scale, dtype, stream) -> int:
    """Raw C-ABI call on device pointers; returns the status."""
    return load_library().fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, ws, ws_bytes, B, H, S, d,
                                 int(causal), float(scale), dtype, stream)


def fa_bwd_deterministic(q, k, v, o, dO, lse, dq, dk, dv, ws, ws_bytes, B, H, S, d, causal, scale, dtype,
                         stream) -> int:
    """Raw C-ABI call of the deterministic backward on device pointers; returns the status."""
    return load_library().fa_bwd_deterministic(q, k, v, o, dO, lse, dq, dk, dv, ws, ws_bytes, B, H, S, d,
                                               int(causal), float(scale), dtype, stream)


def bwd_workspace_size(B: int, H: int, S: int, d: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (FA_BF16 if dtype == torch.bfloat16 else FA_FP32)
    return int(load_library().fa_bwd_workspace_size(B, H, S, d, code))


def check_status(stream=None):
    """Synchronise the stream and raise if a kernel reported a device-side error."""
    _check(load_library().fa_check_status(ctypes.c_void_p(_stream_handle(stream))))


def fwd(q, k, v, causal: bool = False, scale=None, out=None, lse=None, stream=None):
    """Forward pass; returns (o, lse)."""
    dev = _check_qkv(q, k, v)
    if dev != torch.cuda.current_device():
        with torch.cuda.device(dev):
            return fwd(q, k, v, causal, scale, out, lse, stream)
    B, H, S, d = q.shape
    Sk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        o = torch.empty_like(q)
    else:
        o = out
        _check_qkv(q, k, v, o)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    elif not lse.is_contiguous() or lse.dtype is not torch.float32 or tuple(lse.shape) != (B, H, S):
        raise ValueError("lse must be a contiguous fp32 [B, H, N_q] tensor")
    lib = _lib or load_library()
    st = _stream_handle(stream, dev)
    code = _dtype_code(q)
    if _plain(q, k, v, o):
        rc = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, S, d,
                        int(causal), scale, code, st)
    else:
        rc = lib.fa_fwd_strided(
            q.data_ptr(), _strides(q), k.data_ptr(), _strides(k), v.data_ptr(), _strides(v), o.data_ptr(),
            _strides(o), lse.data_ptr(), B, H, S, Sk, d, int(causal), scale, code, st)
    if rc:
        _check(rc)
    return o, lse


def bwd(q, k, v, o, do, lse, causal: bool = False, scale=None, workspace=None, stream=None,
        out=None, deterministic: bool = False):
    """Backward pass; returns (dq, dk, dv).  ``workspace`` (uint8, >= the size
    reported by bwd_workspace_size) is allocated here when not given.
    ``deterministic`` selects fa_bwd_deterministic: dQ from its own
    query-tile-outer pass, bitwise reproducible."""
    dev = _check_qkv(q, k, v, o, do)
    if dev != torch.cuda.current_device():
        with torch.cuda.device(dev):
            return bwd(q, k, v, o, do, lse, causal, scale, workspace, stream, out, deterministic)
    B, H, S, d = q.shape
    Sk = k.shape[2]
    if lse.dtype is not torch.float32 or not lse.is_contiguous() or lse.numel() != B * H * S or lse.get_device() != dev:
        raise ValueError("lse must be the forward's contiguous fp32 [B, H, N_q] tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    code = _dtype_code(q)
    lib = _lib or load_library()
    if workspace is None:
        need = int(lib.fa_bwd_workspace_size(B, H, S, d, code))
        workspace = torch.empty(max(need, 256), device=q.device, dtype=torch.uint8)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
        _check_qkv(dq, dk, dv, q, q)
    st = _stream_handle(stream, dev)
    nbytes = workspace.numel() * workspace.element_size()
    if _plain(q, k, v, o, do, dq, dk, dv):
        entry = lib.fa_bwd_deterministic if deterministic else lib.fa_bwd
        rc = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                   dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), nbytes, B, H, S, d,
                   int(causal), scale, code, st)
    else:
        rc = lib.fa_bwd_strided(
            q.data_ptr(), _strides(q), k.data_ptr(), _strides(k), v.data_ptr(), _strides(v), o.data_ptr(),
            _strides(o), do.data_ptr(), _strides(do), lse.data_ptr(), dq.data_ptr(), _strides(dq), dk.data_ptr(),
            _strides(dk), dv.data_ptr(), _strides(dv), workspace.data_ptr(), nbytes, B, H, S, Sk, d, int(causal),
            scale, code, int(bool(deterministic)), st)
    if rc:
        _check(rc)
    return dq, dk, dv


def fwd_partial(q, k, v, key_begin: int, key_end: int, causal: bool = False, scale=None, out=None, stream=None):
    """Attention of every query over keys [key_begin, key_end) only (causal
    positions are whole-sequence positions); returns (o_part fp32, lse_part
    fp32), with o = 0 and lse = -inf where a query has no admissible key."""
    _check_qkv(q, k, v)
    if not _plain(q, k, v):
        raise ValueError("fwd_partial takes contiguous q, k, v of one length")
    B, H, S, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        o = torch.empty((B, H, S, d), device=q.device, dtype=torch.float32)
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    else:
        o, lse = out
    with torch.cuda.device(q.device):
        rc = load_library().fa_fwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, S, d,
                                           int(key_begin), int(key_end), int(causal), scale, _dtype_code(q),
                                           ctypes.c_void_p(_stream_handle(stream)))
    _check(rc)
    return o, lse


def merge(o_a, lse_a, o_b, lse_b, dtype=torch.bfloat16, out=None, stream=None):
    """Exact merge of two partial results over disjoint key sets: returns
    (o in ``dtype``, lse fp32)."""
    B, H, S, d = o_a.shape
    for t in (o_a, o_b):
        if t.dtype != torch.float32 or t.shape != o_a.shape or not t.is_contiguous():
            raise ValueError("partial outputs must be contiguous fp32 [B, H, S, d] tensors")
    if out is None:
        o = torch.empty((B, H, S, d), device=o_a.device, dtype=dtype)
        lse = torch.empty((B, H, S), device=o_a.device, dtype=torch.float32)
    else:
        o, lse = out
    with torch.cuda.device(o_a.device):
        rc = load_library().fa_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o), _ptr(lse),
                                     B, H, S, d, _dtype_code(o), ctypes.c_void_p(_stream_handle(stream)))
    _check(rc)
    return o, lse


def fwd_bwd_host_buffer_size(B: int, H: int, S: int, d: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (FA_BF16 if dtype == torch.bfloat16 else FA_FP32)
    return int(load_library().fa_fwd_bwd_host_buffer_size(B, H, S, d, code))


def fwd_bwd_host(q, k, v, do, out, dev_buf, causal: bool = False, scale=None, stream=None):
    """One forward + backward step on host tensors (pinned for asynchronous
    copies): ``out`` = (o, lse, dq, dk, dv) host tensors that receive the
    results, ``dev_buf`` a uint8 device tensor of at least
    fwd_bwd_host_buffer_size() bytes.  Returns immediately; the results are
    valid once ``stream`` (default: the current stream of dev_buf's device)
    has completed."""
    for t in (q, k, v, do):
        if t.is_cuda or t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("q, k, v, dO must be contiguous host tensors of one shape and dtype")
    if q.dim() != 4:
        raise ValueError("expected [B, H, S, d] tensors")
    o, lse, dq, dk, dv = out
    B, H, S, d = q.shape
    for t in (o, dq, dk, dv):
        if t.is_cuda or t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("o, dq, dk, dv must be contiguous host tensors like q")
    if lse.is_cuda or lse.shape != (B, H, S) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 host tensor of shape [B, H, S]")
    if not dev_buf.is_cuda:
        raise ValueError("dev_buf must be a device tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(dev_buf.device):
        st = _stream_handle(stream)
        rc = load_library().fa_fwd_bwd_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(dev_buf), dev_buf.numel() * dev_buf.element_size(), B, H, S, d, int(causal), scale,
            _dtype_code(q), ctypes.c_void_p(st))
    _check(rc)


class FlashAttention(torch.autograd.Function):
    """O = softmax(Q K^T * scale) V with the recompute backward."""

    @staticmethod
    def forward(ctx, q, k, v, is_causal=False, scale=None, deterministic=False):
        o, lse = fwd(q, k, v, is_causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.is_causal = bool(is_causal)
        ctx.scale = scale
        ctx.deterministic = bool(deterministic)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, do.contiguous(), lse, ctx.is_causal, ctx.scale,
                         deterministic=ctx.deterministic)
        return dq, dk, dv, None, None, None


def attention(q, k, v, causal: bool = False, scale=None, deterministic: bool = False):
    """Differentiable attention; ``deterministic`` makes the backward bitwise reproducible."""
    return FlashAttention.apply(q, k, v, causal, scale, deterministic)
