"""The C ABI's argument rules, drawn at random (CPU only).

Each case starts from a valid strided forward call (every extent >= 2, so
every stride is checked) and breaks exactly one rule the header states; the
call must return that rule's status code.  Every case is refused by the
host-side checks before the library makes any CUDA call, so no kernel is ever
launched (the pointers are fake addresses that are never dereferenced).  The
module is skipped where a CUDA device is visible: it tests host logic only.
"""
import ctypes
import math

import pytest
import torch

import exact_attention_fa2_gb300 as fa
from exact_attention_fa2_gb300 import build as fabuild

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="host-side argument checks only")

BASE = 1 << 24                    # fake, 16-byte aligned addresses, never dereferenced
RULES = ["negative size", "head dim", "dtype", "scale", "null pointer", "misaligned pointer",
         "stride not positive", "stride not 16 bytes", "no keys", "too many heads"]
EXPECT = {"negative size": -1, "head dim": -2, "dtype": -2, "scale": -1, "null pointer": -1,
          "misaligned pointer": -3, "stride not positive": -1, "stride not 16 bytes": -3, "no keys": -1,
          "too many heads": -2}
MESSAGE = {"negative size": "negative size", "head dim": "head dim", "dtype": "dtype", "scale": "scale",
           "null pointer": "is null", "misaligned pointer": "16-byte aligned", "stride not positive": "not positive",
           "stride not 16 bytes": "multiple of 16 bytes", "no keys": "no key rows", "too many heads": "B*H"}


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


case = st.fixed_dictionaries({
    "B": st.integers(2, 4), "H": st.integers(2, 4), "Sq": st.integers(2, 300), "Sk": st.integers(2, 300),
    "d": st.sampled_from([16, 32, 64, 80, 96, 128]), "dtype": st.sampled_from([0, 1]),
    "pad": st.integers(0, 4), "rule": st.sampled_from(RULES), "which": st.integers(0, 4),
    "dim": st.integers(0, 2), "bad": st.integers(1, 7), "causal": st.booleans(),
})


@settings(max_examples=300, deadline=None)
@given(case)
def test_one_broken_rule_gives_its_status(lib, c):
    B, H, Sq, Sk, d, dtype = c["B"], c["H"], c["Sq"], c["Sk"], c["d"], c["dtype"]
    elt = 2 if dtype == 0 else 4
    unit = 16 // elt                                   # elements per 16 bytes
    scale = 1.0 / math.sqrt(d)
    ptrs = [BASE * (i + 1) for i in range(5)]          # q, k, v, o, lse

    def strides(rows):
        rs = d + unit * c["pad"]                       # row stride: d plus whole 16-byte units
        return [H * rows * rs, rows * rs, rs]
    st_q, st_k, st_v, st_o = strides(Sq), strides(Sk), strides(Sk), strides(Sq)
    views = [st_q, st_k, st_v, st_o]

    rule = c["rule"]
    if rule == "negative size":
        B, H, Sq, Sk = [(-1 if i == c["which"] % 4 else x) for i, x in enumerate((B, H, Sq, Sk))]
    elif rule == "head dim":
        d = [0, 8, 48, 65, 112, 256][c["bad"] % 6]
    elif rule == "dtype":
        dtype = [2, -1, 7][c["bad"] % 3]
    elif rule == "scale":
        scale = [float("nan"), float("inf"), -float("inf")][c["bad"] % 3]
    elif rule == "null pointer":
        ptrs[c["which"]] = 0
    elif rule == "misaligned pointer":
        ptrs[c["which"]] += [1, 2, 4, 8][c["bad"] % 4]
    elif rule == "stride not positive":
        views[c["which"] % 4][c["dim"]] = [0, -unit, -1][c["bad"] % 3]
    elif rule == "stride not 16 bytes":
        views[c["which"] % 4][c["dim"]] += c["bad"] % (unit - 1) + 1     # 1..unit-1 extra elements
    elif rule == "no keys":
        Sk = 0
    elif rule == "too many heads":
        B, H = 300, 300                                # B*H > 65535 (element count kept small by Sq, Sk)
        Sq = Sk = 2
        views = [strides(2) for _ in range(4)]
    arr = [(ctypes.c_longlong * 3)(*v) for v in views]
    rc = lib.fa_fwd_strided(ctypes.c_void_p(ptrs[0]), arr[0], ctypes.c_void_p(ptrs[1]), arr[1],
                            ctypes.c_void_p(ptrs[2]), arr[2], ctypes.c_void_p(ptrs[3]), arr[3],
                            ctypes.c_void_p(ptrs[4]), B, H, Sq, Sk, d, int(c["causal"]),
                            ctypes.c_float(scale), dtype, None)
    msg = lib.fa_get_last_error().decode()
    assert rc == EXPECT[rule], (rule, rc, msg)
    assert MESSAGE[rule] in msg, (rule, msg)           # the refusal names the rule it applied
