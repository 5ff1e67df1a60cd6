"""The product path has no CPU fallback and never reaches the oracle (CPU only).

The Python binding refuses tensors that are not on a CUDA device, raises when
the compiled library is missing, and neither it nor the CUDA sources import
or name the oracle package.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

import exact_attention_fa2_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "exact_attention_fa2_gb300")


def cpu_qkv(dtype=torch.bfloat16):
    return [torch.zeros(1, 2, 128, 64, dtype=dtype) for _ in range(4)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cpu_tensors_are_refused(dtype):
    q, k, v, do = cpu_qkv(dtype)
    with pytest.raises(ValueError, match="no CPU fallback"):
        fa.fwd(q, k, v, True)
    lse = torch.zeros(1, 2, 128)
    with pytest.raises(ValueError, match="no CPU fallback"):
        fa.bwd(q, k, v, q, do, lse, True)
    with pytest.raises(ValueError, match="no CPU fallback"):
        fa.attention(q, k, v, True)


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "_LIB_FILE", str(tmp_path / "libfa_gb300.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        fa.load_library()


def test_package_import_leaves_the_oracle_unloaded():
    from exact_attention_fa2_gb300 import build as fabuild
    fabuild.build()
    code = ("import sys, exact_attention_fa2_gb300 as fa, exact_attention_fa2_gb300.build; "
            "fa.load_library(); "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "assert not bad, bad")
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]


def test_product_sources_do_not_name_the_oracle():
    # an import of the package or an attribute of it (prose that mentions the oracle is fine)
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b)|\boracle\.[A-Za-z_]", re.M)
    offenders = []
    for dirpath, _dirs, files in os.walk(PKG):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                path = os.path.join(dirpath, fn)
                if pat.search(open(path, encoding="utf-8").read()):
                    offenders.append(os.path.relpath(path, ROOT))
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if pat.search(open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()):
            offenders.append(os.path.join("include", fn))
    assert not offenders, offenders
