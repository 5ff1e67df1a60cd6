"""Compile the CUDA library ``libfa_gb300.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled to an object file in parallel with nvcc, then
the objects are linked into a shared library with the CUDA runtime linked
statically (the library then needs only the driver, ``libcuda.so``, at run
time, and loads on a machine without a GPU).

    python -m exact_attention_fa2_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build " + LIB_NAME)
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                               + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")
    if verbose and r.stdout.strip():
        print(r.stdout, flush=True)
    return r.stdout


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Build the library if any source is newer than it; return its path."""
    if not force and _up_to_date():
        return LIB_PATH
    os.makedirs(OBJ_DIR, exist_ok=True)
    nv = nvcc()
    jobs = []
    for src in _sources():
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
        jobs.append((src, obj, [nv, *ARCH, *CFLAGS, *extra_flags, "-c", src, "-o", obj]))
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        list(ex.map(lambda j: _run(j[2], verbose), jobs))
    tmp = LIB_PATH + ".tmp"
    _run([nv, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[j[1] for j in jobs],
          "-ldl", "-lpthread", "-lrt"], verbose)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
