"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no attention arithmetic. It only draws Q, K, V and dO from a
seeded CPU generator, in that order, with the shapes and value distributions of
the workloads below, and rounds them to the working dtype (round to nearest
even, as torch does).  Both the tests and the benchmark feed the same tensors to
the fp64 oracle (after an exact widening to float64) and to the CUDA library.

Workloads (B, H, S, d, dtype, causal, value scale), all self-attention with
N_q = N_k = S and scale = 1/sqrt(d):

* ``c1``  fp32  B1 H2  S128  d64,  causal and non-causal, N(0,1)
* ``c2``  bf16  B4 H12 S1024 d64,  causal, N(0,1)             (small-LM shape)
* ``c3``  bf16  B4 H16 S2048 d64,  causal and non-causal, N(0,1)
* ``c4``  bf16  B4 H32 S4096 d80,  causal, Q,K,V ~ 2*N(0,1), dO ~ N(0,1)
* ``c5``  sweep B1 H16, S = 128..65536, d in {16,32,64,128}, bf16/fp32, causal
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_inputs_rect", "sweep_points", "seed_for"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    d: int
    dtype: str            # "bf16" or "fp32"
    causal: tuple         # causal settings covered by this workload
    qkv_scale: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    "c1": Workload("c1", 1, 2, 128, 64, "fp32", (True, False), 1.0, 1001),
    "c2": Workload("c2", 4, 12, 1024, 64, "bf16", (True,), 1.0, 1002),
    "c3": Workload("c3", 4, 16, 2048, 64, "bf16", (True, False), 1.0, 1003),
    "c4": Workload("c4", 4, 32, 4096, 80, "bf16", (True,), 2.0, 1004),
}


def seed_for(S: int, d: int, dtype: str) -> int:
    """Seed of one point of the B1 H16 causal sweep."""
    return 1005 * 1_000_003 + S * 1009 + d * 17 + (0 if dtype == "bf16" else 1)


def sweep_points(max_S: int = 65536):
    """The causal B1 H16 sweep: S = 2^7..2^16, d in {16,32,64,128}, bf16 and fp32."""
    pts = []
    for dtype in ("bf16", "fp32"):
        for d in (16, 32, 64, 128):
            S = 128
            while S <= max_S:
                pts.append(Workload(f"c5_{dtype}_S{S}_d{d}", 1, 16, S, d, dtype,
                                    (True,), 1.0, seed_for(S, d, dtype)))
                S *= 2
    return pts


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def make_inputs(B: int, H: int, S: int, d: int, dtype: str = "bf16", seed: int = 0,
                qkv_scale: float = 1.0, do_scale: float = 1.0):
    """Draw (Q, K, V, dO) as contiguous CPU tensors of shape [B, H, S, d].

    Values are fp32 N(0,1) draws from ``torch.Generator`` seeded with ``seed``,
    drawn in the order Q, K, V, dO, multiplied by ``qkv_scale`` (Q, K, V) or
    ``do_scale`` (dO), then rounded to ``dtype``.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, S, d)
    tdt = torch_dtype(dtype)
    out = []
    for i in range(4):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        x.mul_(qkv_scale if i < 3 else do_scale)
        out.append(x.to(tdt).contiguous())
    return tuple(out)


def make_inputs_rect(B: int, H: int, Sq: int, Sk: int, d: int, dtype: str = "bf16", seed: int = 0):
    """(Q, K, V, dO) for N_q = Sq queries and N_k = Sk keys: Q, dO of shape
    [B, H, Sq, d] and K, V of shape [B, H, Sk, d], N(0,1) draws in the order
    Q, K, V, dO from one seeded generator, rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    tdt = torch_dtype(dtype)
    shapes = ((B, H, Sq, d), (B, H, Sk, d), (B, H, Sk, d), (B, H, Sq, d))
    return tuple(torch.randn(sh, generator=g, dtype=torch.float32).to(tdt).contiguous() for sh in shapes)


def make_workload_inputs(w: Workload):
    return make_inputs(w.B, w.H, w.S, w.d, w.dtype, w.seed, w.qkv_scale)
