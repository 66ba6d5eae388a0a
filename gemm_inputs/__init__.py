"""Seeded synthetic inputs for the GEMM C = epi(A . B^T).

This module is the only code that both the oracle-side tests and the CUDA
path use.  It holds no part of the method's arithmetic: it draws random
numbers with a seeded CPU ``torch.Generator`` and casts them (round to
nearest even) to fp16/bf16.  Both sides then consume the same bit patterns.

Draw recipe (one generator per workload, seeded with the workload's seed):
A (or X) is drawn first, then B (or W).  Uniform entries are
``torch.rand * (hi - lo) + lo``; normal entries are ``torch.randn * std``;
integer entries are ``torch.randint(lo, hi + 1)`` (exact in fp16/bf16).

The workloads are the problem shapes named for this GEMM: 256^3, 4096^3,
8192^3 fp16; the bf16 3072x16384x4096 tanh-GELU layer (6 x 512 tokens x
hidden 4096, the tensor shape of the XLA:GPU emitters page's GELU example);
the ragged 4095x4097x8191 and skinny 64x8192x8192 fp16 shapes; and the
16896x512x640 shape of the Mosaic GPU pipelining guide's Hopper example.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str            # "f16" | "bf16"
    epilogue: str         # "none" | "gelu"
    dist: str             # "uniform" | "normal_scaled" | "normal_xw" | "uniform01" | "int"
    seed: int
    lo: float = -1.0
    hi: float = 1.0
    description: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    "gemm_256_f16": Workload("gemm_256_f16", 256, 256, 256, "f16", "none", "uniform", 0,
                             description="fp16 256^3, U[-1,1], seed 0"),
    "gemm_256_f16_int": Workload("gemm_256_f16_int", 256, 256, 256, "f16", "none", "int", 0,
                                 lo=-2, hi=2,
                                 description="fp16 256^3, integers U{-2..2}, seed 0 (drawn after "
                                             "the float pair)"),
    "gemm_4096_f16": Workload("gemm_4096_f16", 4096, 4096, 4096, "f16", "none", "normal_scaled", 1,
                              description="fp16 4096^3, N(0,1)/sqrt(K), seed 1"),
    "gemm_8192_f16": Workload("gemm_8192_f16", 8192, 8192, 8192, "f16", "none", "normal_scaled", 2,
                              description="fp16 8192^3, N(0,1)/sqrt(K), seed 2"),
    "gelu_3072x16384x4096_bf16": Workload(
        "gelu_3072x16384x4096_bf16", 3072, 16384, 4096, "bf16", "gelu", "normal_xw", 3,
        description="bf16 Y=gelu_tanh(X.W^T), X[3072,4096]~N(0,1), W[16384,4096]~N(0,0.02), seed 3"),
    "ragged_4095x4097x8191_f16": Workload(
        "ragged_4095x4097x8191_f16", 4095, 4097, 8191, "f16", "none", "uniform", 4,
        description="fp16 4095x4097x8191, U[-1,1], seed 4"),
    "skinny_64x8192x8192_f16": Workload(
        "skinny_64x8192x8192_f16", 64, 8192, 8192, "f16", "none", "uniform", 4,
        description="fp16 64x8192x8192, U[-1,1], seed 4"),
    "mosaic_16896x512x640_f16": Workload(
        "mosaic_16896x512x640_f16", 16896, 512, 640, "f16", "none", "uniform01", 42,
        lo=0.0, hi=1.0, description="fp16 16896x512x640, U[0,1), seed 42"),
}


def _draw(gen: torch.Generator, rows: int, cols: int, w: Workload, which: str) -> torch.Tensor:
    shape = (rows, cols)
    if w.dist in ("uniform", "uniform01"):
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * (w.hi - w.lo) + w.lo
    elif w.dist == "normal_scaled":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) / math.sqrt(w.K)
    elif w.dist == "normal_xw":
        std = 1.0 if which == "A" else 0.02
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * std
    elif w.dist == "int":
        x = torch.randint(int(w.lo), int(w.hi) + 1, shape, generator=gen).to(torch.float32)
    else:
        raise ValueError(w.dist)
    return x.to(_TORCH_DT[w.dtype])


def make(w: Workload | str, M: Optional[int] = None, N: Optional[int] = None,
         K: Optional[int] = None, seed: Optional[int] = None):
    """Return (A, B) as CPU torch tensors of the workload's dtype.

    M/N/K/seed override the workload's own (same distribution), which the
    tests use to draw small cases of a workload's recipe."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if M is not None or N is not None or K is not None or seed is not None:
        w = dataclasses.replace(w, M=M if M is not None else w.M, N=N if N is not None else w.N,
                                K=K if K is not None else w.K,
                                seed=seed if seed is not None else w.seed)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    if w.dist == "int" and w.name == "gemm_256_f16_int":
        # The integer copy is the second draw of seed 0: skip the float pair.
        base = WORKLOADS["gemm_256_f16"]
        _draw(gen, w.M, w.K, base, "A")
        _draw(gen, w.N, w.K, base, "B")
    A = _draw(gen, w.M, w.K, w, "A")
    B = _draw(gen, w.N, w.K, w, "B")
    return A, B


def custom(M: int, N: int, K: int, dtype: str = "f16", dist: str = "uniform", seed: int = 0,
           lo: float = -1.0, hi: float = 1.0, epilogue: str = "none"):
    """Draw (A, B) for an arbitrary shape with one of the recipes above."""
    w = Workload("custom", M, N, K, dtype, epilogue, dist, seed, lo=lo, hi=hi)
    return make(w)


def bias(N: int, dtype: str = "f16", seed: int = 0, dist: str = "uniform", lo: float = -0.5,
         hi: float = 0.5) -> torch.Tensor:
    """A seeded per-column bias vector of N values, cast to fp16/bf16 with RNE.

    dist "uniform": U[lo, hi] (default U[-0.5, 0.5], the scale of a Linear
    layer's bias next to the GELU workload's pre-activations of std 1.28);
    "int": integers U{lo..hi}, exact in both formats for the bit-exact tests.
    The generator is seeded separately from the operands' (seed + 1000003).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 1000003)
    td = torch.bfloat16 if dtype == "bf16" else torch.float16
    if dist == "int":
        v = torch.randint(int(lo), int(hi) + 1, (N,), generator=gen).to(torch.float32)
    else:
        v = torch.rand(N, generator=gen, dtype=torch.float32) * (hi - lo) + lo
    return v.to(td)
