"""Seeded synthetic inputs for C = A @ B.

This module only draws and rounds input matrices; it holds none of the
product's arithmetic.  Both the GPU library's tests and the CPU oracle's
checks take their inputs from here, so the two sides always see the same
already-rounded values.

Recipe (shared by every workload): a ``torch.Generator`` seeded with the
workload's seed draws A first and then B, in FP32 on the CPU; the FP32 values
are then rounded to the input storage type with round-to-nearest-even
(``Tensor.to``).

Workloads:

* ``worked_9x9`` -- the 9 x 9 worked example of "Tiled Matrix Multiplication"
  (shared-memory section): A[i][j] = 9i + j and B = 2A, FP32, 3 x 3 tiles.
* ``square_128_f16`` -- 128^3, FP16 inputs uniform on [-1, 1] (seed 0), FP32
  output; the shape of the traffic example in "Reading a matrix multiply
  through its tiles" ("Count the repeated reads").
* ``edge_96x200x1000_bf16`` -- 96 x 200 x 1000, BF16 inputs N(0, 1) (seed 1),
  FP32 output: partial tiles in every dimension ("Edge tiles still matter").
* ``square_4096_f16`` -- 4096^3, FP16 inputs uniform on [-1, 1] (seed 2), FP16
  output.
* ``square_8192_bf16`` -- 8192^3, BF16 inputs N(0, 1) / sqrt(K) (seed 3), both
  A and B scaled in FP32 before rounding, BF16 output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    in_dtype: str
    out_dtype: str
    dist: str          # "worked", "uniform", "positive", "normal_scaled", "normal", "int"
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w
    for w in (
        Workload("worked_9x9", 9, 9, 9, "f32", "f32", "worked", 0),
        Workload("square_128_f16", 128, 128, 128, "f16", "f32", "uniform", 0),
        Workload("edge_96x200x1000_bf16", 96, 200, 1000, "bf16", "f32", "normal", 1),
        Workload("square_4096_f16", 4096, 4096, 4096, "f16", "f16", "uniform", 2),
        Workload("square_8192_bf16", 8192, 8192, 8192, "bf16", "bf16", "normal_scaled", 3),
    )
}


def worked_example() -> tuple[torch.Tensor, torch.Tensor]:
    """A[i][j] = 9i + j and B = 2A (9 x 9, FP32)."""
    idx = torch.arange(81, dtype=torch.float32).reshape(9, 9)
    return idx.clone(), 2 * idx


def draw(M: int, N: int, K: int, in_dtype: str, dist: str, seed: int,
         lo: int = -4, hi: int = 4) -> tuple[torch.Tensor, torch.Tensor]:
    """Draw A (M x K) then B (K x N) in FP32 with one seeded generator and
    round both to ``in_dtype``.

    dist: "uniform" U[-1, 1]; "positive" U[0, 1] (every product the same
    sign); "normal" N(0, 1); "normal_scaled" N(0, 1)/sqrt(K); "int" integers
    uniform on [lo, hi] (exact in every input type).
    """
    g = torch.Generator().manual_seed(seed)
    shapes = ((M, K), (K, N))
    mats = []
    for shape in shapes:
        if dist == "uniform":
            x = torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
        elif dist == "positive":
            x = torch.rand(shape, generator=g, dtype=torch.float32)
        elif dist == "normal":
            x = torch.randn(shape, generator=g, dtype=torch.float32)
        elif dist == "normal_scaled":
            x = torch.randn(shape, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(max(K, 1)))
        elif dist == "int":
            x = torch.randint(lo, hi + 1, shape, generator=g).to(torch.float32)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        mats.append(x.to(DTYPES[in_dtype]).contiguous())
    return mats[0], mats[1]


def make(w: Workload | str) -> tuple[torch.Tensor, torch.Tensor]:
    """The rounded CPU inputs (A, B) of a named workload."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if w.dist == "worked":
        return worked_example()
    return draw(w.M, w.N, w.K, w.in_dtype, w.dist, w.seed)
