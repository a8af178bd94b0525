"""Seeded synthetic inputs for dense C = A x B.

This module only draws random matrices; it holds none of the product's
arithmetic. It is the one module that the CUDA path's tests and benchmark and
the CPU oracle's checks both take their inputs from, so the two sides always
see identical values.

All draws happen on a CPU ``torch.Generator`` (seed = 20260 + workload index)
so every machine sees the same values; callers copy them to the device.

The workloads are the shapes the library is measured and checked on:

==========  =====================  ==========================================
name        M x N x K              values
==========  =====================  ==========================================
int128      128 x 128 x 128        integers uniform on {-4..4}, stored fp32
u1024       1024 x 1024 x 1024     uniform[-1, 1] fp32
n4096       4096 x 4096 x 4096     normal(0, 1) fp32 (FP32 path and TF32 path)
ragged      3000 x 5001 x 1537     uniform[-1, 1] fp32, packed lda=K, ldb=N
ffn_bf16    8192 x 14336 x 4096    bf16 rounded (RNE) from normal(0, 0.02)
skinny_bf16 16 x 14336 x 4096      bf16 rounded (RNE) from normal(0, 0.02)
skinny_f32  16 x 14336 x 4096      normal(0, 1) fp32 (FP32 path and TF32 path)
==========  =====================  ==========================================

The last two are the FFN shape with only 16 rows (16 tokens): the product is
bound by reading B once from memory, not by arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import torch

SEED_BASE = 20260


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    M: int
    N: int
    K: int
    dist: str            # "int4", "uniform", "normal", "normal002"
    dtype: str           # storage type of A and B: "f32" or "bf16"
    paths: Tuple[str, ...]
    check_rows: Optional[int] = None   # rows the oracle checks (None = all)
    description: str = ""

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    w.name: w for w in [
        Workload(0, "int128", 128, 128, 128, "int4", "f32", ("f32",),
                 description="square 128^3, integers in {-4..4} stored fp32"),
        Workload(1, "u1024", 1024, 1024, 1024, "uniform", "f32", ("f32",),
                 description="square 1024^3, uniform[-1,1] fp32"),
        Workload(2, "n4096", 4096, 4096, 4096, "normal", "f32", ("f32", "tf32"),
                 description="square 4096^3, normal(0,1) fp32"),
        Workload(3, "ragged", 3000, 5001, 1537, "uniform", "f32", ("f32",),
                 description="3000x5001x1537 uniform[-1,1] fp32, lda=K, ldb=N, ldc=N"),
        Workload(4, "ffn_bf16", 8192, 14336, 4096, "normal002", "bf16", ("bf16",),
                 check_rows=256,
                 description="FFN-shaped M=8192 tokens, K=4096, N=14336, bf16 inputs"),
        Workload(5, "skinny_bf16", 16, 14336, 4096, "normal002", "bf16", ("bf16",),
                 description="few rows: M=16 tokens, K=4096, N=14336, bf16 inputs"),
        Workload(6, "skinny_f32", 16, 14336, 4096, "normal", "f32", ("f32", "tf32"),
                 description="few rows: M=16, K=4096, N=14336, normal(0,1) fp32"),
    ]
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw(rows: int, cols: int, dist: str, g: torch.Generator) -> torch.Tensor:
    """A packed rows x cols fp32 matrix drawn from ``dist`` with generator ``g``."""
    shape = (rows, cols)
    if dist == "int4":
        return torch.randint(-4, 5, shape, generator=g, dtype=torch.int64).to(torch.float32)
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "normal002":
        return torch.randn(shape, generator=g, dtype=torch.float32) * 0.02
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def matrix(rows: int, cols: int, dist: str, seed: int, dtype: str = "f32",
           ld: Optional[int] = None, pad_value: float = float("nan"),
           g: Optional[torch.Generator] = None) -> torch.Tensor:
    """A rows x cols matrix as a row-major view with leading dimension ``ld``.

    With ``ld > cols`` the columns between ``cols`` and ``ld`` hold
    ``pad_value`` (NaN by default), so any read of the padding poisons a
    result that uses it.
    """
    if g is None:
        g = generator(seed)
    x = draw(rows, cols, dist, g)
    if dtype == "bf16":
        x = x.to(torch.bfloat16)        # round to nearest even
    elif dtype != "f32":
        raise ValueError(f"unknown storage type {dtype!r}")
    if ld is None or ld == cols:
        return x.contiguous()
    if ld < cols:
        raise ValueError("ld must be >= cols")
    store = torch.full((max(rows, 1), ld), pad_value, dtype=x.dtype)
    store[:rows, :cols] = x
    return store[:rows, :cols]


def operands(w: Workload) -> Tuple[torch.Tensor, torch.Tensor]:
    """Host A (M x K) and B (K x N) of workload ``w``; A is drawn first."""
    g = generator(w.seed)
    A = matrix(w.M, w.K, w.dist, w.seed, w.dtype, g=g)
    B = matrix(w.K, w.N, w.dist, w.seed, w.dtype, g=g)
    return A, B


def check_rows(w: Workload) -> torch.Tensor:
    """Row indices of C the oracle checks: all rows, or a seeded sample.

    The sample is the first ``check_rows`` entries of a permutation of
    0..M-1 drawn with its own generator (seed + 1000), so it does not depend
    on how the operands were drawn.
    """
    if w.check_rows is None:
        return torch.arange(w.M)
    g = generator(w.seed + 1000)
    return torch.randperm(w.M, generator=g)[: w.check_rows].sort().values


def sample_indices(M: int, N: int, count: int, seed: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """``count`` seeded (row, col) positions, always including the four corners."""
    g = generator(seed)
    r = torch.randint(0, max(M, 1), (count,), generator=g)
    c = torch.randint(0, max(N, 1), (count,), generator=g)
    corners_r = torch.tensor([0, 0, M - 1, M - 1])
    corners_c = torch.tensor([0, N - 1, 0, N - 1])
    return torch.cat([corners_r, r]), torch.cat([corners_c, c])
