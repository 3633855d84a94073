"""Seeded synthetic operands for the GEMM workloads.

This module is the one piece shared by the CUDA path's tests/benchmark and the
oracle's: it draws numbers and lays them out, and holds none of the GEMM's
arithmetic.

Recipe (the workloads state a distribution and a seed, not a generator; this
is the reading used everywhere in this project):

* a CPU ``torch.Generator`` seeded with ``seed``;
* A (M x K) is drawn first, then the logical K x N matrix B, from the same
  generator, row-major order;
* ``uniform`` means ``U[-1, 1)`` as ``2*rand - 1``; ``normal`` means
  ``N(0, sigma^2)`` as ``sigma*randn``;
* a column-major B stores the same logical matrix transposed (array shape
  (N, K), element (k, j) at ``j*K + k``, the corner-turning layout of "PMPP
  Chapter 06: Performance considerations", section 1), so values do not
  depend on the layout;
* BF16 operands are the FP32 draws rounded to nearest-even BF16.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

B_ROW_MAJOR = 0
B_COL_MAJOR = 1

# dtype names used by the library's ABI
F32 = "f32"
TF32 = "tf32"
BF16 = "bf16"
F32X3 = "f32x3"  # FP32 operands, FP32-accurate product on the tensor cores


@dataclass(frozen=True)
class Workload:
    """One named GEMM workload: shape, B layout, value distribution, seed."""
    name: str
    M: int
    N: int
    K: int
    layout_b: int
    dist: str
    seed: int
    sigma: float = 1.0
    dtype: str = F32

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads this library is specified and measured on.
WORKLOADS = {
    "fp32_128_row": Workload("fp32_128_row", 128, 128, 128, B_ROW_MAJOR, "uniform", 0),
    "fp32_1024_colB": Workload("fp32_1024_colB", 1024, 1024, 1024, B_COL_MAJOR, "uniform", 1),
    "fp32_4095x3073x2047_row": Workload("fp32_4095x3073x2047_row", 4095, 3073, 2047,
                                        B_ROW_MAJOR, "normal", 2, 1.0),
    "fp32_8192_row": Workload("fp32_8192_row", 8192, 8192, 8192, B_ROW_MAJOR, "uniform", 3),
    "ffn_bf16_8192x14336x4096": Workload("ffn_bf16_8192x14336x4096", 8192, 14336, 4096,
                                         B_ROW_MAJOR, "normal", 4, 0.02, BF16),
    "ffn_tf32_8192x14336x4096": Workload("ffn_tf32_8192x14336x4096", 8192, 14336, 4096,
                                         B_ROW_MAJOR, "normal", 4, 0.02, TF32),
}


# Smaller cases of the same kernels, sized for profiler captures: operands
# still larger than L2 (129 MB) but a few hundred MB in total.
PROFILE_WORKLOADS = {
    "fp32_4096_row": Workload("fp32_4096_row", 4096, 4096, 4096, B_ROW_MAJOR, "uniform", 3),
    # 19 x 32 tiles of 192 x 128 = 4 whole waves on 152 SMs; A, B, C 184 MiB
    "fp32_3648x4096x4096_row": Workload("fp32_3648x4096x4096_row", 3648, 4096, 4096, B_ROW_MAJOR,
                                        "uniform", 3),
    # 20 x 32 tiles of 192 x 128 = 4 waves + 32 tiles: the last 32 shared out
    # as stream-K ranges, as at 8192^3; A, B, C 190 MiB
    "fp32_3840x4096x4096_row": Workload("fp32_3840x4096x4096_row", 3840, 4096, 4096, B_ROW_MAJOR,
                                        "uniform", 3),
    # the same with B column-major (the corner-turning kernel)
    "fp32_3648x4096x4096_colB": Workload("fp32_3648x4096x4096_colB", 3648, 4096, 4096, B_COL_MAJOR,
                                         "uniform", 3),
    # 19 x 32 tiles of 128 x 128 = 4 whole waves on 152 SMs; A, B, C 140 MiB
    "fp32_2432x4096x4096_row": Workload("fp32_2432x4096x4096_row", 2432, 4096, 4096, B_ROW_MAJOR,
                                        "uniform", 3),
    "ffn_bf16_4096x7168x4096": Workload("ffn_bf16_4096x7168x4096", 4096, 7168, 4096,
                                        B_ROW_MAJOR, "normal", 4, 0.02, BF16),
    "ffn_tf32_4096x7168x4096": Workload("ffn_tf32_4096x7168x4096", 4096, 7168, 4096,
                                        B_ROW_MAJOR, "normal", 4, 0.02, TF32),
}
# The 8192^3 FP32 operands (same draws as fp32_8192_row) in the FP32-accurate
# tensor-core mode: an extra, labelled mode, not one of the specified configs.
EXTRA_WORKLOADS = {
    "fp32x3_8192_row": Workload("fp32x3_8192_row", 8192, 8192, 8192, B_ROW_MAJOR, "uniform", 3,
                                dtype=F32X3),
}

ALL_WORKLOADS = {**WORKLOADS, **PROFILE_WORKLOADS, **EXTRA_WORKLOADS}


def _draw(gen: torch.Generator, shape, dist: str, sigma: float) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * sigma
    raise ValueError(f"unknown distribution {dist!r}")


def store_b(B_logical: torch.Tensor, layout_b: int) -> torch.Tensor:
    """Lay the logical K x N matrix out as the ABI's B array."""
    if layout_b == B_ROW_MAJOR:
        return B_logical.contiguous()
    if layout_b == B_COL_MAJOR:
        return B_logical.t().contiguous()
    raise ValueError(f"unknown layout_b {layout_b}")


def make_operands(M: int, N: int, K: int, *, layout_b: int = B_ROW_MAJOR,
                  dist: str = "uniform", seed: int = 0, sigma: float = 1.0,
                  dtype: str = F32):
    """Return ``(A, B)`` as CPU tensors in the storage the ABI expects.

    A is (M, K) row-major; B is (K, N) for row-major or (N, K) for
    column-major.  Both are float32 (``f32``, ``tf32``, ``f32x3``), or bfloat16
    when ``dtype == "bf16"``.
    """
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    A = _draw(gen, (M, K), dist, sigma)
    B = _draw(gen, (K, N), dist, sigma)
    if dtype == BF16:
        A = A.to(torch.bfloat16)
        B = B.to(torch.bfloat16)
    elif dtype not in (F32, TF32, F32X3):
        raise ValueError(f"unknown dtype {dtype!r}")
    return A.contiguous(), store_b(B, layout_b)


def make_workload(w: Workload):
    """Operands of a named workload (see ``WORKLOADS``)."""
    return make_operands(w.M, w.N, w.K, layout_b=w.layout_b, dist=w.dist,
                         seed=w.seed, sigma=w.sigma, dtype=w.dtype)


def make_integer_operands(M: int, N: int, K: int, *, layout_b: int = B_ROW_MAJOR,
                          lo: int = -8, hi: int = 8, seed: int = 0,
                          dtype: str = F32):
    """Integer-valued operands in [lo, hi], exactly representable in FP32,
    TF32 and BF16, for bit-exact checks."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    A = torch.randint(lo, hi + 1, (M, K), generator=gen).to(torch.float32)
    B = torch.randint(lo, hi + 1, (K, N), generator=gen).to(torch.float32)
    if dtype == BF16:
        A = A.to(torch.bfloat16)
        B = B.to(torch.bfloat16)
    return A.contiguous(), store_b(B, layout_b)


def sample_indices(n: int, count: int, seed: int):
    """Sorted distinct indices in [0, n) that always include the first and
    last index (the ragged tail), for sampled checks of large outputs."""
    count = min(count, n)
    if count >= n:
        return list(range(n))
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    inner = (torch.randperm(n - 2, generator=gen)[:max(count - 2, 0)] + 1).tolist()
    return sorted(set(inner) | {0, n - 1})[:max(count, 1)] if count > 1 else [n - 1]
