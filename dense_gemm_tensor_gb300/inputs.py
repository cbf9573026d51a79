"""Seeded synthetic operands for dense GEMM workloads.

This module only draws random numbers and lays them out in memory. It does
no part of the matrix product, so both the CUDA path and the CPU oracle may
take their inputs from here.

Recipe (one host generator, never used by the GPU path or the oracle):

* ``numpy.random.default_rng(seed)`` (PCG64);
* ``uniform``: ``2 * rng.random(dtype=float32) - 1``, i.e. U[-1, 1);
* ``normal``:  ``rng.standard_normal(dtype=float32) * sigma``;
* values are drawn in fp32 and then rounded to the operand dtype with
  PyTorch's round-to-nearest-even cast (bf16/fp16); fp32 (TF32 GEMM) keeps
  the fp32 draw unrounded;
* a matrix with leading dimension ``ld`` larger than its row length gets its
  padding filled with NaN, so any read of the padding shows up in C.

Seeds follow the workload number: A = 1000 + n, B = 2000 + n, sampled output
entries = 3000 + n.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

DTYPES = {
    "bf16": torch.bfloat16,
    "f16": torch.float16,
    "tf32": torch.float32,
    "e4m3": torch.float8_e4m3fn,  # OCP FP8 bytes; the FP8 products write a bfloat16 C
    "e5m2": torch.float8_e5m2,
}


def draw(rows: int, cols: int, dist: str, seed: int, sigma: float = 1.0) -> np.ndarray:
    """fp32 matrix of shape (rows, cols) drawn from ``dist`` with ``seed``."""
    rng = np.random.default_rng(seed)
    if dist == "uniform":
        x = rng.random((rows, cols), dtype=np.float32)
        x *= np.float32(2.0)
        x -= np.float32(1.0)
    elif dist == "normal":
        x = rng.standard_normal((rows, cols), dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x


def to_dtype(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Round an fp32 array to the operand dtype (RNE); fp32 stays as is."""
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(DTYPES[dtype])


def pad_ld(t: torch.Tensor, ld: int) -> torch.Tensor:
    """Return a (rows, ld) buffer holding ``t`` in its first columns and NaN after."""
    rows, cols = t.shape
    if ld == cols:
        return t.contiguous()
    if ld < cols:
        raise ValueError("ld smaller than the row length")
    buf = torch.full((rows, ld), float("nan"), dtype=t.dtype)
    buf[:, :cols] = t
    return buf


@dataclasses.dataclass
class Problem:
    """One GEMM problem: C (M x N) = A (M x K) . B (K x N).

    ``a`` is the row-major A buffer (M rows of ``lda`` elements). ``b`` is the
    B buffer: K rows of ``ldb`` elements when ``layout == 0`` (row-major B), or
    N rows of ``ldb`` elements holding B transposed when ``layout == 1``
    (K-major B). Both are CPU tensors in the operand dtype.
    """

    name: str
    dtype: str
    M: int
    N: int
    K: int
    a: torch.Tensor
    lda: int
    b: torch.Tensor
    ldb: int
    layout: int
    ldc: int

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


def make_problem(name: str, dtype: str, M: int, N: int, K: int, *, dist_a: str = "uniform",
                 dist_b: str = "uniform", sigma_a: float = 1.0, sigma_b: float = 1.0,
                 seed_a: int = 1000, seed_b: int = 2000, layout: int = 0,
                 lda: int | None = None, ldb: int | None = None,
                 ldc: int | None = None) -> Problem:
    """Draw A and B for one problem with the recipe in the module docstring."""
    lda = K if lda is None else lda
    if layout == 0:
        ldb = N if ldb is None else ldb
        b_rows, b_cols = K, N
    else:
        ldb = K if ldb is None else ldb
        b_rows, b_cols = N, K
    ldc = N if ldc is None else ldc
    a = pad_ld(to_dtype(draw(M, K, dist_a, seed_a, sigma_a), dtype), lda)
    b = pad_ld(to_dtype(draw(b_rows, b_cols, dist_b, seed_b, sigma_b), dtype), ldb)
    return Problem(name, dtype, M, N, K, a, lda, b, ldb, layout, ldc)


# The synthetic workloads. Shapes, value distributions and layouts follow the
# benchmark cases of the TF32 and FP16/BF16 GEMM pages (M = N = K = 4096 row-major),
# plus a square sweep, a ragged shape whose B and C rows are 8200 bytes (not a
# multiple of 16), and a transformer projection with a K-major weight.
WORKLOADS = {
    "bf16_512": dict(n=1, dtype="bf16", M=512, N=512, K=512),
    "tf32_4096": dict(n=2, dtype="tf32", M=4096, N=4096, K=4096),
    "f16_4096": dict(n=3, dtype="f16", M=4096, N=4096, K=4096, dist_a="normal", dist_b="normal"),
    "bf16_4096": dict(n=3, dtype="bf16", M=4096, N=4096, K=4096, dist_a="normal", dist_b="normal"),
    "bf16_1024": dict(n=4, dtype="bf16", M=1024, N=1024, K=1024),
    "bf16_2048": dict(n=4, dtype="bf16", M=2048, N=2048, K=2048),
    "bf16_8192": dict(n=4, dtype="bf16", M=8192, N=8192, K=8192),
    "bf16_16384": dict(n=4, dtype="bf16", M=16384, N=16384, K=16384),
    "bf16_ragged": dict(n=4, dtype="bf16", M=4000, N=4100, K=4104),
    "bf16_proj": dict(n=5, dtype="bf16", M=8192, N=28672, K=8192, dist_a="normal",
                      dist_b="normal", sigma_b=0.02, layout=1),
}


def workload(name: str) -> Problem:
    """Build one named workload with its seeds (A = 1000 + n, B = 2000 + n)."""
    spec = dict(WORKLOADS[name])
    n = spec.pop("n")
    return make_problem(name, seed_a=1000 + n, seed_b=2000 + n, **spec)


def sample_entries(M: int, N: int, count: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """``count`` seeded random (i, j) output positions plus the four corners and
    a stride through the last row and the last column (the tails)."""
    rng = np.random.default_rng(seed)
    i = rng.integers(0, M, size=count)
    j = rng.integers(0, N, size=count)
    tail = min(64, max(M, N))
    ti = np.concatenate([[0, 0, M - 1, M - 1], np.full(tail, M - 1),
                         np.linspace(0, M - 1, tail).astype(np.int64)])
    tj = np.concatenate([[0, N - 1, 0, N - 1], np.linspace(0, N - 1, tail).astype(np.int64),
                         np.full(tail, N - 1)])
    return np.concatenate([i, ti]).astype(np.int64), np.concatenate([j, tj]).astype(np.int64)
