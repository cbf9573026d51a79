"""CPU oracle for the dense matrix product C = A . B.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. The CUDA library never calls it, and
it shares no code with the CUDA path.

What it computes
----------------
The plain definition of the product both GEMM pages optimise ("sgemm tf32 -
beating cuBLAS", section 0, and "hgemm - beating cuBLAS", section 0: an
M x K by K x N matrix product, M = N = K = 4096 in their runs), which the
"CUDA GEMM in nine levels" page also takes as its correctness baseline
(sections 2.1 and 3.1: one output element is the sum over k of A[i][k]*B[k][j]):

    C_ref[i][j] = sum_{k < K} A[i][k] * B[k][j]

in float64, on the exact operand values the GPU receives (bf16/fp16 values
are exact in float64; for the TF32 GEMM the unrounded fp32 values are used,
so the tensor core's TF32 input rounding falls inside the tolerance). The
result is not rounded to any output type.

Memory layout (the C interface's definition)
--------------------------------------------
* A: row-major, element (i, k) at ``a[i * lda + k]``.
* B, layout 0 (row-major K x N): element (k, j) at ``b[k * ldb + j]``.
* B, layout 1 (K-major, B transposed, N x K): element (k, j) at ``b[j * ldb + k]``.

A library matrix product in float64 serves as the summation step; nothing is
blocked, fused or reordered beyond the definition.
"""

from __future__ import annotations

import numpy as np

B_ROW_MAJOR = 0
B_K_MAJOR = 1


def _f64(x) -> np.ndarray:
    """Flat float64 copy of a buffer (numpy array or CPU torch tensor)."""
    if hasattr(x, "detach"):  # a torch tensor: the exact widening cast
        import torch
        return x.detach().reshape(-1).to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64).reshape(-1)


def view_a(M: int, K: int, a, lda: int) -> np.ndarray:
    """The logical M x K matrix A read out of its row-major buffer."""
    if M == 0 or K == 0:
        return np.zeros((M, K))
    flat = _f64(a)
    rows = np.lib.stride_tricks.as_strided(
        flat, shape=(M, K), strides=(lda * 8, 8), writeable=False)
    if (M - 1) * lda + K > flat.size:
        raise ValueError("A buffer too small for M, K, lda")
    return np.array(rows)


def view_b(K: int, N: int, b, ldb: int, layout: int) -> np.ndarray:
    """The logical K x N matrix B read out of its buffer for either layout."""
    if K == 0 or N == 0:
        return np.zeros((K, N))
    flat = _f64(b)
    if layout == B_ROW_MAJOR:
        if (K - 1) * ldb + N > flat.size:
            raise ValueError("B buffer too small for K, N, ldb")
        return np.array(np.lib.stride_tricks.as_strided(
            flat, shape=(K, N), strides=(ldb * 8, 8), writeable=False))
    if layout == B_K_MAJOR:
        if (N - 1) * ldb + K > flat.size:
            raise ValueError("B buffer too small for N, K, ldb")
        # element (k, j) sits at b[j * ldb + k]
        return np.array(np.lib.stride_tricks.as_strided(
            flat, shape=(K, N), strides=(8, ldb * 8), writeable=False))
    raise ValueError(f"unknown B layout {layout}")


def gemm(M: int, N: int, K: int, a, lda: int, b, ldb: int, layout: int) -> np.ndarray:
    """C_ref (M x N, float64) = A . B summed in float64; K = 0 gives zeros."""
    A = view_a(M, K, a, lda)
    B = view_b(K, N, b, ldb, layout)
    if K == 0:
        return np.zeros((M, N))
    return A @ B


def abs_gemm(M: int, N: int, K: int, a, lda: int, b, ldb: int, layout: int) -> np.ndarray:
    """S (M x N, float64) = |A| . |B|: the scale of each output's rounding error."""
    A = np.abs(view_a(M, K, a, lda))
    B = np.abs(view_b(K, N, b, ldb, layout))
    if K == 0:
        return np.zeros((M, N))
    return A @ B


def gemm_entries(M: int, N: int, K: int, a, lda: int, b, ldb: int, layout: int,
                 rows: np.ndarray, cols: np.ndarray, chunk: int = 512):
    """C_ref and S at the listed output positions only (for shapes whose full
    product is too large): each entry is the float64 dot product of row i of A
    with column j of B. Returns (c_ref, s), both float64 vectors."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    flat_a = _f64(a) if not hasattr(a, "detach") else None
    c_out = np.empty(rows.size)
    s_out = np.empty(rows.size)
    for lo in range(0, rows.size, chunk):
        r = rows[lo:lo + chunk]
        c = cols[lo:lo + chunk]
        ar = _rows_a(a, flat_a, r, K, lda)          # (n, K)
        bc = _cols_b(b, c, K, ldb, layout)          # (n, K)
        c_out[lo:lo + chunk] = np.einsum("nk,nk->n", ar, bc)
        s_out[lo:lo + chunk] = np.einsum("nk,nk->n", np.abs(ar), np.abs(bc))
    return c_out, s_out


def _rows_a(a, flat_a, r, K, lda):
    if flat_a is not None:
        idx = r[:, None] * lda + np.arange(K)[None, :]
        return flat_a[idx]
    import torch
    t = a.reshape(-1)
    idx = torch.from_numpy(r[:, None] * lda + np.arange(K)[None, :])
    return t[idx].to(torch.float64).numpy()


def _cols_b(b, c, K, ldb, layout):
    if layout == B_ROW_MAJOR:
        idx = np.arange(K)[None, :] * ldb + c[:, None]
    elif layout == B_K_MAJOR:
        idx = c[:, None] * ldb + np.arange(K)[None, :]
    else:
        raise ValueError(f"unknown B layout {layout}")
    if hasattr(b, "detach"):
        import torch
        return b.reshape(-1)[torch.from_numpy(idx)].to(torch.float64).numpy()
    return np.asarray(b, dtype=np.float64).reshape(-1)[idx]
