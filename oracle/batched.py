"""CPU oracle for strided batches of products.

TEST INFRASTRUCTURE ONLY (see ``oracle/gemm.py``).

The GEMM pages compute one product; a strided batch (the ``*_strided_batched``
calls of the C interface) is that product repeated, read plainly:

    C_z = A_z . B_z,  z = 0 .. batch-1,

where matrix z of an operand starts ``stride`` elements after matrix z-1 in
its buffer (stride 0: every z reads the same matrix) and each matrix has the
single product's layout and leading dimension. Each C_z is ``oracle.gemm``
on the buffer from that offset on.
"""

from __future__ import annotations

import numpy as np

from .gemm import _f64, abs_gemm, gemm


def _each(fn, batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, layout):
    flat_a, flat_b = _f64(a), _f64(b)
    out = np.empty((batch, M, N))
    for z in range(batch):
        out[z] = fn(M, N, K, flat_a[z * stride_a:], lda, flat_b[z * stride_b:], ldb, layout)
    return out


def gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, layout=0) -> np.ndarray:
    """batch x M x N float64 array of the products C_z = A_z . B_z."""
    return _each(gemm, batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, layout)


def abs_gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, layout=0) -> np.ndarray:
    """The error scales S_z = |A_z| . |B_z| of the batch."""
    return _each(abs_gemm, batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, layout)
