"""Pins for the strided-batch oracle (oracle/batched.py): the block-diagonal
identity (a batch of products is the diagonal of one product of block-diagonal
matrices, computed here without any strides), broadcast strides, the K-major
layout, NaN gaps between matrices that must never leak, and batch = 1."""

import numpy as np
import pytest

import oracle


def _block_diag(blocks):
    rows = sum(b.shape[0] for b in blocks)
    cols = sum(b.shape[1] for b in blocks)
    out = np.zeros((rows, cols))
    r = c = 0
    for b in blocks:
        out[r:r + b.shape[0], c:c + b.shape[1]] = b
        r += b.shape[0]
        c += b.shape[1]
    return out


@pytest.mark.parametrize("layout", [0, 1])
def test_block_diagonal_identity(layout):
    rng = np.random.default_rng(3)
    batch, M, N, K = 4, 3, 5, 7
    As = [rng.integers(-3, 4, size=(M, K)).astype(float) for _ in range(batch)]
    Bs = [rng.integers(-3, 4, size=(K, N)).astype(float) for _ in range(batch)]
    lda, gap_a = K + 2, 5
    stride_a = M * lda + gap_a
    a = np.full(batch * stride_a, np.nan)
    for z, A in enumerate(As):
        for i in range(M):
            a[z * stride_a + i * lda: z * stride_a + i * lda + K] = A[i]
    if layout == 0:
        ldb, rows_b, mats = N + 1, K, Bs
    else:
        ldb, rows_b, mats = K + 3, N, [B.T for B in Bs]
    stride_b = rows_b * ldb + 2
    b = np.full(batch * stride_b, np.nan)
    for z, Bm in enumerate(mats):
        for r in range(rows_b):
            b[z * stride_b + r * ldb: z * stride_b + r * ldb + Bm.shape[1]] = Bm[r]
    got = oracle.gemm_strided_batched(batch, M, N, K, a, lda, stride_a, b, ldb, stride_b, layout)
    big = _block_diag(As) @ _block_diag(Bs)  # (batch M) x (batch N), exact for small integers
    for z in range(batch):
        np.testing.assert_array_equal(got[z], big[z * M:(z + 1) * M, z * N:(z + 1) * N])
    assert not np.isnan(got).any()


def test_zero_stride_repeats_a_matrix():
    rng = np.random.default_rng(4)
    batch, M, N, K = 3, 2, 4, 5
    a_one = rng.standard_normal(M * K)             # one A for every z
    b_all = rng.standard_normal(batch * K * N)
    got = oracle.gemm_strided_batched(batch, M, N, K, a_one, K, 0, b_all, N, K * N, 0)
    for z in range(batch):
        np.testing.assert_array_equal(got[z], oracle.gemm(M, N, K, a_one, K, b_all[z * K * N:], N, 0))
    a_all = rng.standard_normal(batch * M * K)
    b_one = rng.standard_normal(K * N)             # one B (a shared weight) for every z
    got = oracle.gemm_strided_batched(batch, M, N, K, a_all, K, M * K, b_one, N, 0, 0)
    for z in range(batch):
        np.testing.assert_array_equal(got[z], oracle.gemm(M, N, K, a_all[z * M * K:], K, b_one, N, 0))


def test_batch_of_one_is_the_product_and_scales_match():
    rng = np.random.default_rng(5)
    M, N, K = 4, 3, 6
    a, b = rng.standard_normal(M * K), rng.standard_normal(K * N)
    np.testing.assert_array_equal(oracle.gemm_strided_batched(1, M, N, K, a, K, 0, b, N, 0, 0)[0],
                                  oracle.gemm(M, N, K, a, K, b, N, 0))
    np.testing.assert_array_equal(oracle.abs_gemm_strided_batched(1, M, N, K, a, K, 0, b, N, 0, 0)[0],
                                  oracle.abs_gemm(M, N, K, a, K, b, N, 0))
