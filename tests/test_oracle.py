"""Pins for the CPU oracle: each test fixes the oracle against something other
than itself -- hand-worked examples, exact rational arithmetic, closed forms
and special cases -- so that a dropped term, a wrong sign or index, a
transposed operand or a wrong layout reading fails at least one of them."""

from fractions import Fraction
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    sections, key = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] in ("M", "N", "K"):
                sections[parts[0]] = int(parts[1])
            elif parts[0] in ("A", "B", "C", "S"):
                key = parts[0]
                sections[key] = []
            else:
                sections[key].append([float(v) for v in parts])
    return sections


def _store_b(B, layout, ldb=None, pad=float("nan")):
    """Store a logical K x N matrix B in the buffer a layout flag describes."""
    K, N = B.shape
    if layout == 0:
        ld = N if ldb is None else ldb
        buf = np.full((K, ld), pad)
        buf[:, :N] = B
    else:
        ld = K if ldb is None else ldb
        buf = np.full((N, ld), pad)
        buf[:, :K] = B.T
    return buf.reshape(-1), ld


def _store_a(A, lda=None, pad=float("nan")):
    M, K = A.shape
    ld = K if lda is None else lda
    buf = np.full((M, ld), pad)
    buf[:, :K] = A
    return buf.reshape(-1), ld


def _exact_product(A, B):
    """C and S by exact rational arithmetic (pure Python; tiny shapes only)."""
    M, K = A.shape
    N = B.shape[1]
    Af = [[Fraction(float(A[i, k])) for k in range(K)] for i in range(M)]
    Bf = [[Fraction(float(B[k, j])) for j in range(N)] for k in range(K)]
    C = [[sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    S = [[sum((abs(Af[i][k]) * abs(Bf[k][j]) for k in range(K)), Fraction(0)) for j in range(N)]
         for i in range(M)]
    return C, S


@pytest.mark.parametrize("name", ["gemm_2x2x3_worked.txt", "gemm_3x4x2_signed.txt"])
@pytest.mark.parametrize("layout", [0, 1])
def test_golden_worked_examples(name, layout):
    g = _read_golden(name)
    M, N, K = g["M"], g["N"], g["K"]
    A, B = np.array(g["A"]), np.array(g["B"])
    a, lda = _store_a(A, lda=K + 3)
    b, ldb = _store_b(B, layout, ldb=(N if layout == 0 else K) + 2)
    C = oracle.gemm(M, N, K, a, lda, b, ldb, layout)
    S = oracle.abs_gemm(M, N, K, a, lda, b, ldb, layout)
    assert np.array_equal(C, np.array(g["C"]))
    assert np.array_equal(S, np.array(g["S"]))
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ce, se = oracle.gemm_entries(M, N, K, a, lda, b, ldb, layout, rows.ravel(), cols.ravel())
    assert np.array_equal(ce, np.array(g["C"]).ravel())
    assert np.array_equal(se, np.array(g["S"]).ravel())


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (5, 2, 3), (3, 8, 17), (17, 5, 8), (8, 17, 2)])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
def test_bruteforce_exact_rational(M, N, K, dtype):
    """Tiny shapes against exact rational sums: the float64 result must lie
    within the float64 summation bound K * 2^-52 * S of the exact value."""
    layout = (M + N + K) % 2
    A = inputs.to_dtype(inputs.draw(M, K, "uniform", 11 + M), dtype).to(torch.float64).numpy()
    B = inputs.to_dtype(inputs.draw(K, N, "normal", 12 + N), dtype).to(torch.float64).numpy()
    a, lda = _store_a(A, lda=K + 1)
    b, ldb = _store_b(B, layout)
    C = oracle.gemm(M, N, K, a, lda, b, ldb, layout)
    S = oracle.abs_gemm(M, N, K, a, lda, b, ldb, layout)
    Cx, Sx = _exact_product(A, B)
    for i in range(M):
        for j in range(N):
            bound = Fraction(K) * Fraction(2) ** -52 * Sx[i][j]
            assert abs(Fraction(float(C[i, j])) - Cx[i][j]) <= bound
            assert abs(Fraction(float(S[i, j])) - Sx[i][j]) <= bound


def test_small_integers_exact():
    """Integers in [-8, 8]: every product and partial sum is exact in float64,
    so the oracle must equal a pure-Python integer triple loop exactly."""
    rng = np.random.default_rng(5)
    M, N, K = 19, 23, 41
    A = rng.integers(-8, 9, size=(M, K))
    B = rng.integers(-8, 9, size=(K, N))
    for layout in (0, 1):
        a, lda = _store_a(A.astype(np.float64), lda=K + 7)
        b, ldb = _store_b(B.astype(np.float64), layout, ldb=(N if layout == 0 else K) + 5)
        C = oracle.gemm(M, N, K, a, lda, b, ldb, layout)
        for i in range(M):
            for j in range(N):
                want = 0
                for k in range(K):
                    want += int(A[i, k]) * int(B[k, j])
                assert C[i, j] == want


@pytest.mark.parametrize("layout", [0, 1])
def test_identity_left_and_right(layout):
    """A = I gives C = B and B = I gives C = A, exactly, for a non-square B."""
    K, N = 37, 29
    B = inputs.to_dtype(inputs.draw(K, N, "normal", 3), "bf16").to(torch.float64).numpy()
    a, lda = _store_a(np.eye(K), lda=K + 4)
    b, ldb = _store_b(B, layout, ldb=(N if layout == 0 else K) + 3)
    assert np.array_equal(oracle.gemm(K, N, K, a, lda, b, ldb, layout), B)
    M = 13
    A = inputs.to_dtype(inputs.draw(M, K, "uniform", 4), "f16").to(torch.float64).numpy()
    a, lda = _store_a(A)
    b, ldb = _store_b(np.eye(K), layout)
    assert np.array_equal(oracle.gemm(M, K, K, a, lda, b, ldb, layout), A)


@pytest.mark.parametrize("layout", [0, 1])
def test_permutations(layout):
    """A = P (a permutation) gives the rows of B permuted; B = Q permutes the
    columns of A. Distinct permutations on each side catch swapped indices."""
    rng = np.random.default_rng(9)
    K, N, M = 31, 20, 31
    perm = rng.permutation(K)
    P = np.eye(K)[perm]                   # row i of P is e_{perm[i]}
    B = rng.standard_normal((K, N))
    a, lda = _store_a(P)
    b, ldb = _store_b(B, layout)
    assert np.array_equal(oracle.gemm(M, N, K, a, lda, b, ldb, layout), B[perm])
    A = rng.standard_normal((7, K))
    qperm = rng.permutation(K)
    Q = np.eye(K)[:, qperm]               # column j of Q is e_{qperm[j]}
    a, lda = _store_a(A)
    b, ldb = _store_b(Q, layout)
    assert np.array_equal(oracle.gemm(7, K, K, a, lda, b, ldb, layout), A[:, qperm])


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 300), (64, 33, 4104)])
def test_all_ones_closed_form(M, N, K):
    """All-ones operands: every C entry and every S entry equals K."""
    for layout in (0, 1):
        a, lda = _store_a(np.ones((M, K)))
        b, ldb = _store_b(np.ones((K, N)), layout)
        assert np.array_equal(oracle.gemm(M, N, K, a, lda, b, ldb, layout), np.full((M, N), K))
        assert np.array_equal(oracle.abs_gemm(M, N, K, a, lda, b, ldb, layout), np.full((M, N), K))


def test_row_and_column_sums():
    """A column of B that is all ones yields the row sums of A, and a row of A
    that is all ones yields the column sums of B (math.fsum: correctly rounded)."""
    rng = np.random.default_rng(21)
    M, N, K = 9, 6, 257
    A = rng.uniform(-1, 1, (M, K))
    B = rng.uniform(-1, 1, (K, N))
    B[:, 4] = 1.0
    A[2, :] = 1.0
    for layout in (0, 1):
        a, lda = _store_a(A)
        b, ldb = _store_b(B, layout)
        C = oracle.gemm(M, N, K, a, lda, b, ldb, layout)
        for i in range(M):
            assert C[i, 4] == pytest.approx(math.fsum(A[i]), rel=0, abs=K * 2**-52 * np.abs(A[i]).sum())
        for j in range(N):
            assert C[2, j] == pytest.approx(math.fsum(B[:, j]), rel=0, abs=K * 2**-52 * np.abs(B[:, j]).sum())


def test_one_hot_rows_copy_b_rows():
    """Row i of A = e_{k_i}: row i of C is row k_i of B, exactly."""
    K, N = 50, 40
    rng = np.random.default_rng(1)
    ks = rng.integers(0, K, size=12)
    A = np.zeros((12, K))
    A[np.arange(12), ks] = 1.0
    B = rng.standard_normal((K, N))
    for layout in (0, 1):
        a, lda = _store_a(A, lda=K + 1)
        b, ldb = _store_b(B, layout)
        assert np.array_equal(oracle.gemm(12, N, K, a, lda, b, ldb, layout), B[ks])


def test_layouts_agree_and_padding_ignored():
    """One logical B stored both ways gives the same C; NaN padding beyond
    each row (ld > row length) never reaches the result."""
    p = inputs.make_problem("t", "bf16", 45, 70, 90, lda=96, ldb=80)
    q = inputs.make_problem("t", "bf16", 45, 70, 90, lda=96, ldb=100, layout=1)
    # same seeds draw the same K x N values; q holds them transposed
    Bq = inputs.pad_ld(inputs.to_dtype(inputs.draw(90, 70, "uniform", 2000), "bf16").T.contiguous(), 100)
    c1 = oracle.gemm(45, 70, 90, p.a, p.lda, p.b, p.ldb, 0)
    c2 = oracle.gemm(45, 70, 90, q.a, q.lda, Bq, 100, 1)
    assert np.isfinite(c1).all()
    assert np.array_equal(c1, c2)


def test_zero_sizes():
    a = np.ones(12)
    b = np.ones(12)
    assert oracle.gemm(3, 4, 0, a, 1, b, 4, 0).shape == (3, 4)
    assert not oracle.gemm(3, 4, 0, a, 1, b, 4, 0).any()
    assert oracle.gemm(0, 4, 3, a, 3, b, 4, 0).shape == (0, 4)
    assert oracle.gemm(3, 0, 3, a, 3, b, 1, 1).shape == (3, 0)


def test_sampled_entries_match_full():
    """The per-entry path (row . column dot products) agrees with the full
    product at sampled positions, for both layouts and padded buffers."""
    for layout in (0, 1):
        p = inputs.make_problem("t", "f16", 130, 75, 300, lda=304, layout=layout,
                                ldb=(80 if layout == 0 else 310))
        C = oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, layout)
        S = oracle.abs_gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, layout)
        r, c = inputs.sample_entries(p.M, p.N, 500, 7)
        ce, se = oracle.gemm_entries(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, layout, r, c)
        np.testing.assert_allclose(ce, C[r, c], rtol=0, atol=1e-12)
        np.testing.assert_allclose(se, S[r, c], rtol=0, atol=1e-12)


def test_ulp_against_numpy_spacing():
    """ulp() agrees with numpy's own spacing for IEEE half and single."""
    x = np.concatenate([np.geomspace(1e-7, 6e4, 997), -np.geomspace(1e-3, 1e4, 101), [0.0, 1.0, 2.0]])
    np.testing.assert_array_equal(oracle.ulp(x.astype(np.float16).astype(np.float64), "f16"),
                                  np.abs(np.spacing(x.astype(np.float16))).astype(np.float64))
    y = np.geomspace(1e-30, 1e30, 1001)
    np.testing.assert_array_equal(oracle.ulp(y.astype(np.float32).astype(np.float64), "f32"),
                                  np.abs(np.spacing(y.astype(np.float32))).astype(np.float64))


def test_ulp_bfloat16_known_values():
    """bf16 keeps 8 significant bits: spacing 2^-7 at 1, 32 at 4104, and the
    RNE neighbours of 4104 are 4096 and 4128 (4104 rounds to 4096)."""
    assert oracle.ulp(np.array([1.0]), "bf16")[0] == 2.0**-7
    assert oracle.ulp(np.array([4104.0]), "bf16")[0] == 32.0
    assert oracle.ulp(np.array([0.0]), "bf16")[0] == 2.0**-133
    v = torch.tensor([4104.0]).to(torch.bfloat16).double().item()
    assert v == 4096.0
    # every bf16 value's spacing is the gap to the next bf16 value
    xs = torch.tensor([0.3, 1.0, 7.5, 1000.0, 4104.0, 1e20], dtype=torch.bfloat16)
    bits = xs.view(torch.int16) + 1          # the next bf16 value up (all xs > 0)
    gap = (bits.view(torch.bfloat16).double() - xs.double()).numpy()
    np.testing.assert_array_equal(oracle.ulp(xs.double().numpy(), "bf16"), gap)


def test_tolerance_machinery():
    """One output ulp of error passes for 16-bit outputs; an error of 2e-3 * S
    fails; for TF32, 3e-3 * S passes and 5e-3 * S fails."""
    rng = np.random.default_rng(3)
    c_ref = rng.standard_normal(4000) * 30
    s = np.abs(c_ref) * 3 + 1
    for dt, fmt in (("bf16", "bf16"), ("f16", "f16")):
        one_ulp = oracle.ulp(c_ref, fmt)
        assert oracle.check(c_ref + one_ulp, c_ref, s, dt)["ok"]
        assert not oracle.check(c_ref + 2e-3 * s + one_ulp, c_ref, s, dt)["ok"]
        # a single bad entry is enough to fail
        c = c_ref.copy()
        c[1234] += 2e-3 * s[1234] + one_ulp[1234]
        res = oracle.check(c, c_ref, s, dt)
        assert not res["ok"] and res["n_bad"] == 1 and res["first_bad"] == (1234,)
    assert oracle.check(c_ref + 3e-3 * s, c_ref, s, "tf32")["ok"]
    assert not oracle.check(c_ref + 5e-3 * s, c_ref, s, "tf32")["ok"]
    nan = c_ref.copy()
    nan[7] = np.nan
    assert not oracle.check(nan, c_ref, s, "bf16")["ok"]


def test_all_ones_k4104_needs_the_ulp_term():
    """With all-ones inputs and K = 4104, bf16(4104) = 4096: the bare error
    8/4104 exceeds 1e-3 but one output ulp (32) covers it."""
    c_ref = np.full(4, 4104.0)
    s = np.full(4, 4104.0)
    c = torch.tensor(c_ref).to(torch.bfloat16).double().numpy()
    res = oracle.check(c, c_ref, s, "bf16")
    assert res["ok"] and res["max_e"] > 1e-3
