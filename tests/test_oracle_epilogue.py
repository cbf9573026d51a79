"""Pins for the fused-epilogue oracle (oracle/epilogue.py): a hand-worked
example, normal-table values of GELU, identities the activations must obey,
closed forms with all-ones operands, and the reduction to the plain product,
so that a wrong sign, a dropped term, a bias broadcast along the wrong axis or
a wrong activation fails one of them."""

import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    sec, key = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] in ("M", "N", "K", "act"):
                sec[parts[0]] = int(parts[1])
            elif parts[0] in ("alpha", "beta"):
                sec[parts[0]] = float(parts[1])
            elif len(parts) == 1 and not parts[0].lstrip("-").replace(".", "").isdigit():
                key = parts[0]
                sec[key] = []
            else:
                sec[key].append([float(v) for v in parts])
    return sec


def test_golden_worked_relu_epilogue():
    g = _read("epilogue_2x2x3_relu_worked.txt")
    A, B = np.array(g["A"]), np.array(g["B"])
    c_in, bias = np.array(g["Cin"]), np.array(g["bias"][0])
    kw = dict(alpha=g["alpha"], beta=g["beta"], c_in=c_in, bias=bias)
    for layout, b_buf, ldb in ((0, B.reshape(-1), 2), (1, B.T.reshape(-1), 3)):
        pre = oracle.gemm_epilogue(2, 2, 3, A.reshape(-1), 3, b_buf, ldb, layout, act=oracle.ACT_NONE, **kw)
        out = oracle.gemm_epilogue(2, 2, 3, A.reshape(-1), 3, b_buf, ldb, layout, act=g["act"], **kw)
        s = oracle.gemm_epilogue_scale(2, 2, 3, A.reshape(-1), 3, b_buf, ldb, layout, act=g["act"], **kw)
        np.testing.assert_array_equal(pre, np.array(g["PRE"]))
        np.testing.assert_array_equal(out, np.array(g["C"]))
        np.testing.assert_array_equal(s, np.array(g["S"]))


def test_gelu_normal_table():
    rows = np.loadtxt(os.path.join(GOLDEN, "gelu_normal_table.txt"))
    np.testing.assert_allclose(oracle.gelu(rows[:, 0]), rows[:, 1], rtol=0, atol=1e-15)


@pytest.mark.parametrize("act", [oracle.gelu, oracle.gelu_tanh])
def test_gelu_forms_odd_part_is_identity(act):
    """x Phi(x) - (-x) Phi(-x) = x, and the tanh form obeys the same identity
    (its tanh term is odd): a sign or factor error in either breaks it."""
    x = np.linspace(-6.0, 6.0, 2401)
    np.testing.assert_allclose(act(x) - act(-x), x, rtol=0, atol=1e-12)
    assert act(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(act(np.array([30.0, -30.0])), [30.0, 0.0], atol=1e-12)


def test_gelu_tanh_approximates_gelu():
    """The tanh form is the published approximation of x Phi(x): within 5e-4
    everywhere (its largest deviation is about 2e-4 near |x| = 2)."""
    x = np.linspace(-8.0, 8.0, 16001)
    d = np.abs(oracle.gelu_tanh(x) - oracle.gelu(x))
    assert d.max() < 5e-4
    assert d.max() > 1e-5  # but they are different functions


def test_gelu_derivative_bound():
    """The Lipschitz constant used in the error scale bounds both forms' slopes."""
    x = np.linspace(-8.0, 8.0, 160001)
    for act in (oracle.gelu, oracle.gelu_tanh):
        slope = np.abs(np.diff(act(x)) / np.diff(x))
        assert slope.max() <= oracle.LIPSCHITZ[oracle.ACT_GELU]
    # the peak of Phi(x) + x phi(x) sits at sqrt(2)
    xs = math.sqrt(2.0)
    peak = 0.5 * (1 + math.erf(xs / math.sqrt(2))) + xs * math.exp(-xs * xs / 2) / math.sqrt(2 * math.pi)
    assert 1.128 < peak < 1.13


def test_relu_values_and_nan():
    out = oracle.relu(np.array([-2.0, -0.0, 0.0, 3.5, np.nan]))
    assert list(out[:4]) == [0.0, 0.0, 0.0, 3.5]
    assert math.isnan(out[4])


@pytest.mark.parametrize("act", [oracle.ACT_NONE, oracle.ACT_RELU, oracle.ACT_GELU, oracle.ACT_GELU_TANH])
def test_all_ones_closed_form(act):
    """A = 1 (M x K), B = 1 (K x N): A.B = K everywhere, so
    out[i][j] = act(alpha K + beta C_in[i][j] + bias[j]), entry by entry."""
    M, N, K = 3, 5, 7
    alpha, beta = -0.25, 1.5
    c_in = np.arange(M * N, dtype=np.float64).reshape(M, N) - 6.0
    bias = np.array([0.5, -1.0, 2.0, -3.0, 0.0])
    out = oracle.gemm_epilogue(M, N, K, np.ones(M * K), K, np.ones(K * N), N, 0, alpha, beta, c_in, bias, act)
    f = {0: lambda v: v, 1: lambda v: max(v, 0.0), 2: lambda v: 0.5 * v * (1 + math.erf(v / math.sqrt(2))),
         3: lambda v: 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))}[act]
    for i in range(M):
        for j in range(N):
            assert out[i, j] == pytest.approx(f(alpha * K + beta * c_in[i, j] + bias[j]), abs=1e-12)


def test_bias_is_per_column_and_beta_zero_ignores_c():
    M, N, K = 2, 3, 1
    a = np.array([1.0, 2.0])          # A: 2 x 1
    b = np.array([1.0, 10.0, 100.0])  # B: 1 x 3
    bias = np.array([0.25, 0.5, 0.75])
    nan_c = np.full((M, N), np.nan)
    out = oracle.gemm_epilogue(M, N, K, a, 1, b, 3, 0, 1.0, 0.0, nan_c, bias, oracle.ACT_NONE)
    np.testing.assert_array_equal(out, [[1.25, 10.5, 100.75], [2.25, 20.5, 200.75]])


def test_identity_epilogue_is_the_plain_product():
    rng = np.random.default_rng(5)
    M, N, K = 4, 6, 9
    a, b = rng.standard_normal(M * K), rng.standard_normal(K * N)
    np.testing.assert_array_equal(oracle.gemm_epilogue(M, N, K, a, K, b, N, 0),
                                  oracle.gemm(M, N, K, a, K, b, N, 0))
    np.testing.assert_array_equal(oracle.gemm_epilogue_scale(M, N, K, a, K, b, N, 0),
                                  oracle.abs_gemm(M, N, K, a, K, b, N, 0))
