"""CPU oracle for the fused GEMM epilogue.

TEST INFRASTRUCTURE ONLY (see ``oracle/gemm.py``). The CUDA library never
calls it and shares no code with it.

What it computes
----------------
The GEMM pages end at C = A . B; the epilogue is the usual one of BLAS-style
GEMM libraries, which the C interface's ``gemm_*_ex`` calls add, read plainly:

    C_out[i][j] = act(alpha * (A.B)[i][j] + beta * C_in[i][j] + bias[j])

in float64 on the exact values (A.B from ``oracle.gemm``; C_in and bias as
given, i.e. already in the output type), not rounded to any output type.
``beta == 0`` ignores C_in (it may hold NaN); ``bias`` None adds nothing.

Activations (codes of the C interface):

* 0 none: x
* 1 ReLU: max(x, 0), with NaN kept NaN
* 2 GELU: x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2))), Phi the standard
  normal distribution function (Hendrycks and Gimpel's Gaussian error linear
  unit)
* 3 GELU, tanh form: 0.5 * x * (1 + tanh(sqrt(2 / pi) * (x + 0.044715 * x^3))),
  the same paper's approximation

Error scale for the acceptance test: the product's scale S_ij enters as
|alpha| * S_ij, to which |beta * C_in[i][j]| and |bias[j]| add the scale of
the other terms (each is rounded once in fp32 on the GPU); the activation
multiplies errors by at most its Lipschitz constant L (1 for none and ReLU;
GELU's derivative Phi(x) + x phi(x) peaks at x = sqrt(2), about 1.129, and
the tanh form's peak is as close, so L = 1.13 for both):

    S_epi[i][j] = L * (|alpha| * S_ij + |beta| * |C_in[i][j]| + |bias[j]|)
"""

from __future__ import annotations

import math

import numpy as np

from .gemm import abs_gemm, gemm

ACT_NONE, ACT_RELU, ACT_GELU, ACT_GELU_TANH = 0, 1, 2, 3
LIPSCHITZ = {ACT_NONE: 1.0, ACT_RELU: 1.0, ACT_GELU: 1.13, ACT_GELU_TANH: 1.13}

_erf = np.frompyfunc(math.erf, 1, 1)


def relu(x):
    x = np.asarray(x, dtype=np.float64)
    return np.where(x < 0.0, 0.0, x)


def gelu(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)).astype(np.float64))


def gelu_tanh(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


ACTIVATION = {ACT_NONE: lambda x: np.asarray(x, dtype=np.float64), ACT_RELU: relu, ACT_GELU: gelu,
              ACT_GELU_TANH: gelu_tanh}


def _pre(acc, alpha, beta, c_in, bias):
    v = float(alpha) * np.asarray(acc, dtype=np.float64)
    if beta != 0.0:
        v = v + float(beta) * np.asarray(c_in, dtype=np.float64)
    if bias is not None:
        v = v + np.asarray(bias, dtype=np.float64)[None, :]
    return v


def epilogue(acc, alpha=1.0, beta=0.0, c_in=None, bias=None, act=ACT_NONE):
    """act(alpha * acc + beta * c_in + bias[None, :]) in float64; acc and c_in are M x N."""
    return ACTIVATION[act](_pre(acc, alpha, beta, c_in, bias))


def gemm_epilogue(M, N, K, a, lda, b, ldb, layout=0, alpha=1.0, beta=0.0, c_in=None, bias=None, act=ACT_NONE):
    """The fused product on the buffers of the C interface (see ``oracle.gemm``);
    c_in is the M x N logical C (a 2-D array), bias a length-N vector or None."""
    return epilogue(gemm(M, N, K, a, lda, b, ldb, layout), alpha, beta, c_in, bias, act)


def epilogue_scale(S, alpha=1.0, beta=0.0, c_in=None, bias=None, act=ACT_NONE):
    """S_epi = L * (|alpha| S + |beta| |c_in| + |bias|) (see the module text)."""
    s = abs(float(alpha)) * np.asarray(S, dtype=np.float64)
    if beta != 0.0:
        s = s + abs(float(beta)) * np.abs(np.asarray(c_in, dtype=np.float64))
    if bias is not None:
        s = s + np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    return LIPSCHITZ[act] * s


def gemm_epilogue_scale(M, N, K, a, lda, b, ldb, layout=0, alpha=1.0, beta=0.0, c_in=None, bias=None,
                        act=ACT_NONE):
    return epilogue_scale(abs_gemm(M, N, K, a, lda, b, ldb, layout), alpha, beta, c_in, bias, act)
