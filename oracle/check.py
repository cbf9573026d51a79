"""Acceptance test for a GEMM result against the oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/gemm.py``).

The normalised error of one output is

    e_ij = |C_gpu[i][j] - C_ref[i][j]| / S_ij,    S_ij = sum_k |A[i][k]| |B[k][j]|

and a result is accepted when, for every checked entry,

* FP16 / BF16 inputs (output in the input type):
  |C_gpu - C_ref| <= 1e-3 * S_ij + ulp_T(C_ref)  -- "including one output ulp":
  the output is rounded to a 16-bit type, whose spacing alone can exceed
  1e-3 * S when |C| is close to S (e.g. all-ones inputs);
* TF32 inputs (fp32 output): |C_gpu - C_ref| <= 4e-3 * S_ij.

The TF32 bound covers the tensor core's input rounding: a TF32 operand keeps
10 explicit mantissa bits, so each product is off by at most about 2 * 2^-10
of |a||b| whether the hardware truncates or rounds, plus fp32 accumulation.

``ulp_T(x)`` is the spacing of the output format at |x|: 2^(max(e, emin) - p + 1)
with e = floor(log2 |x|), p the precision (11 fp16, 8 bf16, 24 fp32) and emin
the smallest normal exponent (-14 fp16, -126 bf16/fp32).
"""

from __future__ import annotations

import numpy as np

FORMATS = {
    # name: (precision p incl. the hidden bit, smallest normal exponent)
    "f16": (11, -14),
    "bf16": (8, -126),
    "f32": (24, -126),
}

TOLERANCE = {"f16": 1e-3, "bf16": 1e-3, "tf32": 4e-3}
OUT_FORMAT = {"f16": "f16", "bf16": "bf16", "tf32": "f32"}


def ulp(x: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of format ``fmt`` at |x| (float64 in, float64 out)."""
    p, emin = FORMATS[fmt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e2 = np.frexp(x)               # x = m * 2^e2, 0.5 <= m < 1  ->  floor(log2 x) = e2 - 1
    e = np.where(x > 0, e2 - 1, emin)
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - (p - 1)).astype(np.int64))


def allowed_error(c_ref: np.ndarray, s: np.ndarray, dtype: str) -> np.ndarray:
    """Largest accepted |C_gpu - C_ref| per entry for an input dtype."""
    tol = TOLERANCE[dtype]
    bound = tol * np.asarray(s, dtype=np.float64)
    if dtype in ("f16", "bf16"):
        bound = bound + ulp(c_ref, OUT_FORMAT[dtype])
    return bound


def check(c_gpu, c_ref, s, dtype: str) -> dict:
    """Compare a GPU result with the oracle; returns a summary dict with
    ``ok``, the worst bare e_ij (no ulp allowance), its p99, the number of
    failing entries and the first failing position."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    c_ref = np.asarray(c_ref, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    diff = np.abs(c_gpu - c_ref)
    bad = ~(diff <= allowed_error(c_ref, s, dtype))      # NaN counts as bad
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(s > 0, diff / np.where(s > 0, s, 1.0), np.where(diff > 0, np.inf, 0.0))
    out = {
        "ok": not bool(bad.any()),
        "n": int(diff.size),
        "n_bad": int(bad.sum()),
        "max_e": float(np.nanmax(e)) if e.size else 0.0,
        "p99_e": float(np.nanpercentile(e, 99)) if e.size else 0.0,
    }
    if bad.any():
        pos = np.argwhere(bad)[0]
        out["first_bad"] = tuple(int(v) for v in pos)
        out["first_bad_values"] = (float(c_gpu[tuple(pos)]), float(c_ref[tuple(pos)]),
                                   float(s[tuple(pos)]))
    return out
