"""Decoding of FP8 operand bytes for the oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/gemm.py``).

The two 8-bit formats of the OCP "8-bit Floating Point Specification (OFP8)",
written out from their definitions (sign s, exponent field e, mantissa field m):

* E4M3: 1 + 4 + 3 bits, exponent bias 7. e = 0: (-1)^s * (m / 8) * 2^-6
  (subnormal); otherwise (-1)^s * (1 + m / 8) * 2^(e - 7), except that
  e = 15 with m = 7 is NaN. No infinities; the largest finite value is
  1.75 * 2^8 = 448.
* E5M2: 1 + 5 + 2 bits, exponent bias 15, IEEE 754 conventions. e = 0:
  (-1)^s * (m / 4) * 2^-14; e = 31: infinity (m = 0) or NaN; otherwise
  (-1)^s * (1 + m / 4) * 2^(e - 15). The largest finite value is
  1.75 * 2^15 = 57344.

Every FP8 value is exact in float64, so the product's oracle (``oracle.gemm``)
takes the decoded values as they are.
"""

from __future__ import annotations

import numpy as np


def _bytes(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor of an 8-bit type: its raw bytes
        import torch
        return x.detach().contiguous().view(torch.uint8).numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def decode_e4m3(codes) -> np.ndarray:
    b = _bytes(codes)
    s = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    v = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    v = s * v
    return np.where((e == 15) & ((b & 0x7) == 7), np.nan, v)


def decode_e5m2(codes) -> np.ndarray:
    b = _bytes(codes)
    s = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    m = (b & 0x3).astype(np.float64)
    v = np.where(e == 0, (m / 4.0) * 2.0 ** -14, (1.0 + m / 4.0) * np.exp2(e.astype(np.float64) - 15.0))
    v = np.where(e == 31, np.where((b & 0x3) == 0, np.inf, np.nan), v)
    return s * v


def decode_fp8(codes, fmt: str) -> np.ndarray:
    """float64 values of FP8 bytes; fmt 'e4m3' or 'e5m2'; keeps the input's shape."""
    return {"e4m3": decode_e4m3, "e5m2": decode_e5m2}[fmt](codes)
