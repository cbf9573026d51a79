"""Pins for the FP8 byte decoding of the oracle (oracle/fp8.py): values the OCP
FP8 definition fixes, and every one of the 256 codes of both formats against
PyTorch's own float8 types (a library conversion, independent of the oracle)."""

import math

import numpy as np
import pytest
import torch

import oracle


def test_e4m3_defining_values():
    v = oracle.decode_e4m3([0x00, 0x80, 0x01, 0x07, 0x08, 0x38, 0xB8, 0x3C, 0x7E, 0xFE, 0x7F, 0xFF])
    assert list(v[:10]) == [0.0, -0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, -1.0, 1.5, 448.0, -448.0]
    assert math.copysign(1.0, v[1]) == -1.0
    assert math.isnan(v[10]) and math.isnan(v[11])


def test_e5m2_defining_values():
    v = oracle.decode_e5m2([0x00, 0x01, 0x03, 0x04, 0x3C, 0x3E, 0x7B, 0xFB, 0x7C, 0xFC, 0x7D, 0x7F])
    assert list(v[:10]) == [0.0, 2.0 ** -16, 3 * 2.0 ** -16, 2.0 ** -14, 1.0, 1.5, 57344.0, -57344.0,
                            math.inf, -math.inf]
    assert math.isnan(v[10]) and math.isnan(v[11])


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_all_codes_match_torch(fmt, tdt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ours = oracle.decode_fp8(codes.numpy(), fmt)
    lib = codes.view(tdt).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_decoding_is_monotone_over_positive_codes(fmt):
    """Codes 0x00 .. largest finite are increasing values (a swapped field breaks this)."""
    last = 0x7E if fmt == "e4m3" else 0x7B
    v = oracle.decode_fp8(np.arange(0, last + 1), fmt)
    assert np.all(np.diff(v) > 0)
    np.testing.assert_array_equal(oracle.decode_fp8(np.arange(0x80, 0x80 + last + 1), fmt), -v)


def test_fp8_product_from_decoded_values():
    """A product of FP8 operands is the plain product of their decoded values:
    1.5 * 2 + (-0.5) * 448 = -221 for two short rows (exact)."""
    a = np.array([0x3C, 0xB0], dtype=np.uint8)   # E4M3 1.5, -0.5
    b = np.array([0x40, 0x7E], dtype=np.uint8)   # E4M3 2.0, 448
    av, bv = oracle.decode_e4m3(a), oracle.decode_e4m3(b)
    assert list(av) == [1.5, -0.5] and list(bv) == [2.0, 448.0]
    assert oracle.gemm(1, 1, 2, av, 2, bv, 1, 0)[0, 0] == -221.0
