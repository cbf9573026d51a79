"""The C interface without a GPU: the library builds, loads, exports every
symbol the header declares, and rejects bad arguments before touching a
device."""

import ctypes
import os
import re

import pytest

from dense_gemm_tensor_gb300 import build, gemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dgt_gemm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gemm.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(gemm_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declarations_match_binding():
    assert _declared_functions() == sorted(gemm.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(0, 9):
        s = gemm.status_string(code)
        assert s and s != "unknown status"
    assert gemm.status_string(99) == "unknown status"


def _bf16(M, N, K, A, lda, B, ldb, C, ldc, layout=0):
    return gemm.gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, layout, None)


@pytest.mark.parametrize("args", [
    (-1, 4, 4, 16, 4, 32, 4, 48, 4),          # negative M
    (4, -1, 4, 16, 4, 32, 4, 48, 4),
    (4, 4, -1, 16, 4, 32, 4, 48, 4),
    (4, 4, 4, 16, 3, 32, 4, 48, 4),           # lda < K
    (4, 4, 4, 16, 4, 32, 3, 48, 4),           # ldb < N (row-major B)
    (4, 4, 4, 16, 4, 32, 4, 48, 3),           # ldc < N
    (4, 4, 4, 0, 4, 32, 4, 48, 4),            # NULL A with K > 0
    (4, 4, 4, 16, 4, 0, 4, 48, 4),            # NULL B
    (4, 4, 4, 16, 4, 32, 4, 0, 4),            # NULL C
    (1 << 31, 4, 4, 16, 1 << 31, 32, 4, 48, 4),  # M beyond the limit
])
def test_invalid_arguments(lib, args):
    M, N, K, A, lda, B, ldb, C, ldc = args
    assert _bf16(M, N, K, A or None, lda, B or None, ldb, C or None, ldc) == gemm.GEMM_ERR_INVALID_VALUE


def test_bad_layout_flag(lib):
    assert _bf16(4, 4, 4, 16, 4, 32, 4, 48, 4, layout=2) == gemm.GEMM_ERR_INVALID_VALUE
    # K-major B needs ldb >= K
    assert _bf16(4, 8, 6, 16, 6, 32, 5, 48, 8, layout=1) == gemm.GEMM_ERR_INVALID_VALUE


def test_misaligned_pointers(lib):
    assert _bf16(4, 4, 4, 17, 4, 32, 4, 48, 4) == gemm.GEMM_ERR_MISALIGNED
    assert gemm.gemm_tf32(4, 4, 4, 16, 4, 34, 4, 48, 4, 0, None) == gemm.GEMM_ERR_MISALIGNED


def test_empty_output_is_a_no_op(lib):
    # M = 0 or N = 0: nothing to do, no pointer is read, no device is needed
    assert _bf16(0, 4, 4, None, 4, None, 4, None, 4) == gemm.GEMM_OK
    assert _bf16(4, 0, 4, None, 4, None, 4, None, 0) == gemm.GEMM_OK


def test_no_device_is_reported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _bf16(4, 4, 4, 16, 4, 32, 4, 64, 4) == gemm.GEMM_ERR_UNSUPPORTED_DEVICE
    out = ctypes.c_uint32(7)
    assert lib.gemm_get_device_status(None, ctypes.byref(out)) == gemm.GEMM_ERR_UNSUPPORTED_DEVICE


def test_launch_count_starts_at_zero_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert gemm.launch_count() == 0


def test_tuning_hook_validation(lib):
    assert lib.gemm_set_tuning(0, 100, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_set_tuning(0, 224, -1, 0) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_set_tuning(5, 0, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_set_tuning(4, 96, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_set_tuning(2, 160, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE   # no 160-wide tile
    assert lib.gemm_set_tuning(3, 96, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_set_tuning(2, 64, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE    # 64 and 32: single CTA only
    assert lib.gemm_set_tuning(4, 32, 0, 0) == gemm.GEMM_ERR_INVALID_VALUE
    for v, w in ((0, 0), (1, 256), (1, 224), (1, 192), (1, 128), (1, 64), (1, 32), (0, 64), (2, 256), (2, 224),
                 (2, 192), (2, 128), (0, 224),
                 (3, 256), (3, 224), (3, 192), (3, 128), (3, 0), (4, 0), (4, 224), (4, 128)):
        assert lib.gemm_set_tuning(v, w, 4, 0) == gemm.GEMM_OK
    assert lib.gemm_set_tuning(0, 0, 0, 0) == gemm.GEMM_OK
    assert lib.gemm_set_tuning(0, 0, 0, 3) == gemm.GEMM_ERR_INVALID_VALUE
    assert lib.gemm_set_tuning(2, 256, 0, 1) == gemm.GEMM_OK
    assert lib.gemm_set_tuning(0, 0, 0, 0) == gemm.GEMM_OK
