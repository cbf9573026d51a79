"""CPU oracle for dense C = A . B (float64) and its acceptance check.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA library or its binding.
"""

from .gemm import B_K_MAJOR, B_ROW_MAJOR, abs_gemm, gemm, gemm_entries, view_a, view_b  # noqa: F401
from .check import TOLERANCE, allowed_error, check, ulp  # noqa: F401
