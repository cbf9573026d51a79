"""CPU oracle for dense C = A . B (float64), strided batches of it, its fused epilogue, FP8 decoding and the
acceptance check.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA library or its binding.
"""

from .gemm import B_K_MAJOR, B_ROW_MAJOR, abs_gemm, gemm, gemm_entries, view_a, view_b  # noqa: F401
from .check import TOLERANCE, allowed_error, check, ulp  # noqa: F401
from .epilogue import (ACT_GELU, ACT_GELU_TANH, ACT_NONE, ACT_RELU, LIPSCHITZ, epilogue, epilogue_scale,  # noqa: F401
                       gelu, gelu_tanh, gemm_epilogue, gemm_epilogue_scale, relu)
from .fp8 import decode_e4m3, decode_e5m2, decode_fp8  # noqa: F401
from .batched import abs_gemm_strided_batched, gemm_strided_batched  # noqa: F401
