"""GB300-native (sm_103a) dense GEMM: C = A . B for TF32 and FP16/BF16 inputs.

The product runs in the hand-written tcgen05/TMA kernels of ``libdgt_gemm.so``
(C interface in ``include/dgt_gemm.h``); this package holds the build step,
the ctypes binding and the seeded synthetic-input generators.
"""

from .gemm import (  # noqa: F401
    GEMM_B_K_MAJOR,
    GEMM_B_ROW_MAJOR,
    GemmError,
    device_status,
    gemm_bf16,
    gemm_f16,
    gemm_tf32,
    launch_count,
    matmul,
    matmul_from_host,
    reset_device_status,
    set_debug,
)
