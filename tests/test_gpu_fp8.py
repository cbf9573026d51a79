"""Parity of the FP8 products (gemm_e4m3, gemm_e5m2: OCP FP8 operands, fp32
accumulation, bfloat16 C) with the CPU oracle on the decoded operand values.

Acceptance per entry: |C_gpu - C_ref| <= 1e-3 * S + one bfloat16 ulp of
C_ref (the 16-bit rule of oracle/check.py: FP8 products are exact in fp32,
so the error budget is that of the FP16/BF16 products), with the fused
epilogue's scale where one is applied.
"""

import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_tensor_gb300 import build
    build.build()
    gemm.load()
    gemm.set_debug(0, 0)
    gemm.reset_device_status()
    yield
    gemm.set_tuning(0, 0, 0, 0)
    assert gemm.device_status() == 0


def _decoded(p):
    return oracle.decode_fp8(p.a, p.dtype), oracle.decode_fp8(p.b, p.dtype)


def _run(p, ldc=None, variant=0, tile_n=0, split=0, **epi):
    A, B = p.a.cuda(), p.b.cuda()
    a = A[:, :p.K]
    b = B[:, :p.N] if p.layout == 0 else B[:, :p.K]
    ldc = p.N if ldc is None else ldc
    Cbuf = torch.full((p.M + 1, ldc), 5.0, dtype=torch.bfloat16, device="cuda")
    C = Cbuf[:p.M, :p.N]
    gemm.set_tuning(variant, tile_n, 0, split)
    try:
        gemm.matmul(a, b, C, layout=p.layout, **epi)
        torch.cuda.synchronize()
    finally:
        gemm.set_tuning(0, 0, 0, 0)
    assert torch.all(Cbuf[p.M:, :] == 5.0)
    if ldc > p.N:
        assert torch.all(Cbuf[:, p.N:] == 5.0)
    return C


def _check(p, C, **epi):
    av, bv = _decoded(p)
    if epi:
        bias = epi.get("bias")
        kw = dict(alpha=epi.get("alpha", 1.0), beta=0.0, bias=None if bias is None else bias.double().cpu().numpy(),
                  act={None: 0, "relu": 1, "gelu": 2, "gelu_tanh": 3}[epi.get("activation")])
        ref = oracle.gemm_epilogue(p.M, p.N, p.K, av, p.lda, bv, p.ldb, p.layout, **kw)
        s = oracle.gemm_epilogue_scale(p.M, p.N, p.K, av, p.lda, bv, p.ldb, p.layout, **kw)
    else:
        ref = oracle.gemm(p.M, p.N, p.K, av, p.lda, bv, p.ldb, p.layout)
        s = oracle.abs_gemm(p.M, p.N, p.K, av, p.lda, bv, p.ldb, p.layout)
    res = oracle.check(C.cpu().double().numpy(), ref, s, "bf16")
    assert res["ok"], res


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("variant,tile_n", [(0, 0), (1, 256), (1, 128), (2, 256), (2, 224), (2, 192), (3, 256),
                                            (3, 128)])
def test_fp8_every_kernel(fmt, layout, variant, tile_n):
    """Each kernel family and width on a ragged multi-tile shape with a K
    tail (K = 520 = 4 x 128 + 8); layout 0 goes through the transpose of B."""
    p = inputs.make_problem("f8", fmt, 300, 700, 520, layout=layout, seed_a=71 + layout, seed_b=72,
                            dist_a="normal", dist_b="normal")
    C = _run(p, variant=variant, tile_n=tile_n)
    _check(p, C)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_unaligned_rows_and_c(fmt):
    """Odd leading dimensions (1-byte aligned rows: packed into aligned rows
    first) and an odd C pitch (row-wise stores)."""
    p = inputs.make_problem("f8u", fmt, 257, 389, 333, layout=1, lda=337, ldb=335, seed_a=81, seed_b=82)
    C = _run(p, ldc=391)
    _check(p, C)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_row_major_b_with_unaligned_a(fmt):
    """A with odd rows (packed) and a row-major B (transposed into K-major
    rows) in the same call: the pack and the transpose both write the
    stream's scratch, in separate slots."""
    p = inputs.make_problem("f8r", fmt, 300, 260, 520, layout=0, lda=523, ldb=265, seed_a=85, seed_b=86)
    C = _run(p, ldc=263)
    _check(p, C)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("variant", [2, 3])
def test_fp8_split_tail(fmt, variant):
    p = inputs.make_problem("f8s", fmt, 768, 2560, 4096, layout=1, seed_a=91, seed_b=92, dist_a="normal")
    C = _run(p, variant=variant, tile_n=256, split=2)
    assert gemm.last_plan()["tail_segs"] > 1
    _check(p, C)


def test_fp8_scaled_epilogue():
    """alpha carries per-tensor scales; bias and GELU on top."""
    p = inputs.make_problem("f8e", "e4m3", 520, 390, 1024, layout=1, seed_a=95, seed_b=96, dist_a="normal",
                            dist_b="normal")
    bias = inputs.to_dtype(inputs.draw(1, 390, "uniform", 97), "bf16")[0].cuda()
    epi = dict(alpha=0.03125, bias=bias, activation="gelu")
    C = _run(p, **epi)
    _check(p, C, **epi)


@pytest.mark.parametrize("layout", [0, 1])
def test_fp8_4096_full(layout):
    """M = N = K = 4096 with N(0,1) operands, checked in full."""
    p = inputs.make_problem("f84k", "e4m3", 4096, 4096, 4096, layout=layout, seed_a=98, seed_b=99,
                            dist_a="normal", dist_b="normal")
    C = _run(p)
    _check(p, C)
