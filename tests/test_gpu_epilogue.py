"""Parity of the fused epilogue (gemm_*_ex: C = act(alpha * A.B + beta * C +
bias[j])) with the CPU oracle, through the C interface.

Acceptance per entry (oracle/check.py with the epilogue's error scale,
oracle/epilogue.py): |C_gpu - C_ref| <= tol * S_epi + one output ulp for
FP16/BF16, <= tol * S_epi for TF32, S_epi = L (|alpha| S + |beta| |C_in| +
|bias|), tol 1e-3 (FP16/BF16) or 4e-3 (TF32), L = 1 (none, ReLU) or 1.13 (GELU).
"""

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}
ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu": oracle.ACT_GELU, "gelu_tanh": oracle.ACT_GELU_TANH}


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


def _extra(dtype, M, N, seed):
    """C_in (M x N) and bias (N) in the output type, seeded."""
    c_in = inputs.to_dtype(inputs.draw(M, N, "normal", seed, 2.0), dtype)
    bias = inputs.to_dtype(inputs.draw(1, N, "uniform", seed + 1), dtype)[0]
    return c_in, bias


def _run_and_check(p, alpha, beta, use_bias, act, ldc=None, variant=0, tile_n=0, split=0):
    A, B = p.a.cuda(), p.b.cuda()
    a = A[:, :p.K]
    b = B[:, :p.N] if p.layout == 0 else B[:, :p.K]
    c_in, bias = _extra(p.dtype, p.M, p.N, seed=p.M + 7 * p.N + p.K)
    ldc = p.N if ldc is None else ldc
    Cbuf = torch.full((p.M + 2, ldc), 7.0, dtype=TORCH_DT[p.dtype], device="cuda")
    C = Cbuf[:p.M, :p.N]
    C.copy_(c_in.cuda())
    gemm.set_tuning(variant, tile_n, 0, split)
    try:
        gemm.matmul(a, b, C, layout=p.layout, alpha=alpha, beta=beta,
                    bias=bias.cuda() if use_bias else None, activation=None if act == "none" else act)
        torch.cuda.synchronize()
    finally:
        gemm.set_tuning(0, 0, 0, 0)
    kw = dict(alpha=alpha, beta=beta, c_in=c_in.double().numpy(), bias=bias.double().numpy() if use_bias else None,
              act=ACT[act])
    ref = oracle.gemm_epilogue(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout, **kw)
    s = oracle.gemm_epilogue_scale(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout, **kw)
    res = oracle.check(C.cpu().double().numpy(), ref, s, p.dtype)
    assert res["ok"], res
    # rows past M and columns past N are untouched
    assert torch.all(Cbuf[p.M:, :] == 7.0)
    if ldc > p.N:
        assert torch.all(Cbuf[:, p.N:] == 7.0)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("act", ["none", "relu", "gelu", "gelu_tanh"])
@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_fused_epilogue_every_kernel(dtype, act, variant):
    """alpha, beta, bias and each activation on a ragged multi-tile shape, for
    the single-CTA kernel, the CTA pair, the shared-A pair clusters and the
    pair on the transposed product (bias along the accumulator's rows, C read
    and written column by column)."""
    p = inputs.make_problem("epi", dtype, 300, 700, 520, seed_a=11, seed_b=12, dist_a="normal")
    _run_and_check(p, alpha=0.75, beta=-0.5, use_bias=True, act=act, variant=variant)


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
@pytest.mark.parametrize("beta,use_bias", [(0.0, True), (1.0, False), (2.0, True)])
def test_fused_epilogue_terms(dtype, beta, use_bias):
    """Each term alone and together, K-major B, auto plan."""
    p = inputs.make_problem("epi2", dtype, 520, 390, 260, seed_a=21, seed_b=22, layout=1)
    _run_and_check(p, alpha=-1.25, beta=beta, use_bias=use_bias, act="gelu")


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
@pytest.mark.parametrize("variant", [2, 3, 4])
def test_fused_epilogue_split_tail(dtype, variant):
    """Split tiles: the epilogue applies once, to the summed segments."""
    p = inputs.make_problem("epi3", dtype, 768, 2560, 4096, seed_a=31, seed_b=32, dist_a="normal")
    _run_and_check(p, alpha=0.5, beta=1.0, use_bias=True, act="relu", variant=variant, tile_n=256, split=2)
    assert gemm.last_plan()["tail_segs"] > 1


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
def test_fused_epilogue_unaligned_c(dtype):
    """C rows not a 16-byte multiple: C is read and written by the warps'
    coalesced row accesses instead of TMA."""
    p = inputs.make_problem("epi4", dtype, 333, 301, 200, seed_a=41, seed_b=42)
    _run_and_check(p, alpha=1.0, beta=-1.0, use_bias=True, act="gelu_tanh", ldc=303)


def test_identity_epilogue_is_bitwise_the_plain_call():
    p = inputs.make_problem("epi5", "bf16", 1000, 1500, 700, seed_a=51, seed_b=52)
    A, B = p.a.cuda(), p.b.cuda()
    c1 = gemm.matmul(A, B)
    c2 = torch.full_like(c1, float("nan"))
    gemm.matmul(A, B, c2, alpha=1.0, beta=0.0, bias=None, activation="none")
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
def test_k_zero_with_epilogue(dtype):
    """K = 0: A.B = 0, so C = act(beta * C + bias)."""
    M, N = 37, 70
    c_in, bias = _extra(dtype, M, N, seed=61)
    C = c_in.cuda().clone()
    A = torch.empty((M, 0), dtype=TORCH_DT[dtype], device="cuda")
    B = torch.empty((0, N), dtype=TORCH_DT[dtype], device="cuda")
    gemm.matmul(A, B, C, alpha=3.0, beta=-2.0, bias=bias.cuda(), activation="relu")
    torch.cuda.synchronize()
    ref = oracle.epilogue(np.zeros((M, N)), 3.0, -2.0, c_in.double().numpy(), bias.double().numpy(),
                          oracle.ACT_RELU)
    s = oracle.epilogue_scale(np.zeros((M, N)), 3.0, -2.0, c_in.double().numpy(), bias.double().numpy(),
                              oracle.ACT_RELU)
    assert oracle.check(C.cpu().double().numpy(), ref, s, dtype)["ok"]


@pytest.mark.parametrize("act", ["gelu", "gelu_tanh"])
def test_gelu_precision_dense_grid(act):
    """Both GELU forms on 65536 points of [-12, 12] and at large |x| (where they
    saturate), through the K = 0 product with beta = 1 (C = act(C), fp32 C):
    within 2e-6 * |x| of the float64 oracle, far inside the epilogue's
    acceptance bound."""
    M, N = 64, 1024
    x = np.linspace(-12.0, 12.0, M * N).astype(np.float32)
    x[:8] = [-1000.0, -50.0, -1e-20, 0.0, 1e-20, 50.0, 1000.0, -0.0]
    C = torch.from_numpy(x.reshape(M, N).copy()).cuda()
    A = torch.empty((M, 0), dtype=torch.float32, device="cuda")
    B = torch.empty((0, N), dtype=torch.float32, device="cuda")
    gemm.matmul(A, B, C, beta=1.0, activation=act)
    torch.cuda.synchronize()
    xd = x.astype(np.float64)
    ref = oracle.gelu(xd) if act == "gelu" else oracle.gelu_tanh(xd)
    err = np.abs(C.cpu().double().numpy().ravel() - ref)
    assert np.all(err <= 2e-6 * np.abs(xd)), (act, float(np.max(err / np.maximum(np.abs(xd), 1e-30))))


def test_epilogue_argument_errors():
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(65, dtype=torch.bfloat16, device="cuda")
    pa, pc = A.data_ptr(), C.data_ptr()
    bad_act = gemm.Epilogue(1.0, 0.0, None, 9)
    assert gemm.gemm_ex("bf16", 64, 64, 64, pa, 64, pa, 64, pc, 64, 0, bad_act) == gemm.GEMM_ERR_INVALID_VALUE
    misaligned = gemm.Epilogue(1.0, 0.0, bias.data_ptr() + 1, 0)
    assert gemm.gemm_ex("bf16", 64, 64, 64, pa, 64, pa, 64, pc, 64, 0, misaligned) == gemm.GEMM_ERR_MISALIGNED
    overlapping = gemm.Epilogue(1.0, 0.0, pc + 2 * 64, 0)
    assert gemm.gemm_ex("bf16", 64, 64, 64, pa, 64, pa, 64, pc, 64, 0, overlapping) == gemm.GEMM_ERR_INVALID_VALUE
    host_bias = torch.zeros(64, dtype=torch.bfloat16)
    not_dev = gemm.Epilogue(1.0, 0.0, host_bias.data_ptr(), 0)
    assert gemm.gemm_ex("bf16", 64, 64, 64, pa, 64, pa, 64, pc, 64, 0, not_dev) == gemm.GEMM_ERR_NOT_DEVICE_MEMORY
