"""Parity of the strided-batch products (gemm_*_strided_batched) with the CPU
oracle (oracle/batched.py): every matrix of the batch in full, with the
single product's acceptance rule (oracle/check.py)."""

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32, "e4m3": torch.float8_e4m3fn,
            "e5m2": torch.float8_e5m2}


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


def _batch(dtype, batch, rows, cols, seed, gap_rows=0, dist="uniform"):
    """batch x rows x cols operand whose matrices sit gap_rows padded rows
    apart (NaN in the gaps); returns (tensor view, flat CPU buffer, ld, stride)."""
    pad = 16 // TORCH_DT[dtype].itemsize  # 16-byte rows
    ld = -(-cols // pad) * pad
    stride = (rows + gap_rows) * ld
    buf = torch.full((batch * stride,), float("nan"), dtype=TORCH_DT[dtype])
    for z in range(batch):
        m = inputs.to_dtype(inputs.draw(rows, cols, dist, seed + z), dtype)
        buf[z * stride:z * stride + rows * ld].view(rows, ld)[:, :cols] = m
    view = buf.as_strided((batch, rows, cols), (stride, ld, 1))
    return view, buf, ld, stride


def _check_batch(dtype, C, batch, M, N, K, a, lda, sa, b, ldb, sb, layout):
    ref = oracle.gemm_strided_batched(batch, M, N, K, a, lda, sa, b, ldb, sb, layout)
    s = oracle.abs_gemm_strided_batched(batch, M, N, K, a, lda, sa, b, ldb, sb, layout)
    got = C.cpu().double().numpy()
    for z in range(batch):
        res = oracle.check(got[z], ref[z], s[z], dtype)
        assert res["ok"], (z, res)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_batched_every_kernel(dtype, layout, variant):
    if variant == 4 and layout == 1:
        pytest.skip("the transposed product is the row-major-B kernel")
    batch, M, N, K = 5, 300, 260, 200
    A, a_buf, lda, sa = _batch(dtype, batch, M, K, 100, gap_rows=3)
    if layout == 0:
        B, b_buf, ldb, sb = _batch(dtype, batch, K, N, 200, gap_rows=1)
    else:
        B, b_buf, ldb, sb = _batch(dtype, batch, N, K, 200, gap_rows=2)
    Cbuf = torch.full((batch, M + 2, N + 8), 9.0, dtype=TORCH_DT[dtype], device="cuda")
    C = Cbuf[:, :M, :N]
    gemm.set_tuning(variant, 0, 0, 0)
    try:
        gemm.bmm(_dev(a_buf, A), _dev(b_buf, B), C, layout=layout)
        torch.cuda.synchronize()
    finally:
        gemm.set_tuning(0, 0, 0, 0)
    assert torch.all(Cbuf[:, M:, :] == 9.0) and torch.all(Cbuf[:, :, N:] == 9.0)
    _check_batch(dtype, C, batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, layout)


def _dev(buf, view):
    """The same strided view over a device copy of the buffer."""
    d = buf.cuda()
    return d.as_strided(view.shape, view.stride())


@pytest.mark.parametrize("shared", ["A", "B"])
def test_batched_shared_operand(shared):
    """A stride of 0 repeats one matrix (a shared weight or a shared input)."""
    dtype, batch, M, N, K = "bf16", 6, 200, 330, 180
    if shared == "B":
        A, a_buf, lda, sa = _batch(dtype, batch, M, K, 300)
        B1, b_buf, ldb, _ = _batch(dtype, 1, K, N, 400)
        sb = 0
        Ad, Bd = _dev(a_buf, A), _dev(b_buf, B1).expand(batch, K, N)
    else:
        A1, a_buf, lda, _ = _batch(dtype, 1, M, K, 300)
        B, b_buf, ldb, sb = _batch(dtype, batch, K, N, 400)
        sa = 0
        Ad, Bd = _dev(a_buf, A1).expand(batch, M, K), _dev(b_buf, B)
    C = gemm.bmm(Ad, Bd)
    torch.cuda.synchronize()
    _check_batch(dtype, C, batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)


def test_batched_many_small_products():
    """64 products of 128 x 128 x 256: a few tiles each, one launch."""
    dtype, batch, M, N, K = "bf16", 64, 128, 128, 256
    A, a_buf, lda, sa = _batch(dtype, batch, M, K, 500)
    B, b_buf, ldb, sb = _batch(dtype, batch, K, N, 600)
    C = gemm.bmm(_dev(a_buf, A), _dev(b_buf, B))
    torch.cuda.synchronize()
    assert gemm.last_plan()["work_items"] >= batch
    _check_batch(dtype, C, batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)


@pytest.mark.parametrize("variant", [2, 3, 4])
def test_batched_split_tail(variant):
    """3 x (768 x 1024 x 4096): 36 pair tiles leave a partial round that is split along K."""
    dtype, batch, M, N, K = "bf16", 3, 768, 1024, 4096
    A, a_buf, lda, sa = _batch(dtype, batch, M, K, 700, dist="normal")
    B, b_buf, ldb, sb = _batch(dtype, batch, K, N, 800)
    gemm.set_tuning(variant, 256, 0, 2)
    try:
        C = gemm.bmm(_dev(a_buf, A), _dev(b_buf, B))
        torch.cuda.synchronize()
        assert gemm.last_plan()["tail_segs"] > 1
    finally:
        gemm.set_tuning(0, 0, 0, 0)
    _check_batch(dtype, C, batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)


def test_batched_with_epilogue():
    dtype, batch, M, N, K = "tf32", 4, 260, 200, 300
    A, a_buf, lda, sa = _batch(dtype, batch, M, K, 900)
    B, b_buf, ldb, sb = _batch(dtype, batch, K, N, 950)
    c_in = torch.stack([inputs.to_dtype(inputs.draw(M, N, "normal", 990 + z), dtype) for z in range(batch)])
    bias = inputs.to_dtype(inputs.draw(1, N, "uniform", 999), dtype)[0]
    C = c_in.cuda().clone()
    gemm.bmm(_dev(a_buf, A), _dev(b_buf, B), C, alpha=0.5, beta=-1.0, bias=bias.cuda(), activation="relu")
    torch.cuda.synchronize()
    got = C.cpu().double().numpy()
    acc = oracle.gemm_strided_batched(batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)
    s = oracle.abs_gemm_strided_batched(batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)
    for z in range(batch):
        kw = dict(alpha=0.5, beta=-1.0, c_in=c_in[z].double().numpy(), bias=bias.double().numpy(),
                  act=oracle.ACT_RELU)
        res = oracle.check(got[z], oracle.epilogue(acc[z], **kw), oracle.epilogue_scale(s[z], **kw), dtype)
        assert res["ok"], (z, res)


def test_batched_argument_errors():
    A = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device="cuda")
    pa, pc = A.data_ptr(), C.data_ptr()
    fn = gemm.load().gemm_bf16_strided_batched
    # C matrices overlapping one another
    assert fn(2, 64, 64, 64, pa, 64, 4096, pa, 64, 4096, pc, 64, 100, 0, None, None) == gemm.GEMM_ERR_INVALID_VALUE
    # a matrix stride off 16-byte boundaries
    assert fn(2, 64, 64, 64, pa, 64, 4100, pa, 64, 4096, pc, 64, 4096, 0, None, None) == gemm.GEMM_ERR_INVALID_VALUE \
        or fn(2, 64, 64, 64, pa, 64, 4100, pa, 64, 4096, pc, 64, 4096, 0, None, None) == gemm.GEMM_ERR_MISALIGNED
    assert fn(2, 63, 64, 64, pa, 64, 4036, pa, 64, 4096, pc, 64, 4096, 0, None, None) == gemm.GEMM_ERR_MISALIGNED
    # negative batch; batch 0 is a no-op
    assert fn(-1, 64, 64, 64, pa, 64, 4096, pa, 64, 4096, pc, 64, 4096, 0, None, None) == gemm.GEMM_ERR_INVALID_VALUE
    assert fn(0, 64, 64, 64, pa, 64, 4096, pa, 64, 4096, pc, 64, 4096, 0, None, None) == gemm.GEMM_OK


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_batched_fp8(fmt):
    """FP8 batches (K-major B, bfloat16 C), with a shared B and with one per matrix."""
    batch, M, N, K = 4, 300, 272, 384
    A, a_buf, lda, sa = _batch(fmt, batch, M, K, 1100, dist="normal")
    B, b_buf, ldb, sb = _batch(fmt, batch, N, K, 1200, dist="normal")
    av, bv = oracle.decode_fp8(a_buf, fmt), oracle.decode_fp8(b_buf, fmt)
    C = gemm.bmm(_dev(a_buf, A), _dev(b_buf, B), layout=1)
    torch.cuda.synchronize()
    _check_batch("bf16", C, batch, M, N, K, av, lda, sa, bv, ldb, sb, 1)
    B1 = _dev(b_buf, B)[:1].expand(batch, N, K)
    C = gemm.bmm(_dev(a_buf, A), B1, layout=1)
    torch.cuda.synchronize()
    _check_batch("bf16", C, batch, M, N, K, av, lda, sa, bv, ldb, 0, 1)
    # a row-major FP8 B is not taken in a batch
    fn = gemm.load().gemm_e4m3_strided_batched
    pa, pc = _dev(a_buf, A).data_ptr(), C.data_ptr()
    assert fn(2, 64, 64, 64, pa, 64, 4096, pa, 64, 4096, pc, 64, 4096, 0, None, None) == gemm.GEMM_ERR_INVALID_VALUE


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
@pytest.mark.parametrize("extra", [1, 2, 4])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_batched_c_stride_granularity(dtype, extra, beta):
    """C matrices whose batch stride is not a 16-byte multiple (extra elements
    after each matrix): C is written by row stores no wider than the stride
    allows, for every matrix of the batch (also when beta * C reads it)."""
    batch, M, N, K = 3, 130, 200, 96
    A, a_buf, lda, sa = _batch(dtype, batch, M, K, 300)
    B, b_buf, ldb, sb = _batch(dtype, batch, K, N, 400)
    ldc = N + 8
    sc = M * ldc + extra
    fill = 0.5
    Cflat = torch.full((batch * sc + 16,), fill, dtype=TORCH_DT[dtype], device="cuda")
    C = Cflat.as_strided((batch, M, N), (sc, ldc, 1))
    gemm.bmm(_dev(a_buf, A), _dev(b_buf, B), C, beta=beta)
    torch.cuda.synchronize()
    ref = oracle.gemm_strided_batched(batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)
    s = oracle.abs_gemm_strided_batched(batch, M, N, K, a_buf, lda, sa, b_buf, ldb, sb, 0)
    got = C.cpu().double().numpy()
    c_in = np.full((M, N), fill)
    for z in range(batch):
        want = oracle.epilogue(ref[z], 1.0, beta, c_in)
        scale = oracle.epilogue_scale(s[z], 1.0, beta, c_in)
        res = oracle.check(got[z], want, scale, dtype)
        assert res["ok"], (z, res)
    # everything outside the C matrices keeps its value
    mask = torch.ones(Cflat.numel(), dtype=torch.bool, device="cuda")
    for z in range(batch):
        for r in range(M):
            mask[z * sc + r * ldc:z * sc + r * ldc + N] = False
    assert torch.all(Cflat[mask] == fill)
