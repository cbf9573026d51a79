"""gemm_{tf32,f16,bf16}_host through the C interface: operands and result in
host memory (padded leading dimensions, page-locked or pageable), checked
element by element against the float64 oracle; consecutive calls on one
stream alternating the library's two staging slots; the degenerate and
refused cases."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_tensor_gb300 import build
    build.build()
    gemm.load()
    gemm.set_tuning(0, 0, 0, 0)
    torch.cuda.set_device(0)
    yield
    assert gemm.device_status() == 0


def _check(p, c_host, ldc):
    c = c_host.view(-1)[: (p.M - 1) * ldc + p.N].double().numpy() if p.M else None
    got = np.stack([c[i * ldc: i * ldc + p.N] for i in range(p.M)])
    ref = oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
    s = oracle.abs_gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
    res = oracle.check(got, ref, s, p.dtype)
    assert res["ok"], res


@pytest.mark.parametrize("dtype,layout,pinned", [("bf16", 0, True), ("f16", 1, True), ("tf32", 0, False),
                                                 ("bf16", 1, False)])
def test_padded_host_operands(dtype, layout, pinned):
    """Leading dimensions larger than the rows (NaN padding that must not leak
    into C, padding of C left untouched), 2 row blocks of A."""
    M, N, K = 2100, 333, 517
    ldc = N + 5
    p = inputs.make_problem("hostio", dtype, M, N, K, layout=layout, seed_a=91, seed_b=92, lda=K + 3,
                            ldb=(N + 7) if layout == 0 else (K + 9))
    a, b = (p.a.pin_memory(), p.b.pin_memory()) if pinned else (p.a.clone(), p.b.clone())
    c = torch.full((M, ldc), -3.0, dtype=TORCH[dtype])
    if pinned:
        c = c.pin_memory()
    s = torch.cuda.Stream()
    code = gemm.gemm_host(dtype, M, N, K, a.data_ptr(), p.lda, b.data_ptr(), p.ldb, c.data_ptr(), ldc, layout,
                          s.cuda_stream)
    assert code == gemm.GEMM_OK, gemm.status_string(code)
    s.synchronize()
    _check(p, c, ldc)
    assert torch.all(c[:, N:] == -3.0)


def test_consecutive_calls_alternate_staging():
    """Four calls enqueued back to back on one stream without waiting (two
    shapes and kinds, so the staging slots are reused and regrown); each
    result checked after one synchronisation."""
    s = torch.cuda.Stream()
    probs = [inputs.make_problem("hostio2", dt, M, N, K, seed_a=100 + i, seed_b=200 + i)
             for i, (dt, M, N, K) in enumerate([("bf16", 1500, 400, 600), ("tf32", 2500, 300, 700),
                                                ("bf16", 1500, 400, 600), ("f16", 4100, 260, 300)])]
    outs = []
    for p in probs:
        a, b = p.a.pin_memory(), p.b.pin_memory()
        c = torch.empty((p.M, p.N), dtype=TORCH[p.dtype]).pin_memory()
        outs.append((a, b, c))
        code = gemm.gemm_host(p.dtype, p.M, p.N, p.K, a.data_ptr(), p.lda, b.data_ptr(), p.ldb, c.data_ptr(), p.N,
                              0, s.cuda_stream)
        assert code == gemm.GEMM_OK
    s.synchronize()
    for p, (_, _, c) in zip(probs, outs):
        _check(p, c, p.N)


def test_k_zero_and_empty():
    c = torch.full((3, 4), 5.0, dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream()
    assert gemm.gemm_host("bf16", 3, 4, 0, None, 0, None, 4, c.data_ptr(), 4, 0, s.cuda_stream) == gemm.GEMM_OK
    s.synchronize()
    assert torch.all(c == 0)
    assert gemm.gemm_host("bf16", 0, 4, 8, None, 8, None, 4, None, 4, 0, s.cuda_stream) == gemm.GEMM_OK


def test_refused_arguments():
    a = torch.zeros((8, 8), dtype=torch.bfloat16)
    c = torch.zeros((8, 8), dtype=torch.bfloat16)
    s = torch.cuda.Stream().cuda_stream
    args = (a.data_ptr(), 8, a.data_ptr(), 8, c.data_ptr(), 8)
    assert gemm.gemm_host("bf16", 8, 8, 8, a.data_ptr(), 7, a.data_ptr(), 8, c.data_ptr(), 8, 0, s) == \
        gemm.GEMM_ERR_INVALID_VALUE  # lda < K
    assert gemm.gemm_host("bf16", 8, 8, 8, *args, 2, s) == gemm.GEMM_ERR_INVALID_VALUE  # layout flag
    assert gemm.gemm_host("bf16", 8, 8, 8, a.data_ptr() + 1, 8, a.data_ptr(), 8, c.data_ptr(), 8, 0, s) == \
        gemm.GEMM_ERR_MISALIGNED
    d = torch.zeros((8, 8), dtype=torch.bfloat16, device="cuda")  # device memory where host memory belongs
    assert gemm.gemm_host("bf16", 8, 8, 8, d.data_ptr(), 8, a.data_ptr(), 8, c.data_ptr(), 8, 0, s) == \
        gemm.GEMM_ERR_INVALID_VALUE
    torch.cuda.synchronize()


def test_two_host_threads_on_their_own_streams():
    """Two host threads, each with its own stream (and so its own staging
    slots), enqueue host-memory products at the same time; every result is
    checked."""
    import threading
    probs = [inputs.make_problem("hostio3", dt, M, N, K, seed_a=300 + i, seed_b=400 + i)
             for i, (dt, M, N, K) in enumerate([("bf16", 2048, 320, 520), ("tf32", 1100, 610, 330)])]
    outs = [None, None]
    errors = []

    def work(i):
        try:
            p = probs[i]
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            a, b = p.a.pin_memory(), p.b.pin_memory()
            c = torch.empty((p.M, p.N), dtype=TORCH[p.dtype]).pin_memory()
            for _ in range(3):
                code = gemm.gemm_host(p.dtype, p.M, p.N, p.K, a.data_ptr(), p.lda, b.data_ptr(), p.ldb, c.data_ptr(),
                                      p.N, 0, s.cuda_stream)
                assert code == gemm.GEMM_OK, code
            s.synchronize()
            outs[i] = c
        except Exception as ex:  # noqa: BLE001 - reported below
            errors.append(ex)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for p, c in zip(probs, outs):
        _check(p, c, p.N)
