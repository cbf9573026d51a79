"""The C interface under concurrent use: several host threads, each with its
own stream, running products at the same time (the library's per-stream
scratch, launch counter and plan state are shared); and products captured
into a CUDA graph and replayed."""

import threading

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
    assert gemm.device_status() == 0


def _check(p, C):
    ref = oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
    s = oracle.abs_gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
    res = oracle.check(C.cpu().double().numpy(), ref, s, p.dtype)
    assert res["ok"], res


# shapes whose plans split tiles (partials in the per-stream scratch): the
# plain CTA pair and the pair on the transposed product
SPLIT_SHAPES = [(768, 1024, 8192), (1024, 1536, 6144)]


def test_split_shapes_still_split():
    for sh in SPLIT_SHAPES:
        assert gemm.plan_query("bf16", *sh)["tail_segs"] > 1, sh


def test_threads_with_their_own_streams():
    # two split plans, one plain, and one whose A rows (odd pitch) are packed
    # into the stream's scratch first
    shapes = [SPLIT_SHAPES[0], (1000, 1500, 700), (300, 520, 200), SPLIT_SHAPES[1]]
    probs = [inputs.make_problem(f"thr{i}", "bf16", *sh, seed_a=10 + i, seed_b=20 + i, dist_a="normal",
                                 lda=sh[2] + 3 if i == 2 else None)
             for i, sh in enumerate(shapes)]
    outs = [None] * len(probs)
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            p = probs[i]
            with torch.cuda.stream(s):
                A, B = p.a.cuda()[:, :p.K], p.b.cuda()
                C = torch.empty((p.M, p.N), dtype=A.dtype, device="cuda")
                for _ in range(20):
                    gemm.matmul(A, B, C, stream=s)
            s.synchronize()
            outs[i] = C
        except Exception as ex:  # noqa: BLE001 - reported below
            errors.append((i, repr(ex)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for p, C in zip(probs, outs):
        _check(p, C)


def test_cuda_graph_capture_and_replay():
    probs = [inputs.make_problem("g0", "bf16", *SPLIT_SHAPES[0], seed_a=31, seed_b=32, dist_a="normal"),
             inputs.make_problem("g1", "tf32", 1000, 900, 700, seed_a=33, seed_b=34),
             inputs.make_problem("g2", "f16", 300, 520, 200, layout=1, seed_a=35, seed_b=36),
             # the pair on the transposed product with a split tail (row-major B)
             inputs.make_problem("g3", "bf16", *SPLIT_SHAPES[1], seed_a=37, seed_b=38, dist_a="normal")]
    s = torch.cuda.Stream()
    dev = [(p.a.cuda(), p.b.cuda(), torch.empty((p.M, p.N), dtype=TORCH[p.dtype], device="cuda")) for p in probs]
    with torch.cuda.stream(s):  # first calls outside capture: the stream's scratch is allocated here
        for p, (A, B, C) in zip(probs, dev):
            gemm.matmul(A, B, C, layout=p.layout, stream=s)
    s.synchronize()
    for _, _, C in dev:
        C.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for p, (A, B, C) in zip(probs, dev):
            gemm.matmul(A, B, C, layout=p.layout, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for p, (_, _, C) in zip(probs, dev):
        _check(p, C)


TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}
