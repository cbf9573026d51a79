"""Parity of the CUDA GEMM with the CPU oracle, through the C interface.

Acceptance per output entry (see oracle/check.py): |C_gpu - C_ref| <=
1e-3 * S + one output ulp for FP16/BF16 inputs and <= 4e-3 * S for TF32,
S = sum_k |A[i][k]| |B[k][j]|. Small shapes and every workload up to 4096 are
checked in full; the larger workloads on >= 4096 seeded sampled entries plus
corners and the last row and column.
"""

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}
# gemm_last_plan's kernel field for each forced tuning variant
PLAN_KERNEL = {1: 1, 2: 2, 3: 4, 4: 3}


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


def _views(p, A, B):
    a = A[:, :p.K]
    b = B[:, :p.N] if p.layout == 0 else B[:, :p.K]
    return a, b


def _run(p, ldc=None, out_rows=None, fill=None):
    """Run the product of problem p on the GPU; returns (C logical view, C buffer)."""
    A = p.a.cuda()
    B = p.b.cuda()
    a, b = _views(p, A, B)
    ldc = p.N if ldc is None else ldc
    rows = p.M if out_rows is None else out_rows
    Cbuf = torch.empty((rows, ldc), dtype=TORCH_DT[p.dtype], device="cuda")
    if fill is not None:
        Cbuf.fill_(fill)
    C = Cbuf[:p.M, :p.N]
    gemm.matmul(a, b, C, layout=p.layout)
    torch.cuda.synchronize()
    return C, Cbuf


def _check_full(p, C):
    c_ref = oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
    s = oracle.abs_gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
    res = oracle.check(C.cpu().double().numpy(), c_ref, s, p.dtype)
    assert res["ok"], res
    return res


def _check_sampled(p, C, seed, count=4096):
    r, c = inputs.sample_entries(p.M, p.N, count, seed)
    got = C[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu().double().numpy()
    c_ref, s = oracle.gemm_entries(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout, r, c)
    res = oracle.check(got, c_ref, s, p.dtype)
    assert res["ok"], res
    return res


SMALL_SHAPES = [(1, 1, 1), (7, 13, 5), (128, 256, 64), (129, 257, 65), (300, 520, 200), (257, 300, 1000),
                (64, 600, 8), (1000, 40, 333)]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_small_shapes_full(dtype, layout, shape):
    M, N, K = shape
    # 8-element-padded pitches keep every operand on the TMA path
    pad = 8 if dtype != "tf32" else 4
    lda = -(-K // pad) * pad
    ldb = -(-(N if layout == 0 else K) // pad) * pad
    p = inputs.make_problem("small", dtype, M, N, K, seed_a=M * 7 + K, seed_b=N * 5 + K, layout=layout,
                            lda=lda, ldb=ldb, dist_a="normal")
    C, _ = _run(p)
    _check_full(p, C)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_small_shapes_transposed_product(dtype, shape):
    """The pair kernel on the transposed product (forced) on the small and
    degenerate shapes: one element, K below one k-slab, C narrower than a
    warp's 32 columns or than one CTA's 128, fewer rows of C than a chunk."""
    M, N, K = shape
    pad = 8 if dtype != "tf32" else 4
    p = inputs.make_problem("smallt", dtype, M, N, K, seed_a=M * 3 + K, seed_b=N * 11 + K,
                            lda=-(-K // pad) * pad, ldb=-(-N // pad) * pad, dist_a="normal")
    gemm.set_tuning(4, 0, 0, 0)
    try:
        C, Cbuf = _run(p, ldc=N + 8, fill=3.0)
        assert gemm.last_plan()["kernel"] == PLAN_KERNEL[4]
    finally:
        gemm.set_tuning(0, 0, 0, 0)
    _check_full(p, C)
    assert torch.all(Cbuf[:, N:] == 3.0)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("tile_n", [256, 224, 192, 128, 64, 32])
def test_every_tile_width_full(dtype, layout, tile_n):
    """Each built tile width, forced, on a ragged multi-tile shape (TMA path)
    and on an odd-pitch shape (copy-warp path)."""
    gemm.set_tuning(1, tile_n, 3, 0)
    try:
        for (M, N, K, lda, ldb) in [(300, 700, 520, 520, None), (260, 450, 300, 301, 451)]:
            if ldb is None:
                ldb = N if layout == 0 else K
            elif layout == 1:
                ldb = K + 1
            p = inputs.make_problem("tw", dtype, M, N, K, lda=lda, ldb=ldb, layout=layout,
                                    seed_a=tile_n + M, seed_b=tile_n + N)
            C, _ = _run(p)
            _check_full(p, C)
    finally:
        gemm.set_tuning(0, 0, 0, 0)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("tile_n", [256, 224, 192, 128])
@pytest.mark.parametrize("variant", [2, 3, 4])
def test_pair_kernel_full(dtype, layout, tile_n, variant):
    """The CTA-pair kernel (256-row tiles over two SMs; variant 3: clusters of
    two pairs that share A and take two adjacent tiles; variant 4, row-major
    B: the transposed product, 256 columns of C by tile_n rows), forced, on
    shapes with a ragged pair-row (M = 129: the second CTA's rows are all past
    M; transposed: N = 300, the second tile's second CTA past N), ragged
    columns, an odd number of tile columns (the second pair's tile lies past
    N) and several waves of tiles."""
    if variant == 4 and layout == 1:
        pytest.skip("the transposed product is the row-major-B kernel")
    gemm.set_tuning(variant, tile_n, 2, 0)
    try:
        for (M, N, K) in [(300, 700, 520), (129, 300, 200), (1000, 1500, 336), (2048, 1024, 64)]:
            ldb = N if layout == 0 else K
            pad = 8 if dtype != "tf32" else 4
            ldb = -(-ldb // pad) * pad
            p = inputs.make_problem("pair", dtype, M, N, K, lda=-(-K // pad) * pad, ldb=ldb, layout=layout,
                                    seed_a=tile_n + M + 1, seed_b=tile_n + N + 2, dist_a="normal")
            C, Cbuf = _run(p, ldc=N + 8, fill=3.0)
            assert gemm.last_plan()["kernel"] == PLAN_KERNEL[variant]
            _check_full(p, C)
            assert torch.all(Cbuf[:, N:] == 3.0)
    finally:
        gemm.set_tuning(0, 0, 0, 0)


@pytest.mark.parametrize("dtype", ["bf16", "tf32"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("shape", [(768, 2560, 4096), (1280, 1024, 4096), (768, 1024, 4096), (4096, 4096, 512),
                                   (768, 2816, 4096)])
@pytest.mark.parametrize("variant", [2, 3, 4])
def test_pair_split_tail(dtype, layout, shape, variant):
    """Tiles of the last partial round split along K (2-4 segments, chosen
    from the co-resident cluster count when each segment keeps >= 16
    k-slabs): full parity, and bitwise-equal results over repeated runs
    whatever segment arrives last."""
    M, N, K = shape
    if variant == 4 and layout == 1:
        pytest.skip("the transposed product is the row-major-B kernel")
    gemm.set_tuning(variant, 256, 0, 2)  # split wherever the geometry allows
    try:
        p = inputs.make_problem("split", dtype, M, N, K, layout=layout, seed_a=M + N, seed_b=K, dist_a="normal")
        C1, _ = _run(p)
        plan = gemm.last_plan()
        assert plan["kernel"] == PLAN_KERNEL[variant]
        pairs = 2 if variant == 3 else 1
        tile_cols = -(-N // 256)
        tiles = -(-M // 256) * -(-tile_cols // pairs)  # work tiles: pairs adjacent 256-wide tiles each
        if K == 4096 and tiles % plan["concurrent_tiles"]:
            assert plan["tail_segs"] > 1, plan
        assert plan["work_items"] == plan["tail_start"] + (tiles - plan["tail_start"]) * plan["tail_segs"]
        _check_full(p, C1)
        for _ in range(2):
            C2, _ = _run(p)
            assert torch.equal(C1, C2)
    finally:
        gemm.set_tuning(0, 0, 0, 0)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "tf32"])
@pytest.mark.parametrize("layout", [0, 1])
def test_small_integers_bit_exact(dtype, layout):
    """Integer operands in [-4, 4]: every product and partial sum is exact in
    fp32, so C must equal the oracle rounded once (RNE) to the output type."""
    M, N, K = 300, 520, 700
    rng = np.random.default_rng(17 + layout)
    Ai = torch.from_numpy(rng.integers(-4, 5, size=(M, K)).astype(np.float32)).to(TORCH_DT[dtype])
    Bi = torch.from_numpy(rng.integers(-4, 5, size=(K, N)).astype(np.float32)).to(TORCH_DT[dtype])
    Bs = Bi if layout == 0 else Bi.T.contiguous()
    p = inputs.Problem("int", dtype, M, N, K, Ai, K, Bs, (N if layout == 0 else K), layout, N)
    C, _ = _run(p)
    c_ref = oracle.gemm(M, N, K, p.a, p.lda, p.b, p.ldb, layout)
    want = torch.from_numpy(c_ref).to(TORCH_DT[dtype])
    assert torch.equal(C.cpu(), want)


@pytest.mark.parametrize("dtype,lda,ldb,ldc", [
    ("bf16", 301, 523, 521),   # odd pitches: 2-byte copy granularity, unaligned C
    ("bf16", 302, 522, 522),   # 4-byte granularity
    ("f16", 204, 524, 526),    # 8-byte granularity for A, 4 for B
    ("tf32", 201, 521, 523),   # 4-byte granularity
    ("tf32", 202, 522, 520),   # 8-byte granularity, aligned C
    ("bf16", 304, 524, 524),   # 8-byte granularity for B and C (8-byte row stores of C)
    ("tf32", 204, 522, 522),   # the same for fp32
])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("pack", [True, False])
def test_unaligned_pitches_full(dtype, lda, ldb, ldc, layout, pack):
    """Row pitches TMA cannot address: packed into aligned scratch first (the
    default), or read in place by the kernel's copy warps (test hook)."""
    M, N, K = 300, 520, 200
    if layout == 1:
        ldb = lda + 3
    p = inputs.make_problem("unal", dtype, M, N, K, lda=lda, ldb=ldb, layout=layout, seed_a=5, seed_b=6)
    gemm.set_debug(0 if pack else 2, 0)
    try:
        C, Cbuf = _run(p, ldc=ldc, fill=7.0)
    finally:
        gemm.set_debug(0, 0)
    _check_full(p, C)
    assert torch.all(Cbuf[:, N:] == 7.0)


def test_output_guard_band_untouched():
    """C inside a larger buffer (ldc > N, extra rows): the padding keeps its sentinel."""
    p = inputs.make_problem("guard", "bf16", 200, 300, 128, seed_a=1, seed_b=2)
    C, Cbuf = _run(p, ldc=320, out_rows=210, fill=-3.0)
    _check_full(p, C)
    assert torch.all(Cbuf[:, 300:] == -3.0)
    assert torch.all(Cbuf[200:, :] == -3.0)


def test_k_zero_writes_zeros_and_empty_is_no_op():
    for dt in ("bf16", "tf32"):
        C = torch.full((33, 70), 5.0, dtype=TORCH_DT[dt], device="cuda")
        A = torch.empty((33, 0), dtype=TORCH_DT[dt], device="cuda")
        B = torch.empty((0, 70), dtype=TORCH_DT[dt], device="cuda")
        gemm.matmul(A, B, C)
        torch.cuda.synchronize()
        assert torch.all(C == 0)
    C = torch.full((0, 5), 5.0, dtype=torch.bfloat16, device="cuda")
    gemm.matmul(torch.empty((0, 8), dtype=torch.bfloat16, device="cuda"),
                torch.empty((8, 5), dtype=torch.bfloat16, device="cuda"), C)


def test_deterministic_bitwise():
    p = inputs.make_problem("det", "bf16", 1000, 1500, 2000, seed_a=3, seed_b=4)
    C1, _ = _run(p)
    C2, _ = _run(p)
    assert torch.equal(C1, C2)


def test_rejects_host_memory_and_overlap():
    A = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    H = torch.ones((64, 64), dtype=torch.bfloat16)
    C = torch.empty((64, 64), dtype=torch.bfloat16, device="cuda")
    code = gemm.gemm_bf16(64, 64, 64, H.data_ptr(), 64, B.data_ptr(), 64, C.data_ptr(), 64, 0, None)
    assert code == gemm.GEMM_ERR_NOT_DEVICE_MEMORY
    code = gemm.gemm_bf16(64, 64, 64, A.data_ptr(), 64, B.data_ptr(), 64, A.data_ptr(), 64, 0, None)
    assert code == gemm.GEMM_ERR_INVALID_VALUE


@pytest.mark.parametrize("variant", [1, 2])
def test_wait_time_limit_reports_and_recovers(variant):
    """A producer that issues nothing leaves the MMA issuer's first wait
    unsatisfied: the kernel gives up after the (short) limit, records a
    timeout, and the next normal launch is correct (single-CTA and pair)."""
    p = inputs.make_problem("to", "bf16", 512, 512, 256, seed_a=8, seed_b=9)
    A, B = p.a.cuda(), p.b.cuda()
    C = torch.empty((512, 512), dtype=torch.bfloat16, device="cuda")
    gemm.reset_device_status()
    gemm.set_debug(1, 20_000_000)  # 20 ms
    gemm.set_tuning(variant, 0, 0, 0)
    try:
        gemm.matmul(A, B, C)
        word = gemm.device_status()
    finally:
        gemm.set_debug(0, 0)
        gemm.set_tuning(0, 0, 0, 0)
    assert word & 0xF == 1
    # the MMA issuer (2) or the epilogue (3) runs out first; both wait on the stalled pipeline
    assert (word >> 4) & 0xF in (2, 3)
    gemm.reset_device_status()
    C, _ = _run(p)
    _check_full(p, C)
    assert gemm.device_status() == 0


# ---------------------------------------------------------------- the workloads
@pytest.mark.parametrize("name", ["bf16_512", "bf16_1024", "bf16_2048", "tf32_4096", "f16_4096", "bf16_4096",
                                  "bf16_ragged"])
def test_workload_full(name):
    p = inputs.workload(name)
    C, _ = _run(p)
    res = _check_full(p, C)
    print(name, res, gemm.last_plan())
    if name == "bf16_ragged":
        # 8200-byte rows of B and C: B is packed, so the TMA pair kernel runs
        assert gemm.last_plan()["kernel"] == 2


@pytest.mark.parametrize("name", ["bf16_8192", "bf16_16384", "bf16_proj"])
def test_workload_sampled(name):
    p = inputs.workload(name)
    n = inputs.WORKLOADS[name]["n"]
    C, _ = _run(p)
    res = _check_sampled(p, C, 3000 + n)
    print(name, res)


@pytest.mark.parametrize("dtype,layout,M", [("bf16", 0, 2600), ("tf32", 1, 3100), ("f16", 0, 700)])
def test_matmul_from_host_pipelined(dtype, layout, M):
    """The end-to-end call on pinned host operands (gemm_*_host): row blocks of
    A streamed in (2, 3 and 1 blocks here), blocks of C streamed out while the
    next block computes; every entry checked."""
    N, K = 700, 900
    p = inputs.make_problem("host", dtype, M, N, K, layout=layout, seed_a=61, seed_b=62)
    bufs = {}
    for _ in range(2):  # the second call reuses the library's staging and the pinned result
        C = gemm.matmul_from_host(p.a.pin_memory(), p.b.pin_memory(), layout=layout, buffers=bufs)
    _check_full(p, C)


def test_matmul_from_host_many_in_flight():
    """Three end-to-end products enqueued at once (wait=False): they take the
    stream's two staging slots in turn, so the third waits for the first's
    products before its uploads; every entry of each result checked. A call
    that reuses a pending call's result buffer waits for it, and returns its
    own product."""
    probs = [inputs.make_problem("fly", "tf32", 1500, 900, 700, seed_a=81, seed_b=82),
             inputs.make_problem("fly", "f16", 2100, 640, 1000, layout=1, seed_a=83, seed_b=84),
             inputs.make_problem("fly", "bf16", 3000, 1100, 500, seed_a=85, seed_b=86)]
    host = [(p.a.pin_memory(), p.b.pin_memory()) for p in probs]
    bufs = [{} for _ in probs]
    pending = [gemm.matmul_from_host(a, b, layout=p.layout, buffers=bf, wait=False)
               for (a, b), p, bf in zip(host, probs, bufs)]
    for (C, done), p in zip(pending, probs):
        done.synchronize()
        _check_full(p, C)
    # same buffers, other operands of the same shapes: the second call waits for the first
    q = inputs.make_problem("fly", "tf32", 1500, 900, 700, seed_a=87, seed_b=88)
    first, _ = gemm.matmul_from_host(*host[0], buffers=bufs[0], wait=False)
    C, done = gemm.matmul_from_host(q.a.pin_memory(), q.b.pin_memory(), buffers=bufs[0], wait=False)
    done.synchronize()
    assert C.data_ptr() == first.data_ptr()  # one pinned result per buffers dict
    _check_full(q, C)


@pytest.mark.parametrize("dtype,shape", [
    ("bf16", (256, 200, 1 << 18)),     # 2048 k-slabs: long accumulation, split segments of hundreds of slabs
    ("tf32", (130, 260, 1 << 16)),
    ("bf16", (1 << 20, 8, 64)),        # tall and skinny: 4096 tile rows
    ("f16", (8, 1 << 20, 64)),         # short and wide: thousands of tile columns, one ragged row block
])
def test_extreme_aspect_and_long_k(dtype, shape):
    """Long K (fp32 accumulation over 2^16-2^18 products) and extreme aspect
    ratios (one dimension 2^20, the others tiny), checked on sampled entries
    including every corner and the last row and column."""
    M, N, K = shape
    p = inputs.make_problem("extreme", dtype, M, N, K, seed_a=M % 97 + 1, seed_b=N % 89 + 2, dist_a="normal")
    C, _ = _run(p)
    _check_sampled(p, C, seed=M + N + K, count=2048)


def test_fp16_overflow_is_ieee_infinity():
    """Products beyond the binary16 range round to +-inf (RNE overflow); the
    last representable magnitude 65504 stays finite."""
    M, N, K = 4, 8, 16
    A = torch.full((M, K), 16.0, dtype=torch.float16, device="cuda")
    B = torch.full((K, N), 16.0, dtype=torch.float16, device="cuda")   # each entry 16*16*16 = 4096
    B[:, 1] = 300.0                                                     # 16*300*16 = 76800 > 65504
    B[:, 2] = -300.0
    B[:, 3] = 255.875                                                   # 16*255.875*16 = 65504
    C = gemm.matmul(A, B)
    torch.cuda.synchronize()
    assert torch.all(C[:, 0] == 4096.0)
    assert torch.all(C[:, 1] == float("inf")) and torch.all(C[:, 2] == float("-inf"))
    assert torch.all(C[:, 3] == 65504.0)


@pytest.mark.parametrize("dtype,shape,layout", [
    ("bf16", (4096, 4096, 4096), 0), ("tf32", (4096, 4096, 4096), 0), ("f16", (4096, 4096, 4096), 1),
    ("bf16", (8192, 8192, 2048), 0), ("bf16", (2048, 2048, 2048), 0), ("tf32", (2048, 2048, 2048), 0),
    ("bf16", (6144, 6144, 512), 0), ("tf32", (1024, 8192, 4096), 1), ("bf16", (768, 2560, 4096), 0),
])
def test_plan_query_matches_the_launched_plan(dtype, shape, layout):
    """gemm_plan_query (the cost model without a device, given this GPU's SM
    count) names the plan that the call then launches on a GB300."""
    props = torch.cuda.get_device_properties(0)
    if props.multi_processor_count != 152:
        pytest.skip("the plan query's cluster counts are those of a 152-SM GB300")
    M, N, K = shape
    p = inputs.make_problem("planq", dtype, M, N, K, layout=layout, seed_a=3, seed_b=4)
    _run(p)
    launched = gemm.last_plan()
    predicted = gemm.plan_query(dtype, M, N, K, layout=layout, sms=props.multi_processor_count)
    assert {k: launched[k] for k in predicted} == predicted
