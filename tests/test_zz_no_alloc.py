"""gemm_bf16_static_scratch: the BF16 product for callers that cannot allocate.

Such callers (a serving process whose memory pool owns the whole device, a
plug-in that must not allocate behind its host, a latency-bound path that
cannot absorb a cudaFree) get the same kernels as gemm_bf16 with the
split-tile scratch taken from the library's fixed 16 MiB device array. These
checks call it through the C interface, twice in a row per shape, and hold
each result to the float64 oracle with the acceptance rule of the parity
tests. The shapes whose plan splits its last round of tiles along K are
asserted to split, so their fp32 partial tiles provably pass through the
fixed array.

This file is collected last so that, if it fails, a run stopped at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""

import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20  # fp32 partial tiles the fixed array holds


def split_bytes(plan: dict) -> int:
    """Scratch the plan's split tail needs: every split work item holds one
    128 x tile_n fp32 partial per CTA of its cluster (four CTAs for the
    two-pair kernel, two otherwise)."""
    if plan["tail_segs"] <= 1:
        return 0
    ctas = 4 if plan["kernel"] == 4 else 2
    return (plan["work_items"] - plan["tail_start"]) * ctas * 128 * plan["tile_n"] * 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_gemm_tensor_gb300 import build
    build.build()
    gemm.load()
    gemm.set_debug(0, 0)
    gemm.set_tuning(0, 0, 0, 0)
    gemm.reset_device_status()
    yield
    assert gemm.device_status() == 0


def _reference_plan(p):
    """gemm_bf16's plan for the problem (the static call must launch the same)."""
    A, B = p.a.cuda(), p.b.cuda()
    C = torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda")
    code = gemm.gemm_bf16(p.M, p.N, p.K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, C.data_ptr(), p.N, 0, None)
    assert code == gemm.GEMM_OK
    torch.cuda.synchronize()
    return gemm.last_plan(), A, B


# (M, N, K, splits): the two split shapes take the CTA pair on the transposed
# product (192-row tiles, two K segments per split tile, 13.5 MiB of partials)
# and the plain CTA pair (224-wide tiles, two segments, 15.75 MiB: just inside
# the array); the others split nothing.
SHAPES = [(1024, 1536, 6144, True), (768, 2560, 6144, True), (4096, 4096, 4096, False), (300, 520, 200, False)]


@pytest.mark.parametrize("M,N,K,splits", SHAPES)
def test_matches_oracle_on_two_calls(M, N, K, splits):
    p = inputs.make_problem("noalloc", "bf16", M, N, K, dist_a="normal", dist_b="normal", seed_a=M + 3, seed_b=N + 5)
    plan, A, B = _reference_plan(p)
    need = split_bytes(plan)
    if splits:
        assert plan["tail_segs"] > 1, plan
        assert 0 < need <= SCRATCH_BYTES, (need, plan)
    else:
        assert need == 0, plan
    c_ref = oracle.gemm(M, N, K, p.a, p.lda, p.b, p.ldb, 0)
    s = oracle.abs_gemm(M, N, K, p.a, p.lda, p.b, p.ldb, 0)
    first = None
    for call in range(2):
        out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        code = gemm.gemm_bf16_static_scratch(M, N, K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, out.data_ptr(), N,
                                             0, None)
        assert code == gemm.GEMM_OK, gemm.status_string(code)
        torch.cuda.synchronize()
        assert gemm.last_plan() == plan  # the same kernels and split as gemm_bf16
        res = oracle.check(out.cpu().double().numpy(), c_ref, s, "bf16")
        assert res["ok"], f"call {call}: {res}"
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)  # the second call over the same array gives the same bits
    assert gemm.device_status() == 0


def test_plan_beyond_the_array_is_refused():
    """A plan whose split partials exceed the 16 MiB is refused with
    GEMM_ERR_SCRATCH_LIMIT before anything is launched."""
    M, N, K = 768, 3072, 6144  # CTA pair, 256-wide tiles, two segments: 18 MiB of partials
    p = inputs.make_problem("noalloc_big", "bf16", M, N, K, seed_a=11, seed_b=12)
    plan, A, B = _reference_plan(p)
    assert split_bytes(plan) > SCRATCH_BYTES, plan
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    launches = gemm.launch_count()
    code = gemm.gemm_bf16_static_scratch(M, N, K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, out.data_ptr(), N, 0,
                                         None)
    torch.cuda.synchronize()
    assert code == gemm.GEMM_ERR_SCRATCH_LIMIT
    assert gemm.launch_count() == launches
    assert torch.all(out == 7.0)
    assert "scratch" in gemm.status_string(code)
