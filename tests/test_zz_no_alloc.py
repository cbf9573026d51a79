"""gemm_bf16_static_scratch: the BF16 product for callers that cannot allocate.

Such callers (a serving process whose memory pool owns the whole device, a
plug-in that must not allocate behind its host, a latency-bound path that
cannot absorb a cudaFree) get the same kernels as gemm_bf16 with the
split-tile scratch taken from the library's fixed 16 MiB device array. These
checks call it through the C interface and compare it with gemm_bf16, within
the acceptance tolerance the parity tests use, on two calls in a row.

This file is collected last so that, if it fails, a run stopped at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_tensor_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20          # fp32 partial tiles the fixed array holds
ITEM_BYTES = 2 * 128 * 256 * 4    # one split work item: both CTAs' 128 x 256 fp32 partials


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


def _pointers(p):
    A = p.a.cuda()
    B = p.b.cuda()
    return A, B


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (768, 2560, 4096), (300, 520, 200)])
def test_matches_gemm_bf16_on_two_calls(shape):
    M, N, K = shape
    p = inputs.make_problem("noalloc", "bf16", M, N, K, dist_a="normal", dist_b="normal", seed_a=M + 3, seed_b=N + 5)
    A, B = _pointers(p)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    code = gemm.gemm_bf16(M, N, K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, ref.data_ptr(), N, 0, None)
    assert code == gemm.GEMM_OK
    torch.cuda.synchronize()
    plan = gemm.last_plan()
    s = oracle.abs_gemm(M, N, K, p.a, p.lda, p.b, p.ldb, 0)
    want = ref.cpu().double().numpy()
    for call in range(2):
        out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        code = gemm.gemm_bf16_static_scratch(M, N, K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, out.data_ptr(), N,
                                             0, None)
        assert code == gemm.GEMM_OK, gemm.status_string(code)
        torch.cuda.synchronize()
        assert gemm.last_plan() == plan            # the same kernels and split as gemm_bf16
        got = out.cpu().double().numpy()
        diff = np.abs(got - want)
        assert np.all(diff <= oracle.allowed_error(want, s, "bf16")), f"call {call}: max diff {diff.max()}"
    assert gemm.device_status() == 0


def test_split_shape_uses_the_fixed_scratch_and_big_needs_are_refused():
    """A shape whose last round splits runs inside the 16 MiB; a plan needing
    more is refused with GEMM_ERR_SCRATCH_LIMIT and launches nothing."""
    # 1536 x 4864: 114 tiles of 256 x 256; with 76 co-resident pairs the last
    # round's 38 tiles split in two along K -> 76 items of 256 KiB = 19 MiB
    M, N, K = 1536, 4864, 4096
    p = inputs.make_problem("noalloc_big", "bf16", M, N, K, seed_a=11, seed_b=12)
    A, B = _pointers(p)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert gemm.gemm_bf16(M, N, K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, ref.data_ptr(), N, 0, None) == 0
    torch.cuda.synchronize()
    plan = gemm.last_plan()
    need = (plan["work_items"] - plan["tail_start"]) * ITEM_BYTES if plan["tail_segs"] > 1 else 0
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    launches = gemm.launch_count()
    code = gemm.gemm_bf16_static_scratch(M, N, K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, out.data_ptr(), N, 0,
                                         None)
    torch.cuda.synchronize()
    if need > SCRATCH_BYTES:
        assert code == gemm.GEMM_ERR_SCRATCH_LIMIT
        assert gemm.launch_count() == launches
        assert torch.all(out == 7.0)
        assert "scratch" in gemm.status_string(code)
    else:
        assert code == gemm.GEMM_OK
        assert torch.equal(out, ref)
