"""Runs a set of products through the range-checked build of the library
(libdgt_gemm_checked.so) and reports, as one JSON line, the device status
word and each product's acceptance against the CPU oracle. Run as a separate
process by tests/test_gpu_checked.py (the checked build replaces the default
library in this process)."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from dense_gemm_tensor_gb300 import build, gemm, inputs  # noqa: E402


def main():
    gemm.load(build.build(checked=True))
    gemm.set_debug(0, 0)
    gemm.reset_device_status()
    results = {}

    def check(name, p, C, dtype=None, **epi):
        if p.dtype in ("e4m3", "e5m2"):
            a, b = oracle.decode_fp8(p.a, p.dtype), oracle.decode_fp8(p.b, p.dtype)
        else:
            a, b = p.a, p.b
        ref = oracle.gemm_epilogue(p.M, p.N, p.K, a, p.lda, b, p.ldb, p.layout, **epi)
        s = oracle.gemm_epilogue_scale(p.M, p.N, p.K, a, p.lda, b, p.ldb, p.layout, **epi)
        res = oracle.check(C.cpu().double().numpy(), ref, s, dtype or p.dtype)
        results[name] = bool(res["ok"])

    cases = [("bf16", 0, 1, 256), ("bf16", 1, 2, 224), ("f16", 0, 3, 192), ("tf32", 0, 2, 256), ("tf32", 1, 1, 128),
             ("bf16", 0, 4, 224), ("tf32", 0, 4, 256)]
    for dtype, layout, variant, bn in cases:
        p = inputs.make_problem("chk", dtype, 700, 900, 520, layout=layout, seed_a=1, seed_b=2, dist_a="normal")
        gemm.set_tuning(variant, bn, 0, 0)
        C = gemm.matmul(p.a.cuda(), p.b.cuda(), layout=layout)
        torch.cuda.synchronize()
        check(f"{dtype}-l{layout}-v{variant}-{bn}", p, C)
    # split tail with the fused epilogue
    p = inputs.make_problem("chks", "bf16", 768, 2560, 4096, seed_a=3, seed_b=4, dist_a="normal")
    gemm.set_tuning(2, 256, 0, 0)
    C = gemm.matmul(p.a.cuda(), p.b.cuda(), alpha=0.5, activation="gelu")
    torch.cuda.synchronize()
    results["split_segments"] = gemm.last_plan()["tail_segs"]
    check("bf16-split-gelu", p, C, alpha=0.5, act=oracle.ACT_GELU)
    # the transposed product's split tail with the fused epilogue (beta * C read)
    p = inputs.make_problem("chkt", "tf32", 768, 2560, 4096, seed_a=9, seed_b=10, dist_a="normal")
    C0 = torch.ones(768, 2560, dtype=torch.float32)
    C = C0.cuda()
    gemm.set_tuning(4, 256, 0, 0)
    gemm.matmul(p.a.cuda(), p.b.cuda(), C, beta=-0.5, activation="relu")
    torch.cuda.synchronize()
    results["swap_split_segments"] = gemm.last_plan()["tail_segs"]
    check("tf32-swap-split-relu", p, C, beta=-0.5, c_in=C0.double().numpy(), act=oracle.ACT_RELU)
    gemm.set_tuning(0, 0, 0, 0)
    # copy-warp path (unaligned rows read in place)
    gemm.set_debug(2, 0)
    p = inputs.make_problem("chku", "bf16", 260, 450, 300, lda=301, ldb=451, seed_a=5, seed_b=6)
    C = gemm.matmul(p.a.cuda()[:, :300], p.b.cuda()[:, :450])
    torch.cuda.synchronize()
    gemm.set_debug(0, 0)
    check("bf16-copy-warps", p, C)
    # FP8 with a row-major B (transposed into scratch)
    p = inputs.make_problem("chk8", "e4m3", 520, 390, 1024, seed_a=7, seed_b=8, dist_a="normal")
    C = gemm.matmul(p.a.cuda(), p.b.cuda())
    torch.cuda.synchronize()
    check("e4m3-row-major-b", p, C, dtype="bf16")
    results["status"] = gemm.device_status()
    print(json.dumps(results))


if __name__ == "__main__":
    main()
