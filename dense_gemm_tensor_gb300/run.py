"""Runs and times one product through the library (for profiling and quick
measurements): synthetic seeded operands of a given shape, dtype and B
layout, ``--iters`` launches on the current stream, the plan and the mean
time per launch (CUDA events, L2 not flushed) printed at the end.

    python -m dense_gemm_tensor_gb300.run --dtype e4m3 --M 8192 --N 8192 --K 8192 --layout 1 --iters 5
"""

from __future__ import annotations

import argparse

import torch

from . import build, gemm, inputs


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--dtype", default="bf16", choices=sorted(inputs.DTYPES))
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--layout", type=int, default=0, choices=(0, 1))
    ap.add_argument("--iters", type=int, default=5)
    args = ap.parse_args(argv)
    build.build()
    gemm.load()
    p = inputs.make_problem("run", args.dtype, args.M, args.N, args.K, layout=args.layout, seed_a=1, seed_b=2,
                            dist_a="normal", dist_b="normal")
    A, B = p.a.cuda(), p.b.cuda()
    out_dtype = torch.bfloat16 if args.dtype in ("e4m3", "e5m2") else A.dtype
    C = torch.empty((args.M, args.N), dtype=out_dtype, device="cuda")
    gemm.matmul(A, B, C, layout=args.layout)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.iters):
        gemm.matmul(A, B, C, layout=args.layout)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    flops = 2.0 * args.M * args.N * args.K
    print(f"{args.dtype} {args.M}x{args.N}x{args.K} layout {args.layout}: plan {gemm.last_plan()}, "
          f"{ms * 1e3:.1f} us per launch, {flops / (ms * 1e-3) / 1e12:.1f} TFLOP/s")


if __name__ == "__main__":
    main()
