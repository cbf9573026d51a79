"""Runs and times one product through the library (for profiling and quick
measurements): synthetic seeded operands of a given shape, dtype and B
layout, ``--iters`` launches on the current stream, the plan and the mean
time per launch (CUDA events, L2 not flushed) printed at the end.
``--batch n`` runs a strided batch of n products in one launch (gemm.bmm);
``--beta``, ``--bias`` and ``--activation`` add the fused epilogue.

    python -m dense_gemm_tensor_gb300.run --dtype e4m3 --M 8192 --N 8192 --K 8192 --layout 1 --iters 5
    python -m dense_gemm_tensor_gb300.run --dtype bf16 --batch 128 --M 512 --N 512 --K 512 --iters 3
    python -m dense_gemm_tensor_gb300.run --dtype bf16 --beta 1 --bias --activation gelu --iters 3
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
    ap.add_argument("--batch", type=int, default=1, help="products in one strided-batch launch")
    ap.add_argument("--beta", type=float, default=0.0, help="fused epilogue: beta * C added")
    ap.add_argument("--bias", action="store_true", help="fused epilogue: a seeded bias per column")
    ap.add_argument("--activation", default=None, choices=[a for a in gemm.ACTIVATIONS if a])
    ap.add_argument("--iters", type=int, default=5)
    args = ap.parse_args(argv)
    build.build()
    gemm.load()
    fp8 = args.dtype in ("e4m3", "e5m2")
    mats = []
    for z in range(args.batch):
        p = inputs.make_problem("run", args.dtype, args.M, args.N, args.K, layout=args.layout, seed_a=1 + z,
                                seed_b=2 + z, dist_a="normal", dist_b="normal")
        mats.append((p.a[:, :args.K], p.b[:, :args.N] if args.layout == 0 else p.b[:, :args.K]))
    if args.batch == 1:
        A, B = mats[0][0].cuda(), mats[0][1].cuda()
    else:  # (8-bit operands stacked as bytes)
        def stack(ts):
            return torch.stack([t.view(torch.uint8) for t in ts]).view(ts[0].dtype) if fp8 else torch.stack(ts)
        A = stack([a.contiguous() for a, _ in mats]).cuda()
        B = stack([b.contiguous() for _, b in mats]).cuda()
    out_dtype = torch.bfloat16 if fp8 else A.dtype
    shape = (args.M, args.N) if args.batch == 1 else (args.batch, args.M, args.N)
    C = torch.randn(shape, device="cuda").to(out_dtype)
    epi = {}
    if args.beta != 0.0:
        epi["beta"] = args.beta
    if args.bias:
        epi["bias"] = torch.linspace(-1.0, 1.0, args.N, device="cuda").to(out_dtype)
    if args.activation:
        epi["activation"] = args.activation
    run = gemm.matmul if args.batch == 1 else gemm.bmm
    run(A, B, C, layout=args.layout, **epi)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.iters):
        run(A, B, C, layout=args.layout, **epi)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / max(args.iters, 1)
    flops = 2.0 * args.batch * args.M * args.N * args.K
    what = f"{args.batch} x " if args.batch > 1 else ""
    terms = ", ".join(f"{k}={v}" if k != "bias" else "bias" for k, v in epi.items())
    print(f"{args.dtype} {what}{args.M}x{args.N}x{args.K} layout {args.layout}{' epilogue ' + terms if epi else ''}: "
          f"plan {gemm.last_plan()}, {ms * 1e3:.1f} us per launch, {flops / (ms * 1e-3) / 1e12:.1f} TFLOP/s")


if __name__ == "__main__":
    main()
