"""Parity report: every synthetic workload through the C interface, checked
against the CPU oracle, printed as a Markdown table of the normalised error
e_ij = |C_gpu - C_ref| / sum_k |A_ik||B_kj| (bare, without the one-ulp
allowance that acceptance adds for FP16/BF16 outputs).

    python tests/parity_report.py [--only NAME ...] [--out FILE]

Needs a GB300 and the built library. Products of at most 4096^3
multiply-adds (the ragged 4000x4100x4104 case among them) are checked in
full, larger ones on 4096 seeded sampled entries plus the corners and a
stride through the last row and column. The acceptance rule is the one
the parity tests use: |C_gpu - C_ref| <= 1e-3 * S + one output ulp (FP16,
BF16) or <= 4e-3 * S (TF32).
"""

import argparse
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch  # noqa: E402

import oracle  # noqa: E402
from dense_gemm_tensor_gb300 import gemm, inputs  # noqa: E402

TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}
RULE = {"bf16": "1e-3·S + 1 ulp", "f16": "1e-3·S + 1 ulp", "tf32": "4e-3·S"}
FULL_LIMIT = 4096 ** 3  # products of at most this many multiply-adds are checked in full


def run_one(name: str) -> dict:
    p = inputs.workload(name)
    A = p.a.cuda()
    B = p.b.cuda()
    a = A[:, :p.K]
    b = B[:, :p.N] if p.layout == 0 else B[:, :p.K]
    C = torch.empty((p.M, p.N), dtype=TORCH_DT[p.dtype], device="cuda")
    gemm.matmul(a, b, C, layout=p.layout)
    torch.cuda.synchronize()
    plan = gemm.last_plan()
    t0 = time.perf_counter()
    if p.M * p.N * p.K <= FULL_LIMIT:
        c_ref = oracle.gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
        s = oracle.abs_gemm(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout)
        got = C.cpu().double().numpy()
        how = "full"
    else:
        n = inputs.WORKLOADS[name]["n"]
        r, c = inputs.sample_entries(p.M, p.N, 4096, 3000 + n)
        got = C[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu().double().numpy()
        c_ref, s = oracle.gemm_entries(p.M, p.N, p.K, p.a, p.lda, p.b, p.ldb, p.layout, r, c)
        how = "sampled"
    res = oracle.check(got, c_ref, s, p.dtype)
    res.update(name=name, dtype=p.dtype, shape=f"{p.M}×{p.N}×{p.K}", layout=p.layout, how=how, plan=plan,
               oracle_s=time.perf_counter() - t0)
    del A, B, C
    torch.cuda.empty_cache()
    return res


def _extra(dtype: str, M: int, N: int, seed: int):
    """C_in (N(0, 2^2)) and bias (U[-1, 1)) in the output type, seeded."""
    c_in = inputs.to_dtype(inputs.draw(M, N, "normal", seed, 2.0), dtype)
    bias = inputs.to_dtype(inputs.draw(1, N, "uniform", seed + 1), dtype)[0]
    return c_in, bias


def run_epilogue(name: str, dtype: str, act: str) -> dict:
    """act(0.75 A.B - 0.5 C_in + bias) at 4096^3, N(0,1) operands, in full
    against the oracle's epilogue with its error scale."""
    n = 4096
    p = inputs.make_problem(name, dtype, n, n, n, seed_a=1103, seed_b=2103, dist_a="normal", dist_b="normal")
    c_in, bias = _extra(dtype, n, n, seed=4103)
    C = c_in.cuda()
    gemm.matmul(p.a.cuda()[:, :n], p.b.cuda()[:, :n], C, alpha=0.75, beta=-0.5, bias=bias.cuda(), activation=act)
    torch.cuda.synchronize()
    plan = gemm.last_plan()
    t0 = time.perf_counter()
    kw = dict(alpha=0.75, beta=-0.5, c_in=c_in.double().numpy(), bias=bias.double().numpy(),
              act={"relu": oracle.ACT_RELU, "gelu": oracle.ACT_GELU, "gelu_tanh": oracle.ACT_GELU_TANH}[act])
    ref = oracle.gemm_epilogue(n, n, n, p.a, p.lda, p.b, p.ldb, 0, **kw)
    s = oracle.gemm_epilogue_scale(n, n, n, p.a, p.lda, p.b, p.ldb, 0, **kw)
    res = oracle.check(C.cpu().double().numpy(), ref, s, dtype)
    res.update(name=name, dtype=dtype, shape=f"{n}×{n}×{n}", layout=0, how="full", plan=plan,
               oracle_s=time.perf_counter() - t0, rule=RULE[dtype] + " (S of the epilogue)")
    return res


def run_fp8(name: str, fmt: str, n: int) -> dict:
    """FP8 product, N(0,1) cast to the format, K-major B, bfloat16 C; in full
    up to 4096^3, else on sampled entries, on the decoded operand values."""
    p = inputs.make_problem(name, fmt, n, n, n, layout=1, seed_a=1200 + n % 97, seed_b=2200 + n % 97,
                            dist_a="normal", dist_b="normal")
    C = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
    gemm.matmul(p.a.cuda()[:, :n], p.b.cuda()[:, :n], C, layout=1)
    torch.cuda.synchronize()
    plan = gemm.last_plan()
    t0 = time.perf_counter()
    av, bv = oracle.decode_fp8(p.a, fmt), oracle.decode_fp8(p.b, fmt)
    if n ** 3 <= FULL_LIMIT:
        ref = oracle.gemm(n, n, n, av, p.lda, bv, p.ldb, 1)
        s = oracle.abs_gemm(n, n, n, av, p.lda, bv, p.ldb, 1)
        got, how = C.cpu().double().numpy(), "full"
    else:
        r, c = inputs.sample_entries(n, n, 4096, 3300 + n % 97)
        got = C[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu().double().numpy()
        ref, s = oracle.gemm_entries(n, n, n, av, p.lda, bv, p.ldb, 1, r, c)
        how = "sampled"
    res = oracle.check(got, ref, s, "bf16")
    res.update(name=name, dtype=fmt, shape=f"{n}×{n}×{n}", layout=1, how=how, plan=plan,
               oracle_s=time.perf_counter() - t0, rule=RULE["bf16"] + " (bf16 C)")
    return res


def run_batched(name: str, dtype: str, batch: int, n: int) -> dict:
    """A strided batch of batch x n^3 products, U[-1,1) operands, every matrix in full."""
    A = torch.stack([inputs.to_dtype(inputs.draw(n, n, "uniform", 1300 + z), dtype) for z in range(batch)])
    B = torch.stack([inputs.to_dtype(inputs.draw(n, n, "uniform", 2300 + z), dtype) for z in range(batch)])
    C = gemm.bmm(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    plan = gemm.last_plan()
    t0 = time.perf_counter()
    a, b = A.reshape(-1), B.reshape(-1)
    ref = oracle.gemm_strided_batched(batch, n, n, n, a, n, n * n, b, n, n * n, 0)
    s = oracle.abs_gemm_strided_batched(batch, n, n, n, a, n, n * n, b, n, n * n, 0)
    res = oracle.check(C.cpu().double().numpy(), ref, s, dtype)
    res.update(name=name, dtype=dtype, shape=f"{batch} × {n}×{n}×{n}", layout=0, how="full", plan=plan,
               oracle_s=time.perf_counter() - t0)
    return res


EXTRA = {
    "epi_bf16_4096_gelu": lambda: run_epilogue("epi_bf16_4096_gelu", "bf16", "gelu"),
    "epi_tf32_4096_relu": lambda: run_epilogue("epi_tf32_4096_relu", "tf32", "relu"),
    "e4m3_4096": lambda: run_fp8("e4m3_4096", "e4m3", 4096),
    "e5m2_4096": lambda: run_fp8("e5m2_4096", "e5m2", 4096),
    "e4m3_8192": lambda: run_fp8("e4m3_8192", "e4m3", 8192),
    "bf16_batched_8x1024": lambda: run_batched("bf16_batched_8x1024", "bf16", 8, 1024),
}


def table(rows: list[dict]) -> str:
    out = ["| workload | M×N×K | B layout | checked | entries | failing | max e_ij | p99 e_ij | accepted if | plan |",
           "|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        pl = r["plan"]
        kind = {1: "single CTA", 2: "CTA pair", 3: "CTA pair on C^T",
                4: "2 pairs sharing A"}.get(pl["kernel"], str(pl["kernel"]))
        plan = f"{kind}, N-tile {pl['tile_n']}, last-round K segments {pl['tail_segs']}"
        out.append(f"| {r['name']} | {r['shape']} | {'K-major' if r['layout'] else 'row-major'} | {r['how']} | "
                   f"{r['n']} | {r['n_bad']} | {r['max_e']:.2e} | {r['p99_e']:.2e} | {r.get('rule', RULE.get(r['dtype']))} | "
                   f"{plan} |")
    return "\n".join(out)


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--only", nargs="*", default=None,
                    help="workload names (default: all): " + ", ".join(list(inputs.WORKLOADS) + list(EXTRA)))
    ap.add_argument("--out", default=None, help="also write the table to this file")
    args = ap.parse_args()
    if not torch.cuda.is_available():
        print("parity_report: no CUDA device", file=sys.stderr)
        return 2
    gemm.load()
    names = args.only or list(inputs.WORKLOADS) + list(EXTRA)
    rows = []
    for name in names:
        r = EXTRA[name]() if name in EXTRA else run_one(name)
        print(f"{name}: ok={r['ok']} n={r['n']} max_e={r['max_e']:.3e} p99_e={r['p99_e']:.3e} "
              f"oracle {r['oracle_s']:.1f} s", flush=True)
        rows.append(r)
    text = table(rows)
    print(text)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    return 0 if all(r["ok"] for r in rows) else 1


if __name__ == "__main__":
    sys.exit(main())
