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


def table(rows: list[dict]) -> str:
    out = ["| workload | M×N×K | B layout | checked | entries | failing | max e_ij | p99 e_ij | accepted if | plan |",
           "|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        pl = r["plan"]
        kind = {1: "single CTA", 2: "CTA pair", 4: "2 pairs sharing A"}.get(pl["kernel"], str(pl["kernel"]))
        plan = f"{kind}, N-tile {pl['tile_n']}, last-round K segments {pl['tail_segs']}"
        out.append(f"| {r['name']} | {r['shape']} | {'K-major' if r['layout'] else 'row-major'} | {r['how']} | "
                   f"{r['n']} | {r['n_bad']} | {r['max_e']:.2e} | {r['p99_e']:.2e} | {RULE[r['dtype']]} | {plan} |")
    return "\n".join(out)


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--only", nargs="*", default=None, help="workload names (default: all)")
    ap.add_argument("--out", default=None, help="also write the table to this file")
    args = ap.parse_args()
    if not torch.cuda.is_available():
        print("parity_report: no CUDA device", file=sys.stderr)
        return 2
    gemm.load()
    names = args.only or list(inputs.WORKLOADS)
    rows = []
    for name in names:
        r = run_one(name)
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
