"""Host-side logic of bench.py without a GPU: the max-over-ranks reduction
with two gloo ranks, the reference arm's rank handling, and its JSON line."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(1.5 + rank * 10.0, world)
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 11.5, 1: 11.5}


def test_reduce_max_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25


def test_reference_arm_other_ranks_do_no_work():
    sys.path.insert(0, ROOT)
    import bench
    line, rank = bench.run_reference(None, 2, 1)
    assert line is None and rank == 1


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-rows", "2"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("gemm_4096")


def test_bench_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2", "--impl", "reference"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_kernel_names_and_traffic_record():
    """The launch plan -> kernel name mapping (as ncu names the kernels) for
    every plan kind, and the committed traffic record: it names the kernels of
    the plans it was captured with and carries the device sources' hash."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.kernel_name("bf16", {"kernel": 1, "tile_n": 256}) == "gemm_kernel<1, 0, 256>"
    assert bench.kernel_name("tf32", {"kernel": 2, "tile_n": 224}) == "gemm_kernel_pair<2, 0, 224, 1>"
    assert bench.kernel_name("f16", {"kernel": 3, "tile_n": 224}) == "gemm_kernel_pair<0, 2, 224, 1>"
    assert bench.kernel_name("bf16", {"kernel": 4, "tile_n": 256}) == "gemm_kernel_pair<1, 0, 256, 2>"
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for dt in ("tf32", "f16", "bf16"):
        assert rec[dt]["kernel"].startswith("gemm_kernel") and rec[dt]["bytes"] > 0
    assert len(rec["kernel_sources_sha256"]) == 64
