"""bench.py host logic without a GPU: rank aggregation over gloo (world size 2)
and the reference arm's JSON line (the CPU oracle on bounded samples)."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t_max = bench.reduce_max(1.0 + rank, world)           # per-rank step time
    total = bench.reduce_sum(100.0 * (rank + 1), world)   # bytes each rank streamed
    bench.barrier(world)
    q.put((rank, t_max, total))
    dist.destroy_process_group()


def test_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.0, 300.0), (1, 2.0, 300.0)]    # max time over ranks, sum of units


def _ref_cmd(extra=()):
    return [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "3",
            "--workload", "int8_row_1024x1024_s1", "--sample-seconds", "0.05", *extra]


def test_reference_arm_line():
    out = subprocess.run(_ref_cmd(), capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "int8_row_1024x1024_s1"


def test_reference_arm_two_ranks_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(30500 + os.getpid() % 1000)] + _ref_cmd()[1:]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2


def test_percentiles():
    sys.path.insert(0, ROOT)
    import bench
    p = bench.percentiles(list(range(1, 102)))          # 1 .. 101
    assert p == {"p10": 11.0, "p50": 51.0, "p90": 91.0}


def test_cpu_baseline_all_cores_and_one():
    """The oracle timed on all host cores and on one; the thread count is restored."""
    sys.path.insert(0, ROOT)
    import bench
    from oracle import oracle
    from weight_only_quantized_qgemv_gb300 import synth
    cores = oracle.threads()
    cpu = bench.cpu_baseline(synth.workload("int8_row_1024x1024_s1"), target_s=0.4)
    assert cpu["kind"] == "oracle" and cpu["unit"] == "GB/s" and cpu["value"] > 0
    assert cpu["cores"] == cores
    if cores > 1:
        assert cpu["single_core"]["cores"] == 1 and cpu["single_core"]["value"] > 0
    assert oracle.threads() == cores
