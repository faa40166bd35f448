"""The multi-process host logic of bench.py, on CPU over gloo with two ranks.

Several GPUs run independent replicas of the layer (each rank its own batch, no exchange
on the data path), so the only cross-rank steps are the timing reduction (the slowest
rank's time) and the rule that rank 0 alone prints the result line."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, times, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    q.put((rank, bench.max_over_ranks(times[rank], dist, "cpu")))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 31.25]
    port = free_port()
    procs = [ctx.Process(target=_reduce_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 31.25, 1: 31.25}


def test_single_process_reduction_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.0, None, "cpu") == 7.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "3",
           "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["steps"] == 3 and res["warmup"] == 3
    assert res["value"] > 0 and res["e2e"]["value"] == res["value"]
    assert res["cpu_baseline"]["kind"] == "oracle"
