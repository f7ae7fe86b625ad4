"""The multi-rank host path of the benchmark on CPU (gloo, world size 2).

The layer does not shard across GPUs in this build: N ranks run N
independent replicas with no data-path collective.  What the ranks share is
host plumbing, checked here without a GPU: the max over ranks of the timed
region, the whole-job aggregate, and the reference arm running on rank 0
only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.reduce_max(times[rank], world, device="cpu")
        dist.barrier()
        q.put((rank, m, bench.aggregate_rate(256, 100, world, m)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    world = 2
    times = [12.5, 17.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, rate in got:
        assert m == max(times)
        # 256 units per rank-step, 100 steps, 2 ranks, over the slowest rank's 17.25 ms
        assert rate == pytest.approx(256 * 100 * 2 / 17.25e-3, rel=1e-12)


def test_reduce_max_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate_rate(256, 10, 1, 2.0) == pytest.approx(256 * 10 / 2e-3)


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                           "--gpus", str(world), "--steps", "2", "--warmup", "1"],
                          capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)


def test_reference_arm_runs_on_rank0_only():
    """Under torchrun with N = 2 the reference arm (the CPU oracle) runs and
    prints on rank 0; the other rank exits 0 without work or output."""
    r1 = _reference(1, 2)
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
    r0 = _reference(0, 2)
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
