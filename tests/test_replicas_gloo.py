"""The multi-GPU leg of the benchmark is replicas only: each rank runs the
whole path on its own GPU and the job's figures are the units summed over
ranks and the slowest rank's time.  Checked here on the CPU with two gloo
ranks (no GPU): the aggregation, and the reference arm's rule that only rank
0 runs and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, units, seconds, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        out[rank] = bench.aggregate(units[rank], seconds[rank])
    finally:
        dist.destroy_process_group()


def test_aggregate_sums_units_and_takes_the_slowest_rank():
    world = 2
    units = [1000.0, 3000.0]
    seconds = [0.5, 2.0]
    with mp.get_context("spawn").Manager() as mgr:  # no fork of this (threaded) process
        out = mgr.dict()
        mp.spawn(_rank, args=(world, free_port(), units, seconds, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (4000.0, 2.0)


def test_aggregate_without_a_process_group_is_the_rank_itself():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(12.0, 3.0) == (12.0, 3.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle"
        assert d["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []
