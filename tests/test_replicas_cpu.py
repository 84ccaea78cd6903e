"""Multi-rank host logic of the benchmark, on CPU with the gloo backend.

The path runs as independent replicas, one rank per GPU: no collective on the
data path, only the timing reduction (max over ranks) and rank 0 printing
the line.  These tests run that host logic with world size 2 on CPU.
"""

from __future__ import annotations

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


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (10 + r) ms for the timed steps and (20 - r) ms end to end
        elapsed, e2e = bench.max_over_ranks([10.0 + rank, 20.0 - rank], world)
        rate = bench.job_rate(1e9, 5, elapsed, world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(dict(elapsed=elapsed, e2e=e2e, rate=rate), f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_world2(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["elapsed"] == 11.0          # the slowest rank's time
        assert r["e2e"] == 20.0
        # whole job: 2 ranks x 1e9 units x 5 steps in 11 ms
        assert r["rate"] == pytest.approx(2 * 1e9 * 5 / 11e-3)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_rate(100.0, 2, 1000.0, 1) == pytest.approx(200.0)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
