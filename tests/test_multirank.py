"""Host-side rank logic of the benchmark on CPU: two gloo ranks.

The path shards by request (one independent pool per rank, no exchange), so
the only cross-rank work is the timing barrier and the max / sum reductions
of the whole-job number. These run here on gloo with world size 2."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, outdir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(w, "gloo")
    # rank-dependent step times and byte counts: the job takes the slowest
    # rank's time and the sum of the bytes
    t = 10.0 + 5.0 * rank
    b = 1000.0 * (rank + 1)
    bench.barrier(dist)
    res = {"max": bench.reduce_max(dist, t), "sum": bench.reduce_sum(dist, b)}
    # each rank draws its own inputs (seed + rank): distinct shards
    inp = bench.workloads.prompt_inputs("tiny", 0 + rank, requests=[0])
    res["k0"] = float(inp["k"][0, 0, 0])
    bench.barrier(dist)
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_reduce_and_shard(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    assert r0["max"] == r1["max"] == 15.0
    assert r0["sum"] == r1["sum"] == 3000.0
    assert r0["k0"] != r1["k0"]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.reduce_max(None, 3.5) == 3.5 and bench.reduce_sum(None, 2.0) == 2.0
    bench.barrier(None)


def test_reference_arm_other_ranks_exit_without_work(tmp_path):
    """Under torchrun only rank 0 runs the reference arm; rank 1 prints
    nothing and exits 0."""
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(free_port()))
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside torchrun starts two ranks itself; both join
    the process group and take distinct request shards (seeds 0 and 1)."""
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["n_gpus"] == 2 and line["rank_mask"] == 3 and line["seed_sum"] == 1
