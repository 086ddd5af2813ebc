"""Multi-rank host logic of bench.py, on CPU with two gloo ranks.

Under torchrun every rank runs its own K learners (independent problems) and
the job's throughput is all ranks' bytes over the slowest rank's time.  These
tests run the same aggregation helpers bench.py uses, over a real gloo process
group of world size 2, plus the reference arm's rank handling.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 1.5 ms per step on its own 1 GB of gradient
        ms = bench.max_over_ranks((rank + 1) * 1.5, "cpu")
        gbs = bench.job_gbs(world, 1e9, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "gbs": gbs}, f)
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == 3.0  # max of 1.5 and 3.0, seen identically on every rank
        assert r["gbs"] == pytest.approx(2 * 1e9 / 3.0e-3 / 1e9)


def test_single_process_needs_no_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.job_gbs(1, 4e9, 2.0) == pytest.approx(2000.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
