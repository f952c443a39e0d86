"""Multi-rank path of the benchmark on CPU (gloo, world size 2): every rank
runs its own replica of the workload; the job's time is the slowest rank's and
its throughput counts the work of all ranks.  Only rank 0 of the reference arm
reports."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        dev_ms = 10.0 + 5.0 * rank          # the ranks' own timed regions
        got_ms, value = bench.job_value(dev_ms, world, steps=4, flops_per_step=1e9, dist=dist,
                                        device="cpu")
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": got_ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_job_value_two_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    slowest = 15.0
    for r in res:
        assert r["ms"] == pytest.approx(slowest)
        # 2 ranks x 4 steps x 1 GFLOP over 15 ms
        assert r["value"] == pytest.approx(2 * 4 * 1e9 / (slowest * 1e-3) / 1e12)


def test_job_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.job_value(8.0, 1, steps=2, flops_per_step=3e9)
    assert ms == 8.0 and value == pytest.approx(2 * 3e9 / 8e-3 / 1e12)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
