"""The replicas-only multi-GPU path of bench.py, run as two gloo ranks on
the CPU: the timed region is the slowest rank's, and the reported value
counts the bytes of every rank."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, ms_by_rank, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(ms_by_rank[rank], torch.device("cpu"), dist)
        out[rank] = (ms, bench.whole_job_gbs(1_000_000, 10, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_bytes():
    world, port = 2, _free_port()
    ms_by_rank = [1.5, 4.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, ms_by_rank, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, gbs = res[rank]
        assert ms == 4.0
        # 2 ranks x 10 steps x 1 MB in 4 ms = 5 GB/s
        assert gbs == pytest.approx(5.0)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(2.5, torch.device("cpu"), None) == 2.5
    assert bench.whole_job_gbs(2_000_000, 5, 1, 2.0) == pytest.approx(5.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank but 0 exits without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """Rank 0 prints one JSON line with the reference arm's keys (one step of
    the oracle on the host cores)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
