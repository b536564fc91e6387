"""The N > 1 path of bench.py on the CPU: world_size-2 gloo process groups
stand in for the ranks of a torchrun launch (one process per GPU). The
layer does not shard (capacity and expert choice couple every token of a
batch), so ranks are replicas: the job's time is the slowest rank's and its
throughput counts every rank's tokens; only rank 0 prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as td
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]                       # rank 1 is the straggler
        got = bench.max_over_ranks(ms, torch.device("cpu"))
        rate = bench.job_rate(world, 4096, 10, got)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump({"max_ms": got, "rate": rate}, fh)
    finally:
        td.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_with_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["max_ms"] == 20.0                    # every rank sees the slowest time
        assert r["rate"] == pytest.approx(2 * 4096 * 10 / 0.020)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0, torch.device("cpu")) == 7.0
    assert bench.job_rate(1, 100, 5, 1000.0) == pytest.approx(500.0)


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs the reference arm; the others exit 0
    without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
