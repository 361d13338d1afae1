"""Host logic of bench.py for N > 1 ranks, on CPU: world_size-2 gloo groups.

With one process per GPU every rank verifies its own bs=64 batch (replicas,
no data-path collective); the job's step time is the slowest rank's, taken
with one all-reduce of a scalar, and the rate counts every rank's units.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        job_ms = bench.max_over_ranks(ms[rank], dist, "cpu")
        out[rank] = job_ms
        out[world + rank] = bench.whole_job_rate(512, world, job_ms)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_rate_gloo(world):
    ms = [0.150, 0.175][:world]
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    tmp.spawn(_rank_main, args=(world, _free_port(), ms, out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == pytest.approx(max(ms))                       # slowest rank's time
        assert out[world + r] == pytest.approx(world * 512 / (max(ms) / 1e3))


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(0.2, None, "cpu") == 0.2
    assert bench.whole_job_rate(512, 1, 0.2) == pytest.approx(512 / 2e-4)


def test_config_names_replicas():
    assert bench.config_dict(0.5, 1)["parallelism"] == "single GPU"
    assert bench.config_dict(0.5, 4)["parallelism"] == "replicas x4"


def test_reference_arm_non_zero_rank_exits_quietly():
    # under torchrun only rank 0 runs and prints the oracle line
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
