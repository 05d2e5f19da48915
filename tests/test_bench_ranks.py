"""Host logic of bench.py's multi-rank runs (one process per GPU, replicas of
the same workload): the timed region is the slowest rank's, and the reported
value is the whole job's throughput. Checked with two gloo ranks on the CPU."""
import os
import sys
import tempfile

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [120.0, 150.0][rank]  # rank 1 is the slow one
    ms = bench.reduce_max(local_ms, world, "cpu")
    value = bench.job_tflops(world, 9.0e11, 10, ms)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{ms} {value}\n")
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_max_time_and_job_throughput():
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(2, _free_port(), d), nprocs=2, join=True, start_method="spawn")
        got = [tuple(map(float, open(os.path.join(d, f"r{r}.txt")).read().split())) for r in range(2)]
    for ms, value in got:
        assert ms == 150.0  # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 9.0e11 * 10 / 0.150 / 1e12)  # both ranks' work over that time


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(12.5, 1, "cpu") == 12.5
    assert bench.job_tflops(1, 1e12, 4, 1000.0) == pytest.approx(4.0)
