"""The multi-process (torchrun) path of bench.py on CPU: two gloo ranks meet
at the barrier and agree on the max-over-ranks time and the whole-job
throughput (weak scaling: each rank verifies its own sequences)."""
import os
import socket
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup(world, backend="gloo")
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    local_ms = 10.0 * (rank + 1)            # rank 1 is the slower one
    value, ms = bench.job_throughput(local_ms, w, units_per_step_per_rank=40, steps=100)
    out[rank] = (value, ms)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_time_and_throughput():
    world = 2
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    value, ms = out[0]
    assert ms == 20.0                        # the max over ranks
    assert value == pytest.approx(world * 40 * 100 / 0.020)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(5.0, 1, units_per_step_per_rank=40, steps=10)
    assert ms == 5.0 and value == pytest.approx(40 * 10 / 0.005)
