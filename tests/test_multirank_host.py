"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

The decode shards by sequence with no exchange on the data path (each rank
runs its own replica of the workload); the ranks share only a barrier and a
max-reduction of their times, and for the reference arm rank 0 alone runs.
These run as two spawned processes with a gloo process group on 127.0.0.1.
"""
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


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._barrier(world)
    results[f"max{rank}"] = bench._max_over_ranks(10.0 * (rank + 1), world)  # rank r reports 10 (r + 1)
    bench._barrier(world)
    dist.destroy_process_group()
    # the reference arm: only rank 0 works; the others return at once without a process group
    if rank != 0:
        results[f"ref{rank}"] = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"])


@pytest.mark.timeout(300)
def test_two_gloo_ranks_share_only_a_barrier_and_a_max():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True,
                       start_method="spawn")
    assert results["max0"] == results["max1"] == 20.0
    assert results["ref1"] == 0
