"""Host logic of the multi-rank benchmark path, on CPU with gloo.

bench.py --gpus N runs one independent replica per rank (the retention path
has no exchange step); the job's time is the slowest rank's and its
throughput counts the units of every rank.  Two gloo ranks on 127.0.0.1 check
the max-over-ranks reduction and the aggregation that bench.py uses.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [12.5, 20.0][rank]              # rank 1 is the slower one
        ms = bench.max_over_ranks(per_rank_ms, world)
        value = bench.replica_throughput(16384 * 10, ms / 1e3, world)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_aggregate():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 20.0
        assert value == pytest.approx(2 * 16384 * 10 / 0.020)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.replica_throughput(100.0, 2.0, 1) == 50.0
