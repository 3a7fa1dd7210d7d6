"""The N > 1 host logic of bench.py on CPU: two gloo ranks, max-over-ranks timing and
the weak-scaling shard assignment (no GPU needed)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    results[rank] = (ms, bench.rank_shard(rank, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        got = dict(results)
    assert got[0][0] == got[1][0] == 15.0
    assert got[0][1] == {"replica": 0, "of": 2} and got[1][1] == {"replica": 1, "of": 2}


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
