"""The multi-process (replica) path of bench.py on the CPU: two gloo ranks on 127.0.0.1
reduce their step times to the slowest one, and the whole-job throughput counts both
replicas' work over that time."""
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


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.0 + 0.5 * rank  # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, dist, "cpu")
        results[rank] = (ms_max, bench.replica_throughput(10.0, world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    # the port is free when picked but can be taken before the rendezvous binds it: a few tries
    for attempt in range(3):
        try:
            with mp.get_context("spawn").Manager() as m:
                results = m.dict()
                mp.spawn(_rank, args=(world, _free_port(), results), nprocs=world, join=True)
                got = dict(results)
            break
        except Exception:
            if attempt == 2:
                raise
    assert got[0][0] == got[1][0] == pytest.approx(1.5)
    # 2 replicas x 10 units in 1.5 ms
    assert got[0][1] == pytest.approx(2 * 10.0 / 1.5e-3)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.replica_throughput(4.0, 1, 2.0) == pytest.approx(2000.0)
