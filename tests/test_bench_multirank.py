"""Host logic of the multi-process benchmark: world_size-2 gloo ranks on CPU.

Each rank of `bench.py` under torchrun runs its own full replica of the
workload (independent problems, weak scaling).  The job's throughput is the
tokens all ranks processed divided by the slowest rank's time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    ms, value = bench.aggregate_over_ranks(local_ms[rank], 1000, 5, dist, torch.device("cpu"))
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    local_ms = [40.0, 50.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == pytest.approx(50.0)
        # 2 ranks x 1000 tokens x 5 steps in 50 ms
        assert value == pytest.approx(2 * 1000 * 5 / 0.050)


def test_single_process_needs_no_process_group():
    import bench
    ms, value = bench.aggregate_over_ranks(20.0, 100, 4)
    assert ms == 20.0 and value == pytest.approx(100 * 4 / 0.020)
