"""The bench's N > 1 path (replicas, one rank per GPU) with two gloo ranks on
CPU: each rank reports its own timed-region time, every rank sees the
slowest one, and the whole-job value counts the work of all ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank             # rank 1 is the slow one
    slowest = bench.aggregate_ranks(ms, world, dist, "cpu")
    value = bench.whole_job_value(100, 1e9, slowest, world, 1e9)
    out[rank] = (slowest, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == 15.0
    # 2 ranks x 100 steps x 1 GB over 15 ms
    assert value == pytest.approx(2 * 100 * 1.0 / 0.015)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.aggregate_ranks(12.5, 1) == 12.5
    assert bench.whole_job_value(10, 2e9, 20.0, 1, 1e9) == pytest.approx(1000.0)
