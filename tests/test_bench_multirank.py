"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing
an independent replica, agree on the slowest rank's step time and report the
whole job's throughput (weak scaling, no data-path collective)."""

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


def _worker(rank, world, port, ms_by_rank, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier(world)
        value, ms = bench.job_throughput(4096, ms_by_rank[rank], world, device="cpu")
        out[rank] = (value, ms)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_take_slowest_rank():
    world = 2
    ms_by_rank = [0.25, 0.40]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), ms_by_rank, out), nprocs=world,
                 join=True)
        res = dict(out)
    for r in range(world):
        value, ms = res[r]
        assert ms == pytest.approx(0.40)
        assert value == pytest.approx(4096 * world / 0.40e-3)


def test_single_rank_is_local_time():
    import bench

    value, ms = bench.job_throughput(100, 2.0, 1)
    assert ms == 2.0 and value == pytest.approx(100 / 2e-3)
