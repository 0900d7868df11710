"""The bench's N > 1 path without GPUs: two gloo ranks on the CPU agree on
the slowest rank's time and on the whole-job throughput (independent
replicas, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 0.5 + rank          # rank 1 is the slow one
        m = bench.max_over_ranks(local)
        r, w, lr = bench.dist_env()
        out[rank] = (m, bench.job_throughput(w, 4096, 100, m), r, w, lr)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, value, r, w, lr = res[rank]
        assert m == pytest.approx(1.5)
        assert value == pytest.approx(2 * 4096 * 100 / 1.5)
        assert (r, w, lr) == (rank, world, rank)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.job_throughput(1, 4096, 10, 2.0) == pytest.approx(20480.0)
