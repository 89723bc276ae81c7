"""Multi-process (world size 2, gloo, CPU) check of the benchmark's replica
aggregation: each rank runs an independent replica, the job's time is the
maximum over ranks and its units the sum (weak scaling, no data exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        secs, units = bench.reduce_max_sum(1.0 + rank, 100 * (rank + 1))
        bench.barrier()
        out[rank] = (secs, units)
    finally:
        dist.destroy_process_group()


def test_max_time_sum_units_over_two_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res == {0: (2.0, 300.0), 1: (2.0, 300.0)}


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max_sum(0.5, 7) == (0.5, 7)
