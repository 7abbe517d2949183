"""The N>1 bench path on CPU: two gloo ranks, each timing its own replica
(weak scaling, no collective on the data path); the job figure takes the sum
of bytes and the max of elapsed times across ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = 0.5 + rank          # rank 1 is the slow one
    nbytes = 1000 * (rank + 1)
    t, b = bench.aggregate(elapsed, nbytes)
    results[rank] = (t, b, bench.dist_env())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, port, results), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        t, b, env = results[r]
        assert t == pytest.approx(1.5)      # max over ranks
        assert b == 3000                    # sum over ranks
        assert env == (2, r, 0)


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.aggregate(0.25, 123) == (0.25, 123)
