"""The benchmark's multi-rank logic on CPU: two gloo ranks, as torchrun would
launch them, agree on the job-wide (max over ranks) step time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    dist, r, w = bench._dist()
    assert (r, w) == (rank, world)
    out[rank] = bench.job_max(dist, 1.5 + rank)  # rank 1 is the slower one
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    dist, r, w = bench._dist()
    assert dist is None and (r, w) == (0, 1)
    assert bench.job_max(None, 3.0) == 3.0
