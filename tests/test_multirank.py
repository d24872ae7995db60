"""The benchmark's multi-rank host logic on CPU with gloo, world size 2:
ranks run independent replicas, the job time is the maximum over ranks and
the whole-job value counts every rank's sequences."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, rank, world)
    local = 100.0 + 50.0 * rank          # rank 1 is the slow replica
    mx = bench.max_over_ranks(local)
    results[rank] = (mx, bench.job_tokens_per_s(world, 100, 30, mx))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 150.0
    assert res[0][1] == pytest.approx(2 * 100 * 30 / 0.150)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_tokens_per_s(1, 100, 10, 500.0) == pytest.approx(2000.0)
