"""Host logic of the benchmark's multi-GPU mode, on CPU: every rank runs an
independent replica (the GEMM has no exchange step); the job's time is the
slowest rank's and its throughput counts the work of all ranks.  Two gloo
ranks in separate processes, rendezvous on 127.0.0.1."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]                   # rank 1 is the slow one
    m = bench.max_over_ranks(ms)
    out[rank] = (m, bench.job_throughput(2.0 * 8192 ** 3, world, 5, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 12.5
    expect = 2.0 * 8192 ** 3 * 2 * 5 / 12.5e-3 / 1e12
    assert res[0][1] == pytest.approx(expect)


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(1e12, 1, 10, 1000.0) == pytest.approx(10.0)
