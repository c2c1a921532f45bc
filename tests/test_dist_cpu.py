"""The multi-process benchmark path on CPU (gloo, world_size 2): ranks meet at
the barrier, the step time is the slowest rank's, and the whole-job value
counts every rank's tokens."""
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


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    ms = [2.0, 3.5][rank]  # the second rank is slower
    slow = bench.max_over_ranks(ms, world, device="cpu")
    out[rank] = (slow, bench.whole_job_throughput(8192, world, slow))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_value():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.5
    assert res[0][1] == pytest.approx(8192 * 2 / 3.5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.whole_job_throughput(128, 1, 0.5) == pytest.approx(256000.0)
