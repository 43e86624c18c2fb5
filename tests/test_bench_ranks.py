"""The benchmark's whole-job reduction over ranks, with two gloo ranks on the
CPU: work is summed, times are the slowest rank's (weak scaling, no data
exchange between ranks)."""
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

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sums, maxs = bench.reduce_across_ranks([100 * (rank + 1), 7], [0.5 + rank, 2.0 - rank], "cpu")
        out[rank] = (sums, maxs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sum_work_and_max_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            sums, maxs = out[r]
            assert sums == [300.0, 14.0]
            assert maxs == [1.5, 2.0]


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_across_ranks([3, 4], [1.5], "cpu") == ([3.0, 4.0], [1.5])
