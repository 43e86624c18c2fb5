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


def test_code_hash_ignores_comments_and_whitespace_only(tmp_path):
    """A profile summary stays attached to its kernel across comment edits:
    the hash that bench.py compares drops comments and whitespace, and any
    change to the code itself changes it."""
    import bench

    a = tmp_path / "a.cu"
    a.write_text("// header\n__global__ void k(int *p) {\n  p[0] = 1;  /* one */\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// a different header\n\n__global__ void k(int *p)\n{ p[0] = 1; }\n")
    c = tmp_path / "c.cu"
    c.write_text("// header\n__global__ void k(int *p) {\n  p[0] = 2;  /* one */\n}\n")
    assert bench._code_sha256(str(a)) == bench._code_sha256(str(b))
    assert bench._code_sha256(str(a)) != bench._code_sha256(str(c))
