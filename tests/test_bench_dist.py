"""Host logic of the benchmark's multi-rank path on CPU (gloo, world size 2):
the timings are reduced with a max over ranks and the whole-job throughput
counts every rank's work over the slowest rank's time (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        local_ms = [10.0 + rank, 5.0 - rank, 0.0]
        got = bench.reduce_max(local_ms)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 5.0, 0.0]


def test_whole_job_value_is_weak_scaling():
    one = bench.whole_job_tflops(10.988e12, 1, 7.0)
    assert bench.whole_job_tflops(10.988e12, 4, 7.0) == pytest.approx(4 * one)
    assert one == pytest.approx(10.988e12 / 7e-3 / 1e12)


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max([1.5, 2.5]) == [1.5, 2.5]
