"""The multi-GPU path is replicas only (each rank runs the whole step on its own GPU; no
data-path collective).  Its host logic -- the slowest rank's step time through a MAX
all-reduce, and the whole-job throughput -- checked with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(0.5 + rank, world, "cpu")  # rank 1 is the slower one
        q.put((rank, ms, bench.job_tflops(1e9, 3, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tf in out:
        assert ms == 1.5                                   # MAX over ranks
        assert abs(tf - 2 * 3 * 1e9 / 1.5e-3 / 1e12) < 1e-9  # all ranks' FLOP / slowest time


def test_single_rank_is_unchanged():
    import bench
    assert bench.slowest_rank_ms(0.7, 1, "cpu") == 0.7
    assert abs(bench.job_tflops(1e9, 3, 1, 0.7) - 3e9 / 0.7e-3 / 1e12) < 1e-12
