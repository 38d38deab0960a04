"""Replicas across GPUs: the benchmark's cross-rank timing logic, run as two
gloo ranks on CPU (the decode path itself has no exchange step)."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [12.5, 17.0][rank]  # rank 1 is the slow one
        ms = bench.max_over_ranks(my_ms, dist, "cpu")
        value = bench.whole_job_gbs(3_000_000_000, 10, world, ms)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_whole_job_value():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 17.0
        assert value == pytest.approx(3e9 * 10 * 2 / 17e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_gbs(1_000_000_000, 4, 1, 2.0) == pytest.approx(2000.0)
