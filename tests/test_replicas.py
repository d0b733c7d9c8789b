"""The multi-GPU path is independent replicas: each rank times its own steps
and rank 0 reports all ranks' bytes over the slowest rank's time.  This runs
that host logic on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local = [10.0 + rank, 2.0 * (world - rank), 0.5]
        got = bench.max_over_ranks(local)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res[0] == res[1] == [11.0, 4.0, 0.5]


def test_whole_job_value_counts_every_rank():
    import bench

    # 2 ranks, 3.375 GB each, slowest step 0.66 ms
    v = bench.whole_job_gbs(3_375_329_280, 2, 0.66)
    assert v == pytest.approx(2 * 3_375_329_280 / 0.66e-3 / 1e9)
    assert bench.whole_job_gbs(10**9, 1, 1.0) == pytest.approx(1000.0)
