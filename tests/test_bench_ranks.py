"""The benchmark's multi-rank logic on CPU: two gloo ranks (one process per
rank, as torchrun would start them) agree on the slowest rank's time and on
the whole-job throughput."""
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


def _rank_main(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]
        got = bench.max_over_ranks(ms, dist, "cpu")
        tput = bench.whole_job_tflops(1e12, 4, world, got)
        out[rank] = (got, tput)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    # 2 ranks x 4 steps x 1 TFLOP in 20 ms -> 400 TFLOP/s
    assert res[0][1] == pytest.approx(400.0)


def test_single_process_is_the_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(2e12, 10, 1, 100.0) == pytest.approx(200.0)
