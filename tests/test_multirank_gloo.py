"""The benchmark's multi-GPU arithmetic on CPU: two gloo ranks, no GPU.

Each rank runs its own batch (the path needs no exchange: heads and PSA
batches are independent), the step time is the maximum over ranks, and the
job throughput counts every rank's work.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.5, 4.25][rank]  # rank 1 is the slow one
        ms = bench.reduce_max(local_ms, dist, "cpu")
        out[rank] = (ms, bench.job_throughput(world, 1e12, ms), bench.env_rank())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time_and_count_all_work():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, tflops, env = out[rank]
        assert ms == 4.25
        assert abs(tflops - 2 * 1e12 / 4.25e-3 / 1e12) < 1e-9
        assert env[0] == rank and env[1] == world


def test_single_rank_without_process_group():
    import bench
    assert bench.reduce_max(2.0) == 2.0
    assert bench.job_throughput(1, 2e12, 4.0) == pytest.approx(500.0)
