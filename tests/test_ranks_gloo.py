"""The bench's multi-rank path on CPU: two gloo ranks, each timing its own
batch, agree on the slowest rank's time and on the whole-job throughput."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local_ms = [120.0, 150.0][rank]          # rank 1 is the slow one
        dist.barrier()
        slowest = bench.max_over_ranks(local_ms, torch.device("cpu"), world)
        tflops = bench.job_tflops(2.0e12, 10, slowest, world)
        out[rank] = (slowest, tflops)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_slowest_time_and_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
        results = dict(out)
    assert results[0] == results[1]
    slowest, tflops = results[0]
    assert slowest == 150.0
    # 2 ranks × 10 steps × 2 TFLOP in 0.15 s
    assert abs(tflops - 2 * 10 * 2.0 / 0.150) < 1e-9


def test_single_rank_is_passthrough():
    import bench

    assert bench.max_over_ranks(42.0, torch.device("cpu"), 1) == 42.0
    assert abs(bench.job_tflops(1e12, 4, 2000.0, 1) - 2.0) < 1e-12
