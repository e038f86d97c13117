"""The multi-rank host logic of bench.py (replicas: barrier, max-over-ranks time,
whole-job throughput) on two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist.barrier()
    local_ms = 10.0 + 5.0 * rank              # rank 1 is the slow one
    ms = bench.max_over_ranks(torch, dist, local_ms, torch.device("cpu"))
    value = bench.job_throughput(world, 8, 100, ms)
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == 15.0                                  # the slowest rank's time, on every rank
        assert abs(value - 2 * 8 * 100 / 0.015) < 1e-6      # all ranks' units / max time


def test_single_process_helpers():
    assert bench.max_over_ranks(torch, None, 3.5, None) == 3.5
    assert bench.job_throughput(1, 8, 1000, 50.0) == 8 * 1000 / 0.05
