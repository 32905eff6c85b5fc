"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2): replicas
only - each rank times its own copy of the workload, the job time is the max
over ranks and the job throughput counts every rank's work."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, _ = bench.dist_env()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow replica
        ms = bench.reduce_max(local_ms, ws, torch.device("cpu"))
        q.put((r, ws, ms, bench.job_tflops(ws, 1e12, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for _, ws, ms, tf in out:
        assert ws == 2 and ms == 15.0
        assert tf == pytest.approx(2 * 1e12 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1, None) == 3.5
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)
