"""The multi-rank path of bench.py on the CPU: independent replicas, one per
rank, no data-path collective; the job's time is the slowest rank's and its
throughput counts the tokens of every rank.  Two gloo ranks on 127.0.0.1."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [1000.0, 1500.0][rank]      # rank 1 is the slow one
        ms_max, value = bench.job_rate(local_ms, world, tokens_per_rank=131072, steps=3, dist=dist)
        out.put((rank, ms_max, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, ms_max, value in res:
        assert ms_max == 1500.0
        assert value == pytest.approx(2 * 131072 * 3 / 1.5)


def test_job_rate_single_rank():
    ms_max, value = bench.job_rate(2000.0, 1, tokens_per_rank=1000, steps=4)
    assert ms_max == 2000.0 and value == pytest.approx(2000.0)
