"""Multi-rank bookkeeping of the benchmark on CPU (gloo, world size 2): the job's step
time is the slowest rank's and throughput counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_attention_decode_02_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.5 if rank == 0 else 2.5  # rank 1 is the slow one
        m = replicas.max_over_ranks(ms)
        q.put((rank, m, replicas.job_throughput(1e9, m, world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, gbs in got:
        assert m == 2.5
        assert gbs == pytest.approx(2e9 / 2.5e-3 / 1e9)


def test_single_process_is_identity():
    assert replicas.max_over_ranks(3.25) == 3.25
    assert replicas.job_throughput(5e8, 1.0, 1) == pytest.approx(500.0)
