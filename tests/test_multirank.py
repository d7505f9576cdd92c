"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each timing its own replica.

The verify step has no exchange between sequences, so N GPUs run N independent replicas; the only
collective is the max over ranks of the timed region, and rank 0 reports the whole-job throughput.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [120.0, 150.0][rank]  # rank 1 is the slower replica
    m = bench.max_over_ranks(ms)
    v = bench.aggregate_nodes_per_s(world, 3, 100, m)
    q.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == 150.0
        assert v == pytest.approx(2 * 3 * 100 / 0.150)
