"""The bench's multi-rank host logic on CPU ranks (gloo, world size 2).

N > 1 runs independent replicas of the single-GPU layer; the only
cross-rank operations are a barrier and the max-over-ranks reduction of the
step time, and the whole-job throughput is N x tokens / slowest time.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.dist_barrier(world)
        # rank r pretends its timed region took 10 + 5 r ms
        slowest = bench.dist_max(10.0 + 5.0 * rank, world, device="cpu")
        q.put((rank, slowest, bench.replica_throughput(world, 4096, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_agree_on_the_slowest_time():
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
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] == pytest.approx(2 * 4096 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.dist_max(3.5, 1) == 3.5
    bench.dist_barrier(1)
    assert bench.replica_throughput(1, 4096, 2.0) == pytest.approx(2048000.0)
