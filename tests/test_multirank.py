"""Host logic of the multi-GPU benchmark path on CPU: two gloo ranks (world size 2) agree on the
element-wise maximum of their timings, which is what the benchmark reports at N > 1."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        got = bench.max_over_ranks([1.0 + r, 10.0 - r, 0.5 * r], w)
        q.put((rank, r, w, local, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, local, got in results:
        assert (r, w, local) == (rank, 2, rank)
        assert got == [2.0, 10.0, 0.5]


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
