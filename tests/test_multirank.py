"""Host-side logic of the N-rank benchmark (replicas, weak scaling) on 2 gloo ranks (CPU)."""
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
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]                      # rank 1 is the slow replica
        m = bench.rank_max(dist, ms)
        thr = bench.weak_throughput(1000, world, m)
        dist.barrier()
        q.put((rank, m, thr))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, thr in res:
        assert m == 5.0                            # both ranks see the slowest time
        assert thr == pytest.approx(2 * 1000 / 5e-3)


def test_single_rank_is_identity():
    assert bench.rank_max(None, 2.5) == 2.5
    assert bench.weak_throughput(655360, 1, 1.0) == pytest.approx(655360e3)
