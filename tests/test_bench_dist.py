"""The multi-process path of bench.py on CPU: two gloo ranks on 127.0.0.1 run the
same setup and aggregation code the GPU ranks run (replicas, no collective on the
data path): the whole-job time is the slowest rank's, the value counts the calls
of both ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    w, r, local, pg = bench.dist_setup()
    assert (w, r) == (world, rank) and pg is not None
    bench.barrier(pg)
    ms, us = bench.whole_job(pg, 1.0 + rank, w, torch.device("cpu"))
    q.put((rank, ms, us))
    pg.destroy_process_group()


def test_two_gloo_ranks_aggregate_as_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, us in got:
        assert ms == pytest.approx(2.0)      # the slower rank's time
        assert us == pytest.approx(1000.0)   # 2 calls (one per rank) in 2 ms
