"""The multi-rank host logic of bench.py (replicas: barrier, max of step time over
ranks) on two CPU processes with the gloo backend."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    ws, r, local = bench.dist_setup("gloo")
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    got = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))
    q.put((rank, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_two_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
