"""The multi-rank path of bench.py on CPU (gloo, world size 2): every rank
runs its own replica, and the only collective is the max over ranks of the
timings, taken after a barrier."""
import multiprocessing as mp
import os
import socket

import pytest
import torch
import torch.distributed as dist


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    out = bench.max_over_ranks([float(rank + 1), 10.0 * (world - rank)], world, torch.device("cpu"))
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 20.0]


def test_max_over_ranks_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 3.0], 1, torch.device("cpu")) == [1.5, 3.0]
