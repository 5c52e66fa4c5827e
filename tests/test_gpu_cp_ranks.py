"""Context parallelism through the CUDA library on real ranks: two processes
(gloo group, collectives staged through host copies) each run cp.step with
LibraryLocal, both on one GPU, and every rank's O, lse, dQ, dK, dV
is compared with the oracle's rows of the whole mask.  The ranks' kernels
never wait on each other: every exchange is a host-side collective between
complete library calls."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_all, mode_for

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, queue, name, splits):
    import torch
    import torch.distributed as dist

    from long_context_fm_gb300 import cp, fm

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = W.SMALL[name] if name in W.SMALL else W.FULL[name]
        m = W.make_mask(wl)
        q, k, v, dO = W.make_inputs(wl)
        r0, r1 = splits[rank], splits[rank + 1]
        local_bounds = [torch.from_numpy(np.ascontiguousarray(m[x][:, :, r0:r1])).cuda()
                        for x in ("lts", "lte", "uts", "ute")]
        shard = [t[:, :, r0:r1].contiguous().cuda() for t in (q, k, v, dO)]
        flags = fm.FM_FLAG_PRECISE if mode_for(wl) else 0
        out = cp.step(*shard, local_bounds, splits, rank, wl.scale, cp.LibraryLocal(flags))
        torch.cuda.synchronize()
        queue.put((rank, [t.cpu().numpy() for t in out]))
        dist.barrier()
    except BaseException as e:          # report instead of leaving the parent waiting
        queue.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,world", [("docs_small", 2), ("window_sink_small", 2), ("lognormal_small", 2)])
def test_cp_step_through_the_library_matches_the_oracle(name, world):
    from long_context_fm_gb300 import cp

    wl = W.SMALL[name]
    m = W.make_mask(wl)
    costs = (oracle.tile_labels_all(m, 128, 128) != oracle.SKIP).sum(axis=(0, 1, 3))
    splits = cp.balanced_splits(costs, wl.N, world)
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, queue, name, splits)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in procs:
            r, val = queue.get(timeout=600)
            res[r] = val
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.kill()
    for r in range(world):
        assert not isinstance(res[r], str), f"rank {r}: {res[r]}"
    assert all(p.exitcode == 0 for p in procs)
    q, k, v, dO = W.make_inputs(wl)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    for r in range(world):
        r0, r1 = splits[r], splits[r + 1]
        o, lse, dq, dk, dv = res[r]
        check_all([(f"O rank {r}", o, O[:, :, r0:r1]), ("lse", lse, L[:, :, r0:r1]),
                   (f"dQ rank {r}", dq, g["dq"][:, :, r0:r1]), (f"dK rank {r}", dk, g["dk"][:, :, r0:r1]),
                   (f"dV rank {r}", dv, g["dv"][:, :, r0:r1])])
