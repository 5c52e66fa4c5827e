"""Context parallelism on CPU ranks (gloo): the row split, the gathers and the
gradient reduction of long_context_fm_gb300.cp, with the oracle as each
rank's computation.  Every rank's O, lse, dQ, dK, dV must equal the rows of
one single-process oracle run (fp64; the split changes only the order in
which dK and dV contributions are added)."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
from long_context_fm_gb300 import cp
from long_context_fm_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleLocal:
    """A rank's computation by the oracle: Q and dO are zero outside the
    rank's rows, so those rows add nothing to dK, dV (dP = 0, D = 0, dS = 0)."""

    def _mask(self, bounds):
        return {k: b.numpy() for k, b in zip(("lts", "lte", "uts", "ute"), bounds)}

    def _pad(self, x, k, q_row0):
        full = torch.zeros(k.shape, dtype=torch.float32)
        full[:, :, q_row0:q_row0 + x.shape[2]] = x
        return full

    def forward(self, q, k, v, bounds, q_row0, scale):
        rows = np.arange(q_row0, q_row0 + q.shape[2])
        O, L = oracle.forward(self._pad(q, k, q_row0), k, v, self._mask(bounds), scale, rows=rows)
        return torch.from_numpy(O), torch.from_numpy(L)

    def backward(self, q, k, v, o, lse, dO, bounds, q_row0, scale):
        rows = np.arange(q_row0, q_row0 + q.shape[2])
        g = oracle.backward(self._pad(q, k, q_row0), k, v, self._pad(dO, k, q_row0), self._mask(bounds), scale,
                            rows=rows)
        return torch.from_numpy(g["dq"]), torch.from_numpy(g["dk"]), torch.from_numpy(g["dv"])


def _inputs(wl):
    return tuple(t.float() for t in W.make_inputs(wl))


def _worker(rank, world, port, queue, wl, splits):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = W.make_mask(wl)
    q, k, v, dO = _inputs(wl)
    r0, r1 = splits[rank], splits[rank + 1]
    local_bounds = [torch.from_numpy(np.ascontiguousarray(m[x][:, :, r0:r1])) for x in ("lts", "lte", "uts", "ute")]
    shard = [t[:, :, r0:r1].contiguous() for t in (q, k, v, dO)]
    out = cp.step(*shard, local_bounds, splits, rank, wl.scale, OracleLocal())
    queue.put((rank, [t.numpy() for t in out]))
    dist.barrier()
    dist.destroy_process_group()


def _tile_costs(wl, m):
    lbl = oracle.tile_labels_all(m, 128, 128)            # [B, Hm, n_q, n_k]
    return (lbl != oracle.SKIP).sum(axis=(0, 1, 3))


@pytest.mark.parametrize("name,world", [("causal", 2), ("docs", 3)])
def test_cp_step_matches_single_process(name, world):
    if name == "causal":
        wl = W.Workload("cp_causal", B=1, H=2, N=600, d=16, mask="causal")
    else:
        wl = W.Workload("cp_docs", B=1, H=2, N=700, d=16, mask="docs_uniform", params=dict(lo=40, hi=260))
    m = W.make_mask(wl)
    splits = cp.balanced_splits(_tile_costs(wl, m), wl.N, world)
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, queue, wl, splits)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(queue.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    q, k, v, dO = _inputs(wl)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    for r in range(world):
        r0, r1 = splits[r], splits[r + 1]
        o, lse, dq, dk, dv = res[r]
        assert np.array_equal(o, O[:, :, r0:r1])                  # same arithmetic, same rows
        assert np.array_equal(lse, L[:, :, r0:r1])
        assert np.array_equal(dq, g["dq"][:, :, r0:r1])
        np.testing.assert_allclose(dk, g["dk"][:, :, r0:r1], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv, g["dv"][:, :, r0:r1], rtol=1e-12, atol=1e-13)


def test_balanced_splits_properties():
    rng = np.random.default_rng(3)
    for _ in range(50):
        N = int(rng.integers(128, 5000))
        n_t = -(-N // 128)
        world = int(rng.integers(1, min(n_t, 8) + 1))
        costs = rng.integers(0, 40, size=n_t)
        s = cp.balanced_splits(costs, N, world)
        assert s[0] == 0 and s[-1] == N and len(s) == world + 1
        assert all(s[r] < s[r + 1] for r in range(world))
        assert all(x % 128 == 0 for x in s[:-1])
        # greedy bound: no window exceeds the mean by more than one tile's cost
        parts = cp.split_costs(costs, s)
        assert max(parts) <= sum(parts) / world + costs.max() + 1e-6 or min(parts) == 0


def test_balanced_splits_beat_equal_rows_on_causal():
    """Causal tiles cost t + 1 key tiles: equal row counts leave the last rank
    with most of the work; the balanced split evens it out."""
    n_t, world = 64, 4
    costs = np.arange(1, n_t + 1)
    N = n_t * 128
    s = cp.balanced_splits(costs, N, world)
    bal = cp.split_costs(costs, s)
    eq = cp.split_costs(costs, [r * N // world for r in range(world)] + [N])
    assert max(bal) < 0.75 * max(eq)
    # every cut lands within one tile after its target, so each window is
    # within one tile's cost of the mean and two windows differ by less than two
    assert max(bal) - min(bal) < 2 * costs.max()
    assert s[1] > N // world                  # the first window gets more rows than N / world


def test_balanced_splits_rejects_bad_input():
    with pytest.raises(ValueError):
        cp.balanced_splits(np.ones(3), 1000, 2)             # wrong number of tiles
    with pytest.raises(ValueError):
        cp.balanced_splits(np.ones(2), 200, 3)              # more ranks than tiles
