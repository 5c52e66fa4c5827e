"""Context parallelism: one sequence split over ranks by rows.

Blog "FlashMask技术" §4.3 (sequence-parallel integration): the column
intervals are all-gathered (item 1), key/value shards that a rank's rows
never attend are skipped whole (item 2), and the work is split by the number
of effective (non-skipped) blocks (item 3).

Rank r holds rows [s_r, s_{r+1}) of Q, K, V, dO and the column bounds of its
columns [s_r, s_{r+1}).  One step:

1. all-gather the column bounds: every rank holds the whole O(N) mask;
2. all-gather the K and V shards into full-length K, V in local memory (no
   remote reads inside a kernel), while the rank's row window is classified
   (once, for the forward and the backward);
3. forward for the rank's rows against all keys (``fm_attn_fwd_rows``); the
   tile labels of the row window skip every key tile, hence every key shard,
   that those rows never attend;
4. backward for the rank's rows (``fm_attn_bwd_rows``): dQ is complete
   locally; the dK, dV contributions of all ranks are summed and scattered in
   one reduce-scatter, so each rank receives only the sum over its own rows.

The split ``balanced_splits`` is chosen before the data is distributed, from
per-Q-tile costs (non-skip key tiles per Q tile, over batches and mask
heads): contiguous, 128-row aligned windows of nearly equal cost.

The per-rank computation is a parameter (``LibraryLocal`` runs the CUDA
library on the rank's GPU); the collectives come from ``torch.distributed``
and run over NCCL or gloo alike.  A gloo group moves host tensors only, so
with gloo the device tensors of a collective are staged through host copies
(NCCL takes them as they are).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

TILE = 128


def balanced_splits(costs, N: int, world: int, tile: int = TILE):
    """Row boundaries s_0 = 0 < s_1 < ... < s_world = N (multiples of `tile`
    except the last) that split the per-Q-tile `costs` (length ceil(N / tile))
    into `world` contiguous parts of nearly equal sum.  Greedy on the prefix
    sums: window r ends at the first tile where the running cost reaches
    (r + 1) / world of the total; every window keeps at least one tile."""
    costs = np.asarray(costs, dtype=np.float64)
    n_t = -(-N // tile)
    if costs.shape != (n_t,):
        raise ValueError(f"costs must have ceil(N / {tile}) = {n_t} entries")
    if world < 1 or world > n_t:
        raise ValueError(f"world must be in [1, {n_t}]")
    w = np.maximum(costs, 0) + 1e-9              # empty tiles still cost a launch slot
    prefix = np.cumsum(w)
    total = prefix[-1]
    cuts = [0]
    for r in range(1, world):
        target = total * r / world
        t = int(np.searchsorted(prefix, target, side="left")) + 1     # tiles in windows 0..r-1
        t = max(t, cuts[-1] + 1)                                      # at least one tile each
        t = min(t, n_t - (world - r))                                 # leave one for every later window
        cuts.append(t)
    cuts.append(n_t)
    return [min(c * tile, N) for c in cuts]


def split_costs(costs, splits, tile: int = TILE):
    """Cost of each window of `splits`."""
    costs = np.asarray(costs, dtype=np.float64)
    return [float(costs[splits[r] // tile: -(-splits[r + 1] // tile)].sum()) for r in range(len(splits) - 1)]


def _host_staged(group, t: torch.Tensor) -> bool:
    """True when the group's backend moves host tensors only (gloo) and `t`
    lives on a GPU: the collective then runs on a host copy."""
    return t.is_cuda and dist.get_backend(group) == "gloo"


def _gather_dim(local: torch.Tensor, splits, dim: int, group=None) -> torch.Tensor:
    """All-gather the per-rank slices of one axis (lengths from `splits`) into
    the full axis; pieces are padded to the longest so the collective sees
    equal sizes."""
    world = len(splits) - 1
    lens = [splits[r + 1] - splits[r] for r in range(world)]
    Lmax = max(lens)
    pad_shape = list(local.shape)
    pad_shape[dim] = Lmax
    staged = _host_staged(group, local)
    send = local.new_zeros(pad_shape, device="cpu" if staged else local.device)
    send.narrow(dim, 0, local.shape[dim]).copy_(local)
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    out = torch.cat([recv[r].narrow(dim, 0, lens[r]) for r in range(world)], dim=dim).contiguous()
    return out.to(local.device) if staged else out


def _gather_dim_start(local: torch.Tensor, splits, dim: int, group=None):
    """Start the all-gather of ``_gather_dim`` without waiting for it; returns
    a function that waits and assembles the full axis."""
    world = len(splits) - 1
    lens = [splits[r + 1] - splits[r] for r in range(world)]
    pad_shape = list(local.shape)
    pad_shape[dim] = max(lens)
    staged = _host_staged(group, local)
    send = local.new_zeros(pad_shape, device="cpu" if staged else local.device)
    send.narrow(dim, 0, local.shape[dim]).copy_(local)
    recv = [torch.empty_like(send) for _ in range(world)]
    work = dist.all_gather(recv, send, group=group, async_op=True)

    def finish() -> torch.Tensor:
        work.wait()
        out = torch.cat([recv[r].narrow(dim, 0, lens[r]) for r in range(world)], dim=dim).contiguous()
        return out.to(local.device) if staged else out

    return finish


def reduce_scatter_rows(full: torch.Tensor, splits, rank: int, group=None) -> torch.Tensor:
    """Sum the ranks' full-length contributions [B, H, N, d] and return this
    rank's rows [B, H, L_r, d] of the sum: one reduce-scatter over pieces
    padded to the longest window (each rank receives only its own rows)."""
    world = len(splits) - 1
    lens = [splits[r + 1] - splits[r] for r in range(world)]
    Lmax = max(lens)
    staged = _host_staged(group, full)
    src = full.cpu() if staged else full
    shape = list(full.shape)
    shape[2] = Lmax
    pieces = []
    for r in range(world):
        p = src.new_zeros(shape)
        p.narrow(2, 0, lens[r]).copy_(src.narrow(2, splits[r], lens[r]))
        pieces.append(p)
    out = src.new_empty(shape)
    dist.reduce_scatter(out, pieces, group=group)
    out = out.narrow(2, 0, lens[rank]).contiguous()
    return out.to(full.device) if staged else out


def gather_bounds(local_bounds, splits, group=None):
    """The pages' allgather of the column intervals: each rank holds the four
    bound arrays [B, Hm, L_r] of its columns; returns the whole [B, Hm, N]."""
    return [_gather_dim(b, splits, 2, group) for b in local_bounds]


def gather_rows(local: torch.Tensor, splits, group=None) -> torch.Tensor:
    """[B, H, L_r, d] shards -> [B, H, N, d]."""
    return _gather_dim(local, splits, 2, group)


class LibraryLocal:
    """The rank's computation on its GPU through the C ABI (row windows)."""

    def __init__(self, flags: int = 0):
        from . import fm
        self.fm = fm
        self.flags = flags

    def _plan(self, bounds, q_row0, Nq):
        fm = self.fm
        lts, lte, uts, ute = bounds
        B, Hm, N = lts.shape
        bnd = fm.make_bounds(lts, lte, uts, ute)
        plan = torch.empty(fm.fm_plan_bytes_rows(B, Hm, N, q_row0, Nq), dtype=torch.uint8, device=lts.device)
        status = torch.zeros(1, dtype=torch.int32, device=lts.device)
        fm.fm_tile_classify_rows(bnd, q_row0, Nq, plan, status)
        return bnd, plan, status

    def prepare(self, bounds, q_row0, Nq):
        """Classify the row window once (device work on the current stream);
        the result serves the forward and the backward of the step."""
        return self._plan(bounds, q_row0, Nq)

    def forward(self, q, k, v, bounds, q_row0, scale, prep=None):
        fm = self.fm
        Nq = q.shape[2]
        bnd, plan, status = prep if prep is not None else self._plan(bounds, q_row0, Nq)
        o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
        fm.fm_attn_fwd_rows(q, k, v, bnd, plan, q_row0, scale, o, lse, status, flags=self.flags)
        self._check(status)
        return o, lse

    def backward(self, q, k, v, o, lse, dO, bounds, q_row0, scale, prep=None):
        fm = self.fm
        B, H, Nq, d = q.shape
        bnd, plan, status = prep if prep is not None else self._plan(bounds, q_row0, Nq)
        dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
        dv = torch.empty(k.shape, dtype=torch.float32, device=q.device)
        ws = torch.empty(fm.fm_bwd_workspace_bytes(B, H, Nq, d), dtype=torch.uint8, device=q.device)
        fm.fm_attn_bwd_rows(q, k, v, o, lse, dO, bnd, plan, q_row0, scale, dq, dk, dv, ws, status,
                            flags=self.flags)
        self._check(status)
        return dq, dk, dv

    def _check(self, status):
        code = int(status.item())
        if code != 0:
            raise self.fm.FmError(code, "device")


def step(q, k, v, dO, local_bounds, splits, rank, scale, local, group=None):
    """One forward + backward of the rank's rows.  q, k, v, dO: the rank's
    rows [B, H, L_r, d]; local_bounds: the bounds of its columns [B, Hm, L_r].
    Returns O, lse, dQ, dK, dV of the rank's rows."""
    bounds = gather_bounds(local_bounds, splits, group)
    # K and V move while the row window is classified (a computation with a
    # ``prepare`` step does it once for the forward and the backward).
    k_done = _gather_dim_start(k, splits, 2, group)
    v_done = _gather_dim_start(v, splits, 2, group)
    q_row0 = splits[rank]
    prep = local.prepare(bounds, q_row0, q.shape[2]) if hasattr(local, "prepare") else None
    k_full, v_full = k_done(), v_done()
    extra = {} if prep is None else {"prep": prep}
    o, lse = local.forward(q, k_full, v_full, bounds, q_row0, scale, **extra)
    dq, dk_part, dv_part = local.backward(q, k_full, v_full, o, lse, dO, bounds, q_row0, scale, **extra)
    dk = reduce_scatter_rows(dk_part, splits, rank, group)
    dv = reduce_scatter_rows(dv_part, splits, rank, group)
    return o, lse, dq, dk, dv
