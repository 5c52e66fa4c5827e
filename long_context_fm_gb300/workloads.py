"""Seeded synthetic workloads for masked attention.

This module only draws numbers: tensor values, document lengths and the
column-bound arrays that a workload's mask description spells out.  It holds
none of the attention arithmetic, none of the tile logic and none of the
row-to-column conversion; the CUDA library, its tests and the oracle all take
their inputs from here.

Mask encoding (FlashMask, "column-wise sparse" representation, arXiv
2410.01359 abstract): per key column j two masked row ranges, lower
``[lts_j, lte_j)`` and upper ``[uts_j, ute_j)``, half-open.  An empty range is
written in canonical form: lower ``(N, N)``, upper ``(0, 0)``.

The row form of the blog post "FlashMask技术" (§2.1 causal example, §3.3
document-packing example) is an inclusive attend interval
``[col_start_i, col_end_i]`` per query row.  Workloads whose mask has such a
form also return it, so the host converter can be checked against it.  The
multi-interval form (same blog, §6.1 item 1) gives each row K inclusive
intervals; the window with sink tokens of the §5 streaming example (row i
attends the first ``sink`` keys and the last ``window`` keys up to i) needs
K = 2.

Value recipe: fp32 N(0, 1) from ``torch.Generator`` seeded with ``seed`` in
the order Q, K, V, dO, multiplied by ``input_scale`` and rounded to bf16
(round-to-nearest-even).  Document lengths come from one
``numpy.random.default_rng(seed)`` stream, batches in order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    mask: str                 # causal | docs_uniform | docs_lognormal | window | window_sink | prefix
                              # | prefix_random | random_cols | full | none_attended
    Hm: int = 1               # mask heads: 1 (shared) or H (per head)
    input_scale: float = 1.0
    params: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "Workload":
        f = dict(name=self.name, B=self.B, H=self.H, N=self.N, d=self.d, mask=self.mask,
                 Hm=self.Hm, input_scale=self.input_scale, params=dict(self.params))
        f.update(kw)
        return Workload(**f)


# The five workloads of the pages' SFT / packing / window / 128K settings.
FULL = {
    "tiny_causal": Workload("tiny_causal", B=1, H=2, N=256, d=64, mask="causal"),
    "doc_packing": Workload("doc_packing", B=2, H=8, N=8192, d=128, mask="docs_uniform",
                            params=dict(lo=128, hi=2048)),
    "sliding_window": Workload("sliding_window", B=1, H=16, N=32768, d=128, mask="window",
                               params=dict(window=1024)),
    "prefix_lm": Workload("prefix_lm", B=1, H=16, N=16384, d=128, mask="prefix",
                          input_scale=2.0, params=dict(prefix=4096)),
    "prefix_random": Workload("prefix_random", B=1, H=16, N=16384, d=128, mask="prefix_random",
                              input_scale=2.0, params=dict(prefix=4096)),
    "long_packing_128k": Workload("long_packing_128k", B=1, H=8, N=131072, d=128,
                                  mask="docs_lognormal",
                                  params=dict(median=4096, sigma=1.0, lo=256, hi=32768)),
    # The streaming-inference window (1024 keys) with 10 sink tokens, at the
    # sliding-window workload's sizes.
    "sliding_window_sink": Workload("sliding_window_sink", B=1, H=16, N=32768, d=128,
                                    mask="window_sink", params=dict(window=1024, sink=10)),
}

# Small cases the oracle finishes in seconds: several tiles and a ragged tail.
SMALL = {
    "causal_ragged": Workload("causal_ragged", B=1, H=2, N=300, d=64, mask="causal"),
    "docs_small": Workload("docs_small", B=2, H=2, N=1000, d=128, mask="docs_uniform",
                           params=dict(lo=16, hi=300)),
    "window_small": Workload("window_small", B=1, H=2, N=777, d=128, mask="window",
                             params=dict(window=100)),
    "prefix_small": Workload("prefix_small", B=1, H=2, N=640, d=128, mask="prefix",
                             input_scale=2.0, params=dict(prefix=200)),
    "prefix_random_small": Workload("prefix_random_small", B=1, H=2, N=520, d=128,
                                    mask="prefix_random", input_scale=2.0,
                                    params=dict(prefix=130)),
    "random_cols_small": Workload("random_cols_small", B=2, H=2, Hm=2, N=384, d=128,
                                  mask="random_cols"),
    "random_cols_d64": Workload("random_cols_d64", B=1, H=3, Hm=3, N=450, d=64,
                                mask="random_cols"),
    "lognormal_small": Workload("lognormal_small", B=1, H=2, N=2048, d=128,
                                mask="docs_lognormal",
                                params=dict(median=200, sigma=1.0, lo=20, hi=900)),
    "window_sink_small": Workload("window_sink_small", B=1, H=2, N=777, d=128, mask="window_sink",
                                 params=dict(window=100, sink=10)),
    "window_sink_d64": Workload("window_sink_d64", B=1, H=3, N=650, d=64, mask="window_sink",
                                params=dict(window=200, sink=150)),
    "unmasked_small": Workload("unmasked_small", B=1, H=2, N=256, d=128, mask="full"),
    "all_masked_small": Workload("all_masked_small", B=1, H=1, N=200, d=64, mask="none_attended"),
}


# ---------------------------------------------------------------------------
# document lengths
# ---------------------------------------------------------------------------
def _pack(lengths_iter, N):
    out, total = [], 0
    while total < N:
        L = int(next(lengths_iter))
        L = min(L, N - total)           # the last document is truncated
        out.append(L)
        total += L
    return out


def doc_lengths(wl: Workload, seed: int = 0):
    """Per-batch document lengths, one rng stream, batches in order."""
    rng = np.random.default_rng(seed)
    p = wl.params
    if wl.mask == "docs_uniform":
        def gen():
            while True:
                yield rng.integers(p["lo"], p["hi"], endpoint=True)
    elif wl.mask == "docs_lognormal":
        mu = math.log(p["median"])

        def gen():
            while True:
                z = rng.standard_normal()
                yield int(np.clip(np.rint(math.exp(mu + p["sigma"] * z)), p["lo"], p["hi"]))
    else:
        raise ValueError(wl.mask)
    g = gen()
    return [_pack(g, wl.N) for _ in range(wl.B)]


# ---------------------------------------------------------------------------
# masks
# ---------------------------------------------------------------------------
def _empty_bounds(N):
    lts = np.full(N, N, np.int32)
    lte = np.full(N, N, np.int32)
    uts = np.zeros(N, np.int32)
    ute = np.zeros(N, np.int32)
    return lts, lte, uts, ute


def _one_mask(wl: Workload, b: int, hm: int, docs, rng):
    """Column bounds, the one-interval row form when the mask has one, and
    the K-interval row form ``(starts, ends)`` [N, K] when only that exists,
    of one (batch, mask head)."""
    N = wl.N
    j = np.arange(N, dtype=np.int64)
    lts, lte, uts, ute = _empty_bounds(N)
    cs = ce = None
    multi = None
    if wl.mask == "causal":
        ute[:] = j                                          # rows i < j masked
        cs = np.zeros(N, np.int32)
        ce = j.astype(np.int32)
    elif wl.mask in ("docs_uniform", "docs_lognormal"):
        cs = np.empty(N, np.int32)
        ce = j.astype(np.int32)
        off = 0
        for L in docs[b]:
            end = off + L
            ute[off:end] = j[off:end]                       # rows above the diagonal
            lts[off:end] = end                              # rows of later documents
            lte[off:end] = N
            cs[off:end] = off
            off = end
        empty = lts >= lte
        lts[empty] = N
        lte[empty] = N
    elif wl.mask == "window":
        W = wl.params["window"]
        ute[:] = j
        lo = np.minimum(j + W, N)
        lts[:] = lo
        lte[:] = N
        empty = lts >= lte
        lts[empty] = N
        cs = np.maximum(0, j - (W - 1)).astype(np.int32)
        ce = j.astype(np.int32)
    elif wl.mask == "window_sink":
        W, S = wl.params["window"], wl.params["sink"]
        ute[:] = j                                          # causal: rows i < j
        lo = np.minimum(j + W, N)                           # past the window ...
        lts[:] = np.where(j < S, N, lo)                     # ... except sink columns
        lte[:] = N
        empty = lts >= lte
        lts[empty] = N
        starts = np.stack([np.zeros(N, np.int64), np.maximum(0, j - (W - 1))], axis=1)
        ends = np.stack([np.minimum(S - 1, j), j], axis=1)
        multi = (starts.astype(np.int32), ends.astype(np.int32))
    elif wl.mask in ("prefix", "prefix_random"):
        P = wl.params["prefix"]
        ute[P:] = j[P:]
        if wl.mask == "prefix":
            cs = np.zeros(N, np.int32)
            ce = np.where(j < P, P - 1, j).astype(np.int32)
        else:
            draw = rng.integers(j, N, endpoint=True)        # lts_j uniform in [j, N]
            lts[:] = draw
            lte[:] = N
            empty = lts >= lte
            lts[empty] = N
    elif wl.mask == "random_cols":
        # Two arbitrary ranges per column: empty, overlapping, in either order,
        # whole-column and single-row ranges all occur.
        a = rng.integers(0, N, endpoint=True, size=(4, N))
        kind = rng.integers(0, 8, size=(2, N))
        s0, e0 = np.minimum(a[0], a[1]), np.maximum(a[0], a[1])
        s1, e1 = np.minimum(a[2], a[3]), np.maximum(a[2], a[3])
        s0 = np.where(kind[0] == 0, N, s0); e0 = np.where(kind[0] == 0, N, e0)     # empty
        s0 = np.where(kind[0] == 1, 0, s0); e0 = np.where(kind[0] == 1, N, e0)     # whole column
        s0, e0 = np.where(kind[0] == 2, e0, s0), np.where(kind[0] == 2, s0, e0)  # start > end: empty
        s1 = np.where(kind[1] == 0, 0, s1); e1 = np.where(kind[1] == 0, 0, e1)     # empty
        e1 = np.where(kind[1] == 2, np.minimum(s1 + 1, N), e1)                     # one row
        s1 = np.where(kind[1] == 3, e1, s1)                                        # start == end
        lts[:], lte[:], uts[:], ute[:] = s0, e0, s1, e1
    elif wl.mask == "full":
        cs = np.zeros(N, np.int32)
        ce = np.full(N, N - 1, np.int32)
    elif wl.mask == "none_attended":
        uts[:] = 0
        ute[:] = N
        cs = np.ones(N, np.int32)                           # cs > ce: empty row
        ce = np.zeros(N, np.int32)
    else:
        raise ValueError(wl.mask)
    if cs is not None:
        multi = (cs[:, None], ce[:, None])
    return (lts, lte, uts, ute), (None if cs is None else (cs, ce)), multi


def make_mask(wl: Workload, seed: int = 0):
    """Column bounds ``lts, lte, uts, ute`` as int32 ``[B, Hm, N]``, the row
    form ``rows = (cs, ce)`` as int32 ``[B, Hm, N]`` or ``None``, and the
    K-interval row form ``row_intervals = (starts, ends)`` as int32
    ``[B, Hm, N, K]`` or ``None`` (K = 1 wherever ``rows`` exists)."""
    docs = doc_lengths(wl, seed) if wl.mask.startswith("docs") else None
    rng = np.random.default_rng(seed)
    cols = np.empty((4, wl.B, wl.Hm, wl.N), np.int32)
    rows = np.empty((2, wl.B, wl.Hm, wl.N), np.int32)
    multi = None
    has_rows = has_multi = True
    for b in range(wl.B):
        for hm in range(wl.Hm):
            c, r, mi = _one_mask(wl, b, hm, docs, rng)
            cols[:, b, hm] = np.stack(c)
            if r is None:
                has_rows = False
            else:
                rows[:, b, hm] = np.stack(r)
            if mi is None:
                has_multi = False
            else:
                if multi is None:
                    multi = np.empty((2, wl.B, wl.Hm) + mi[0].shape, np.int32)
                multi[:, b, hm] = np.stack(mi)
    return dict(lts=cols[0], lte=cols[1], uts=cols[2], ute=cols[3],
                rows=(rows[0], rows[1]) if has_rows else None,
                row_intervals=(multi[0], multi[1]) if has_multi else None, docs=docs)


def make_inputs(wl: Workload, seed: int = 0, device="cpu", need_do: bool = True):
    """bf16 Q, K, V, dO of shape ``[B, H, N, d]``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (wl.B, wl.H, wl.N, wl.d)
    out = []
    for _ in range(4 if need_do else 3):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if wl.input_scale != 1.0:
            t.mul_(wl.input_scale)
        out.append(t.to(torch.bfloat16))
    return tuple(out)
