"""Long backward lists against the oracle, in the standard precision mode the
benchmark times.

The backward walks, for every 128-column key tile, the list of Q tiles that
attend it; the longest lists dominate the long-context workloads.  These
tests compare dK and dV on key tiles whose lists run to 100-256 Q tiles:

* one long causal document (N = 16384): key tile 0 walks all 128 Q tiles;
  every element of O, lse, dQ, dK, dV is compared with the oracle;
* at full size, the columns with the most attending rows: the first columns
  of the longest document of the 128K packing workload (a list of ~126 Q
  tiles), column 0 of the sliding window with sink tokens (every one of the
  256 Q tiles attends it) and column 0 of the prefix-LM workload (all 128 Q
  tiles), on the first and last heads.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_all, mode_for, run_fm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


def test_long_causal_document_every_element(fm):
    wl = W.Workload("causal_16k", B=1, H=1, N=16384, d=128, mask="causal")
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl, seed=11)
    out = run_fm(fm, wl, m, q, k, v, dO, flags=0)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    check_all([("O", out["o"].cpu().numpy(), O), ("lse", out["lse"].cpu().numpy(), L),
               ("dQ", out["dq"].cpu().numpy(), g["dq"]), ("dK", out["dk"].cpu().numpy(), g["dk"]),
               ("dV", out["dv"].cpu().numpy(), g["dv"])])
    # key tile 0 is the one with the 128-entry list: checked on its own too
    check_all([("dK tile 0", out["dk"][0, 0, :128].cpu().numpy(), g["dk"][0, 0, :128]),
               ("dV tile 0", out["dv"][0, 0, :128].cpu().numpy(), g["dv"][0, 0, :128])])


def _attend_counts(m, b, hm, N):
    l0, l1, u0, u1 = (m[x][b, hm].astype(np.int64) for x in ("lts", "lte", "uts", "ute"))
    ln, un = np.maximum(l1 - l0, 0), np.maximum(u1 - u0, 0)
    inter = np.where((ln > 0) & (un > 0), np.maximum(np.minimum(l1, u1) - np.maximum(l0, u0), 0), 0)
    return N - (ln + un - inter)


@pytest.mark.parametrize("name", ["long_packing_128k", "sliding_window_sink", "prefix_lm"])
def test_full_size_longest_columns(fm, name):
    wl = W.FULL[name]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    out = run_fm(fm, wl, m, q, k, v, dO, flags=mode_for(wl))
    N = wl.N
    for b, h in sorted({(0, 0), (wl.B - 1, wl.H - 1)}):
        hm = h if wl.Hm == wl.H else 0
        cnt = _attend_counts(m, b, hm, N)
        j0 = int(np.argmax(cnt))
        assert cnt[j0] >= 10000, (name, cnt[j0])
        # the column with the most attending rows, the rest of its key tile's
        # edges and a column further into the same run of long columns
        cand = {j0, j0 + 1, j0 + 9, (j0 // 128) * 128, (j0 // 128) * 128 + 127, j0 + 64, j0 + 200}
        cols = np.array(sorted(c for c in cand if 0 <= c < N and cnt[c] >= cnt[j0] // 2), np.int64)
        msl = {x: m[x][b:b + 1, hm:hm + 1] for x in ("lts", "lte", "uts", "ute")}
        sl = [t[b:b + 1, h:h + 1] for t in (q, k, v, dO)]
        g = oracle.backward(*sl, msl, wl.scale, rows=np.array([0], np.int64), cols=cols)
        print(name, (b, h), "columns", cols.tolist(), "attending rows", cnt[cols].tolist())
        check_all([(f"dK[{b},{h}] long columns", out["dk"][b, h, cols].cpu().numpy(), g["dk"][0, 0]),
                   (f"dV[{b},{h}] long columns", out["dv"][b, h, cols].cpu().numpy(), g["dv"][0, 0])])
