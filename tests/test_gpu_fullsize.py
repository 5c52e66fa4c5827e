"""The five workloads at full size, in the launch configuration the benchmark
times (fp32 outputs, plan from the classifier, same kernels): outputs are
compared with the oracle on sampled rows (O, lse, dQ) and sampled columns
(dK, dV) of the first and last heads; every output element is checked for NaN."""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_all, run_fm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


def _attend_counts(lts, lte, uts, ute, N):
    """Rows attending each column, from interval arithmetic on the bounds."""
    l0, l1 = lts.astype(np.int64), lte.astype(np.int64)
    u0, u1 = uts.astype(np.int64), ute.astype(np.int64)
    ln = np.maximum(l1 - l0, 0)
    un = np.maximum(u1 - u0, 0)
    inter = np.maximum(np.minimum(l1, u1) - np.maximum(l0, u0), 0)
    inter = np.where((ln > 0) & (un > 0), inter, 0)
    return N - (ln + un - inter)


def _pick(rng, eligible, k):
    eligible = np.asarray(eligible)
    if eligible.size <= k:
        return np.sort(eligible)
    return np.sort(eligible[np.linspace(0, eligible.size - 1, k).astype(int)])


@pytest.mark.parametrize("name", list(W.FULL))
def test_full_size_sampled_against_oracle(fm, name):
    wl = W.FULL[name]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    out = run_fm(fm, wl, m, q, k, v, dO)
    for key in ("o", "dq", "dk", "dv", "lse"):
        assert not torch.isnan(out[key]).any(), key
    rng = np.random.default_rng(123)
    N = wl.N
    for b, h in sorted({(0, 0), (wl.B - 1, wl.H - 1)}):
        hm = h if wl.Hm == wl.H else 0
        msl = {key: m[key][b:b + 1, hm:hm + 1] for key in ("lts", "lte", "uts", "ute")}
        sl = [t[b:b + 1, h:h + 1] for t in (q, k, v, dO)]
        rows = set(rng.choice(N, 40, replace=False).tolist()) | {0, N - 1, N // 2}
        if m["docs"] is not None:
            starts = np.cumsum([0] + m["docs"][b][:-1])
            rows |= set(starts[:6].tolist()) | set((starts[1:6] - 1).tolist())
        rows = np.array(sorted(rows), np.int64)
        cnt = _attend_counts(*[x[0, 0] for x in msl.values()], N)
        cols = _pick(rng, np.nonzero((cnt > 0) & (cnt <= 256))[0], 12)
        cols = np.union1d(cols, _pick(rng, np.nonzero(cnt == 0)[0], 3)).astype(np.int64)
        O, L = oracle.forward(*sl[:3], msl, wl.scale, rows=rows)
        g = oracle.backward(*sl, msl, wl.scale, rows=rows, cols=cols)
        items = [(f"O[{b},{h}]", out["o"][b, h, rows].cpu().numpy(), O[0, 0]),
                 ("lse", out["lse"][b, h, rows].cpu().numpy(), L[0, 0]),
                 (f"dQ[{b},{h}]", out["dq"][b, h, rows].cpu().numpy(), g["dq"][0, 0])]
        if cols.size:
            items += [(f"dK[{b},{h}]", out["dk"][b, h, cols].cpu().numpy(), g["dk"][0, 0]),
                      (f"dV[{b},{h}]", out["dv"][b, h, cols].cpu().numpy(), g["dv"][0, 0])]
        check_all(items)
