"""Compressed column bounds expanded on the GPU: fm_bounds_decompress gives
the original int32 bounds bit for bit (and so the same tile labels and
attention), and a buffer that does not match the call is refused with
FM_ERR_INVALID_ARG without reading beyond it."""
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


def _expand(fm, c, B, Hm, N, status):
    arr = [torch.full((B, Hm, N), -7, dtype=torch.int32, device="cuda") for _ in range(4)]
    bnd = fm.make_bounds(*arr)
    fm.fm_bounds_decompress(torch.from_numpy(c).cuda(), bnd, status)
    torch.cuda.synchronize()
    return arr


@pytest.mark.parametrize("name", ["causal_ragged", "docs_small", "random_cols_small", "window_sink_small",
                                  "prefix_random", "long_packing_128k", "sliding_window_sink"])
def test_device_expansion_is_exact(fm, name):
    wl = W.SMALL.get(name) or W.FULL[name]
    m = W.make_mask(wl)
    c = fm.fm_bounds_compress(m["lts"], m["lte"], m["uts"], m["ute"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B, Hm, N = m["lts"].shape
    arr = _expand(fm, c, B, Hm, N, status)
    assert int(status.item()) == 0
    for t, key in zip(arr, ("lts", "lte", "uts", "ute")):
        assert np.array_equal(t.cpu().numpy(), m[key]), key


def test_attention_on_expanded_bounds_matches_the_oracle(fm):
    wl = W.SMALL["docs_small"]
    m = W.make_mask(wl)
    c = fm.fm_bounds_compress(m["lts"], m["lte"], m["uts"], m["ute"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    arr = _expand(fm, c, *m["lts"].shape, status)
    assert int(status.item()) == 0
    me = dict(m)
    me.update({k: t.cpu().numpy() for k, t in zip(("lts", "lte", "uts", "ute"), arr)})
    q, k, v, dO = W.make_inputs(wl)
    out = run_fm(fm, wl, me, q, k, v, dO)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    check_all([("O", out["o"].cpu().numpy(), O), ("lse", out["lse"].cpu().numpy(), L),
               ("dQ", out["dq"].cpu().numpy(), g["dq"]), ("dK", out["dk"].cpu().numpy(), g["dk"]),
               ("dV", out["dv"].cpu().numpy(), g["dv"])])


def test_mismatched_buffers_are_refused(fm):
    m = W.make_mask(W.SMALL["causal_ragged"])
    c = fm.fm_bounds_compress(m["lts"], m["lte"], m["uts"], m["ute"])
    B, Hm, N = m["lts"].shape
    for mutate, shape in ((lambda b: b.__setitem__(0, b[0] ^ 1), (B, Hm, N)),          # magic
                          (lambda b: None, (B, Hm, N + 1)),                              # shape of the call
                          (lambda b: b[32:36].view(np.uint32).__setitem__(0, 0xFFFFFFF0), (B, Hm, N))):  # entry
        bad = c.copy()
        mutate(bad)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        _expand(fm, bad, *shape, status)
        assert int(status.item()) == fm.FM_ERR_INVALID_ARG
