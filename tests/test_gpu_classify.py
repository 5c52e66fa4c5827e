"""Tile classification on the GPU: labels bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


CASES = list(W.SMALL) + list(W.FULL)


@pytest.mark.parametrize("name", CASES)
@pytest.mark.parametrize("bq,bk", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_labels_bit_exact(fm, name, bq, bk):
    wl = W.SMALL.get(name) or W.FULL[name]
    if name == "long_packing_128k" and (bq, bk) != (128, 128):
        pytest.skip("128K labels checked at the contract tile size")
    m = W.make_mask(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    got = att.labels(bq, bk).cpu().numpy()
    torch.cuda.synchronize()
    att.check_status()
    ref = oracle.tile_labels_all(m, bq, bk)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref), f"{(got != ref).sum()} labels differ"


def test_causal_128k_skips_about_half(fm):
    wl = W.Workload("c", 1, 1, 131072, 128, "causal")
    m = W.make_mask(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    lbl = att.labels().cpu().numpy()
    n = 1024
    assert (lbl == 0).sum() == n * (n - 1) // 2 and (lbl == 1).sum() == n * (n - 1) // 2
    assert (lbl == 2).sum() == n


def test_bad_bounds_reported_on_device(fm):
    wl = W.SMALL["causal_ragged"]
    m = W.make_mask(wl)
    m["ute"] = m["ute"].copy()
    m["ute"][0, 0, 7] = wl.N + 1
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    torch.cuda.synchronize()
    assert int(att.status.item()) == fm.FM_ERR_BAD_BOUNDS


def test_host_argument_errors(fm):
    wl = W.SMALL["causal_ragged"]
    m = W.make_mask(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_tile_classify(att.bounds, small, att.status)
    assert e.value.code == fm.FM_ERR_WORKSPACE
    with pytest.raises(fm.FmError) as e:
        fm.fm_tile_classify(att.bounds, att.plan, att.status, bq=96)
    assert e.value.code == fm.FM_ERR_INVALID_ARG
