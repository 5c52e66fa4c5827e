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


def _bucket(n):
    """Length bucket of a work list: half-octaves, longest first, empty lists last."""
    n = np.asarray(n, np.int64)
    lg = np.where(n > 0, np.floor(np.log2(np.maximum(n, 1))), 0).astype(np.int64)
    half = np.where(lg > 0, (n >> np.maximum(lg - 1, 0)) & 1, 0)
    return np.where(n > 0, 62 - (2 * lg + half), 63)


def test_bucket_rule_is_monotone():
    n = np.arange(0, 1 << 16)
    b = _bucket(n)
    assert b[0] == 63 and b[1] == 62 and b[2] == 60 and b[3] == 59 and b[256] == 46
    assert np.all(np.diff(b[1:]) <= 0)


def _group_weights(lab):
    """Per KV tile of one (b, hm) segment (rows of `lab` = KV tiles, columns =
    Q tiles): the longest non-skip list among the KV tiles whose lists end at
    the same Q tile; 0 for an empty list."""
    nz = lab != oracle.SKIP
    cnt = nz.sum(axis=1)
    key = np.where(cnt > 0, nz.shape[1] - 1 - np.argmax(nz[:, ::-1], axis=1), -1)
    w = np.zeros_like(cnt)
    for k in np.unique(key[key >= 0]):
        sel = key == k
        w[sel] = cnt[sel].max()
    return w


@pytest.mark.parametrize("name", ["causal_ragged", "docs_small", "window_sink_small", "random_cols_small",
                                  "random_cols_d64", "all_masked_small", "long_packing_128k",
                                  "sliding_window_sink"])
def test_work_order_longest_first_and_stable(fm, name):
    """The plan's two work orders (read at the offsets its header records) are
    the stable sorts, longest bucket first, of the oracle's labels: per
    (b, hm, Q tile) for the forward by the tile's own non-skip count, and per
    (b, hm, KV tile) for the backward by the longest count of its group (the
    KV tiles whose Q lists end at the same tile); entries s * n_tiles + tile;
    the bucket starts delimit the buckets."""
    wl = W.SMALL.get(name) or W.FULL[name]
    m = W.make_mask(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    torch.cuda.synchronize()
    att.check_status()
    plan = att.plan.cpu().numpy()
    hdr = plan[:128]
    n_q, n_k = (int(x) for x in hdr[24:32].view(np.int32))
    off_row, off_col, off_rb, off_cb = (int(x) for x in hdr[40:72].view(np.int64))
    ref = oracle.tile_labels_all(m, 128, 128)                  # [B, Hm, n_q, n_k]
    S = wl.B * wl.Hm
    wrow = (ref != oracle.SKIP).sum(axis=3).reshape(S * n_q)
    wcol = np.concatenate([_group_weights(ref[b, hm].T) for b in range(wl.B) for hm in range(wl.Hm)])
    for wts, off, offb, n_t in ((wrow, off_row, off_rb, n_q), (wcol, off_col, off_cb, n_k)):
        bkt = _bucket(wts)
        got = plan[off:off + 4 * S * n_t].view(np.int32)
        assert np.array_equal(got, np.argsort(bkt, kind="stable"))
        starts = plan[offb:offb + 4 * 65].view(np.int32)
        assert np.array_equal(starts, np.concatenate([[0], np.cumsum(np.bincount(bkt, minlength=64))]))
