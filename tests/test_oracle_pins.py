"""Pins for the oracle: checks against things other than the oracle itself.

- brute force in torch fp64 (dense mask, softmax, autograd) on tiny inputs;
- central finite differences of the oracle's own forward for the gradients;
- invariants the method's definition fixes (constant V, a single attended key,
  fully masked rows, D = dO.O, invariance of O and dQ under a shift of every key);
- closed forms: attended-pair counts and the tile counts of causal masks
  ("about half of the GEMMs skipped", blog "FlashMask技术" §1 item 2 and §2.2);
- the pages' worked examples (blog §2.1 causal row form, §3.3 document packing,
  §6.1 multi-interval rows) stored under tests/golden/.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _mask_np(wl, seed=0):
    return W.make_mask(wl, seed)


def _bounds(m, b=0, hm=0):
    return [m[k][b, hm] for k in ("lts", "lte", "uts", "ute")]


def _rand_mask(N, rng, Hm=1, B=1):
    """Arbitrary column bounds: empty, reversed, overlapping and whole-column ranges."""
    a = rng.integers(0, N + 1, size=(4, B, Hm, N)).astype(np.int32)
    return dict(lts=a[0], lte=a[1], uts=a[2], ute=a[3])


def _torch_reference(q, k, v, dO, M, scale):
    """Masked attention by the textbook formula, fp64, gradients by autograd."""
    q = q.clone().requires_grad_(True)
    k = k.clone().requires_grad_(True)
    v = v.clone().requires_grad_(True)
    s = scale * q @ k.transpose(-1, -2)
    dead = M.all(dim=-1, keepdim=True)                 # rows with nothing attended
    s = s.masked_fill(M, float("-inf")).masked_fill(dead, 0.0)
    p = torch.softmax(s, dim=-1).masked_fill(dead, 0.0)
    o = p @ v
    lse = torch.logsumexp(s, dim=-1).masked_fill(dead.squeeze(-1), float("-inf"))
    o.backward(dO)
    return o.detach(), lse.detach(), q.grad, k.grad, v.grad


@pytest.mark.parametrize("seed,N,d", [(0, 40, 16), (1, 64, 32), (2, 17, 8), (3, 50, 16)])
def test_oracle_matches_torch_bruteforce(seed, N, d):
    rng = np.random.default_rng(seed)
    m = _rand_mask(N, rng)
    if seed == 3:                      # causal plus a block of fully masked rows
        m = dict(lts=np.full((1, 1, N), 10, np.int32), lte=np.full((1, 1, N), 14, np.int32),
                 uts=np.zeros((1, 1, N), np.int32), ute=np.arange(N, dtype=np.int32)[None, None])
    g = torch.Generator().manual_seed(seed)
    q, k, v, dO = (torch.randn(1, 1, N, d, generator=g, dtype=torch.float64).to(torch.bfloat16)
                   for _ in range(4))
    scale = 1.0 / np.sqrt(d)
    M = torch.from_numpy(oracle.dense_from_cols(*_bounds(m)))
    ro, rl, rdq, rdk, rdv = _torch_reference(*(t[0, 0].double() for t in (q, k, v, dO)), M, scale)
    O, lse = oracle.forward(q, k, v, m, scale)
    gr = oracle.backward(q, k, v, dO, m, scale)
    np.testing.assert_allclose(O[0, 0], ro.numpy(), atol=1e-12, rtol=1e-10)
    fin = np.isfinite(rl.numpy())
    assert np.array_equal(fin, np.isfinite(lse[0, 0]))
    np.testing.assert_allclose(lse[0, 0][fin], rl.numpy()[fin], atol=1e-12, rtol=1e-10)
    assert np.all(lse[0, 0][~fin] == -np.inf)
    for ours, ref in ((gr["dq"], rdq), (gr["dk"], rdk), (gr["dv"], rdv)):
        np.testing.assert_allclose(ours[0, 0], ref.numpy(), atol=1e-11, rtol=1e-9)
    np.testing.assert_allclose(gr["lse"][0, 0][fin], rl.numpy()[fin], atol=1e-12)
    if seed == 3:
        assert (~fin).sum() == 4         # rows 10..13 see nothing


def test_oracle_gradients_by_finite_differences():
    """Central differences of L = sum(O * dO) through the oracle's forward."""
    rng = np.random.default_rng(7)
    N, d = 24, 8
    m = _rand_mask(N, rng)
    g = torch.Generator().manual_seed(7)
    q, k, v, dO = (torch.randn(1, 1, N, d, generator=g).to(torch.bfloat16).float() for _ in range(4))
    scale = 0.35
    gr = oracle.backward(q, k, v, dO, m, scale)
    h = 2.0 ** -12                     # exact in fp32 next to bf16 values

    def loss(qq, kk, vv):
        O, _ = oracle.forward(qq, kk, vv, m, scale)
        return float((O[0, 0] * dO[0, 0].double().numpy()).sum())

    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        for _ in range(8):
            r, c = int(rng.integers(N)), int(rng.integers(d))
            ins = [q.clone(), k.clone(), v.clone()]
            ins[idx][0, 0, r, c] += h
            lp = loss(*ins)
            ins[idx][0, 0, r, c] -= 2 * h
            lm = loss(*ins)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - gr[name][0, 0, r, c]) < 2e-5 * max(1.0, abs(fd)), (name, r, c)


def test_invariants_constant_v_single_key_dead_rows():
    N, d = 96, 16
    # rows 0..9 see only column 5, rows 10..19 see nothing, the rest see a causal window.
    lts = np.full(N, N, np.int32); lte = np.full(N, N, np.int32)
    uts = np.zeros(N, np.int32); ute = np.arange(N, dtype=np.int32)
    uts[:] = 0
    ute[:] = np.maximum(np.arange(N), 20)          # rows < max(j, 20) masked ...
    ute[5] = 0; lts[5] = 10; lte[5] = 20           # ... except column 5: rows 0..9 attend it
    ute[N - 1] = N                                 # the last column is attended by nobody
    m = dict(lts=lts[None, None], lte=lte[None, None], uts=uts[None, None], ute=ute[None, None])
    M = oracle.dense_from_cols(lts, lte, uts, ute)
    assert M[:10].sum(1).tolist() == [N - 1] * 10 and M[10:20].all()
    g = torch.Generator().manual_seed(3)
    q, k, dO = (torch.randn(1, 1, N, d, generator=g).to(torch.bfloat16) for _ in range(3))
    vrow = torch.randn(d, generator=g).to(torch.bfloat16)
    v = vrow.expand(1, 1, N, d).contiguous()
    O, lse = oracle.forward(q, k, v, m, 0.25)
    live = ~M.all(1)
    np.testing.assert_allclose(O[0, 0][live], np.broadcast_to(vrow.double().numpy(), (live.sum(), d)),
                               atol=1e-13)                          # constant V returns V
    assert np.all(O[0, 0][~live] == 0) and np.all(lse[0, 0][~live] == -np.inf)
    v2 = torch.randn(1, 1, N, d, generator=g).to(torch.bfloat16)
    O2, lse2 = oracle.forward(q, k, v2, m, 0.25)
    np.testing.assert_allclose(O2[0, 0][:10], np.broadcast_to(v2[0, 0, 5].double().numpy(), (10, d)),
                               atol=1e-13)                          # single key returns its row
    s5 = 0.25 * (q[0, 0, :10].double() @ k[0, 0, 5].double()).numpy()
    np.testing.assert_allclose(lse2[0, 0][:10], s5, atol=1e-13)     # lse = that key's score
    gr = oracle.backward(q, k, v2, dO, m, 0.25)
    assert np.all(gr["dq"][0, 0][~live] == 0)
    never = M.all(0)                                                 # columns nobody attends
    assert never.any()
    assert np.all(gr["dk"][0, 0][never] == 0) and np.all(gr["dv"][0, 0][never] == 0)
    # D_i = dO_i . O_i
    np.testing.assert_allclose(gr["D"][0, 0], (O2[0, 0] * dO[0, 0].double().numpy()).sum(1), atol=1e-12)


def test_key_shift_invariance():
    """Adding c to every key leaves P, O and dQ unchanged (sum_j dS_ij = 0) and
    moves lse_i by scale * q_i . c."""
    rng = np.random.default_rng(11)
    N, d = 48, 16
    m = _rand_mask(N, rng)
    g = torch.Generator().manual_seed(11)
    q, k, v, dO = (torch.randn(1, 1, N, d, generator=g).to(torch.bfloat16) for _ in range(4))
    c = torch.full((d,), 0.5)
    k2 = k.float() + c                 # fp32 input: the shift is exact for bf16 keys
    assert torch.equal(k2 - c, k.float())
    scale = 0.3
    O, lse = oracle.forward(q, k, v, m, scale)
    O2, lse2 = oracle.forward(q, k2, v, m, scale)
    gr, gr2 = oracle.backward(q, k, v, dO, m, scale), oracle.backward(q, k2, v, dO, m, scale)
    np.testing.assert_allclose(O2, O, atol=1e-12)
    np.testing.assert_allclose(gr2["dq"], gr["dq"], atol=1e-11)
    fin = np.isfinite(lse)
    shift = scale * (q[0, 0].double() @ c.double()).numpy()
    np.testing.assert_allclose((lse2 - lse)[fin], np.broadcast_to(shift, lse.shape)[fin], atol=1e-11)


def test_row_and_column_forms_give_the_same_dense_mask():
    for wl in list(W.SMALL.values()) + [W.FULL["tiny_causal"], W.FULL["doc_packing"].with_(B=1)]:
        m = _mask_np(wl)
        if m["rows"] is None:
            continue
        for b in range(wl.B):
            for hm in range(wl.Hm):
                Mr = oracle.dense_from_rows(m["rows"][0][b, hm], m["rows"][1][b, hm])
                Mc = oracle.dense_from_cols(*_bounds(m, b, hm))
                assert np.array_equal(Mr, Mc), (wl.name, b, hm)


def _multi_from_golden(gd):
    N = gd["N"]
    K = max(len(v) for v in gd["rows"].values())
    starts = np.ones((N, K), np.int32)          # unused slots: start > end
    ends = np.zeros((N, K), np.int32)
    for r, ivs in gd["rows"].items():
        for k, (a, b) in enumerate(ivs):
            starts[int(r), k], ends[int(r), k] = a, b
    return starts, ends


def test_golden_multi_interval_example():
    """Blog §6.1 item 1: the printed two-row example, hand-derived counts and columns."""
    gd = json.load(open(os.path.join(GOLDEN, "multi_interval_example.json")))
    N = gd["N"]
    starts, ends = _multi_from_golden(gd)
    M = oracle.dense_from_row_intervals(starts, ends)
    for r, n in gd["attended_per_row"].items():
        assert int((~M[int(r)]).sum()) == n
    assert int((~M).sum()) == gd["attended_pairs"]
    assert np.array_equal(np.flatnonzero(~M[0]), np.r_[0:101, 200:301])
    # the hand-written column spot values describe the same mask
    for j, (a, b, c, d) in gd["expect_columns"].items():
        col = np.zeros(N, bool)
        col[a:b] = True
        col[c:d] = True
        assert np.array_equal(M[:, int(j)], col), j


def test_multi_interval_reduces_to_one_interval_rows():
    """K = 1 is the one-interval row rule; extra unused slots change nothing."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        N = int(rng.integers(1, 60))
        cs = rng.integers(0, N, size=N).astype(np.int32)
        ce = (cs + rng.integers(-3, N, size=N)).clip(max=N - 1).astype(np.int32)
        Mr = oracle.dense_from_rows(cs, ce)
        assert np.array_equal(oracle.dense_from_row_intervals(cs[:, None], ce[:, None]), Mr)
        pad_s = np.concatenate([cs[:, None], np.full((N, 2), 7, np.int32)], axis=1)
        pad_e = np.concatenate([ce[:, None], np.full((N, 2), 3, np.int32)], axis=1)
        assert np.array_equal(oracle.dense_from_row_intervals(pad_s, pad_e), Mr)


def test_multi_interval_union_invariants():
    """The attended set is the union of the slots: slot order does not matter, an
    interval split into two touching pieces or covered by an overlapping one
    changes nothing, and counts equal the size of the union."""
    rng = np.random.default_rng(6)
    for _ in range(20):
        N = int(rng.integers(2, 50))
        K = int(rng.integers(1, 5))
        a = rng.integers(0, N, size=(N, K)); b = rng.integers(0, N, size=(N, K))
        s, e = np.minimum(a, b).astype(np.int32), np.maximum(a, b).astype(np.int32)
        M = oracle.dense_from_row_intervals(s, e)
        perm = rng.permutation(K)
        assert np.array_equal(oracle.dense_from_row_intervals(s[:, perm], e[:, perm]), M)
        mid = (s[:, :1] + e[:, :1]) // 2                                  # slot 0 -> [s, mid], [mid + 1, e]
        s2 = np.concatenate([s, mid + 1], axis=1).astype(np.int32)
        e2 = np.concatenate([mid, e[:, 1:], e[:, :1]], axis=1).astype(np.int32)
        assert np.array_equal(oracle.dense_from_row_intervals(s2, e2), M)
        s3 = np.concatenate([s, s[:, :1]], axis=1).astype(np.int32)      # slot 0 repeated
        e3 = np.concatenate([e, e[:, :1]], axis=1).astype(np.int32)
        assert np.array_equal(oracle.dense_from_row_intervals(s3, e3), M)
        for i in range(N):
            want = set()
            for k in range(K):
                want |= set(range(s[i, k], e[i, k] + 1))
            assert int((~M[i]).sum()) == len(want)


def test_window_sink_row_and_column_forms_agree():
    for name in ("window_sink_small", "window_sink_d64"):
        wl = W.SMALL[name]
        m = _mask_np(wl)
        assert m["rows"] is None and m["row_intervals"][0].shape == (1, 1, wl.N, 2)
        Mi = oracle.dense_from_row_intervals(m["row_intervals"][0][0, 0], m["row_intervals"][1][0, 0])
        assert np.array_equal(Mi, oracle.dense_from_cols(*_bounds(m)))


@pytest.mark.parametrize("name", ["window_sink_small", "window_sink_d64", "sliding_window_sink"])
def test_window_sink_attended_pairs_closed_form(name):
    """Row i attends min(i + 1, W) window keys plus the sink keys left of its
    window: max(0, min(S, i - W + 1))."""
    wl = W.SMALL.get(name) or W.FULL[name]
    Wn, S, N = wl.params["window"], wl.params["sink"], wl.N
    i = np.arange(N, dtype=np.int64)
    want = int((np.minimum(i + 1, Wn) + np.maximum(0, np.minimum(S, i - Wn + 1))).sum())
    if name == "sliding_window_sink":
        assert want == 33030656 + 10 * (N - 1033) + 45
    m = _mask_np(wl)
    assert oracle.attended_pairs(*_bounds(m)) == want


def _counts(lbl):
    return dict(skip=int((lbl == 0).sum()), full=int((lbl == 1).sum()), partial=int((lbl == 2).sum()))


def test_golden_causal_example():
    gd = json.load(open(os.path.join(GOLDEN, "causal_row_form.json")))
    N = gd["N"]
    Mr = oracle.dense_from_rows(gd["col_start"], gd["col_end"])
    e = gd["expect_columns"]
    Mc = oracle.dense_from_cols(e["lts"], e["lte"], e["uts"], e["ute"])
    assert np.array_equal(Mr, Mc) and Mr.shape == (N, N)
    for tc in gd["tile_counts"]:
        wl = W.Workload("c", 1, 1, tc["N"], 64, "causal")
        m = _mask_np(wl)
        got = _counts(oracle.tile_labels(*_bounds(m), tc["bq"], tc["bk"]))
        assert got == {k: tc[k] for k in ("skip", "full", "partial")}, tc
        if tc["N"] <= 4096:
            exact = _counts(oracle.tile_labels(*_bounds(m), tc["bq"], tc["bk"], exact=True))
            assert exact == got
    wl = W.Workload("c", 1, 1, gd["attended_pairs"]["N"], 64, "causal")
    assert oracle.attended_pairs(*_bounds(_mask_np(wl))) == gd["attended_pairs"]["pairs"]


def test_golden_doc_packing_example():
    gd = json.load(open(os.path.join(GOLDEN, "doc_packing_example.json")))
    N = gd["N"]
    # The page's construction: rows of a document at offset o get (o, o + i).
    cs, ce, off = [], [], 0
    for L in gd["doc_lengths"]:
        for i in range(L):
            cs.append(off); ce.append(off + i)
        off += L
    assert off == N
    for row, a, b in gd["row_spot_checks"]:
        assert (cs[row], ce[row]) == (a, b)
    # Independent column form: the generator's document-packing bounds.
    wl = W.Workload("docs", 1, 1, N, 128, "docs_uniform")
    docs = [gd["doc_lengths"]]
    cols = W._one_mask(wl, 0, 0, docs, None)[0]
    Mr = oracle.dense_from_rows(cs, ce)
    assert np.array_equal(Mr, oracle.dense_from_cols(*cols))
    assert int((~Mr).sum()) == gd["attended_pairs"] == oracle.attended_pairs(*cols)
    lbl = oracle.tile_labels(*cols, 128, 128)
    assert _counts(lbl) == {k: gd["tile_counts_128"][k] for k in ("skip", "full", "partial")}
    assert np.array_equal(lbl, oracle.tile_labels(*cols, 128, 128, exact=True))
    sm = gd["small"]
    e = sm["expect_columns"]
    assert np.array_equal(oracle.dense_from_rows(sm["col_start"], sm["col_end"]),
                          oracle.dense_from_cols(e["lts"], e["lte"], e["uts"], e["ute"]))


@pytest.mark.parametrize("name,pairs", [
    ("tiny_causal", 32896),
    ("sliding_window", 33030656),        # sum_i min(i + 1, 1024)
    ("prefix_lm", 142612480),            # 4096^2 + sum_{i=4096}^{16383} (i + 1)
])
def test_attended_pairs_closed_form(name, pairs):
    wl = W.FULL[name]
    m = _mask_np(wl)
    assert oracle.attended_pairs(*_bounds(m)) == pairs
    N = wl.N
    if name == "sliding_window":
        assert pairs == sum(min(i + 1, 1024) for i in range(N))
    if name == "prefix_lm":
        assert pairs == 4096 ** 2 + sum(i + 1 for i in range(4096, N))


def test_attended_pairs_docs_closed_form():
    for wl in (W.FULL["doc_packing"], W.SMALL["docs_small"], W.SMALL["lognormal_small"]):
        m = _mask_np(wl)
        for b in range(wl.B):
            want = sum(L * (L + 1) // 2 for L in m["docs"][b])
            assert oracle.attended_pairs(*_bounds(m, b)) == want
            assert sum(m["docs"][b]) == wl.N


@pytest.mark.parametrize("name", ["tiny_causal", "doc_packing", "sliding_window", "prefix_lm",
                                  "causal_ragged", "docs_small", "window_small", "prefix_small",
                                  "lognormal_small", "unmasked_small", "all_masked_small",
                                  "window_sink_small", "window_sink_d64", "sliding_window_sink"])
@pytest.mark.parametrize("bq,bk", [(128, 128), (64, 128), (64, 64), (128, 64)])
def test_labels_equal_exact_on_structured_masks(name, bq, bk):
    wl = W.FULL.get(name) or W.SMALL[name]
    m = _mask_np(wl)
    for b in range(wl.B):
        lbl = oracle.tile_labels(*_bounds(m, b), bq, bk)
        ex = oracle.tile_labels(*_bounds(m, b), bq, bk, exact=True)
        assert np.array_equal(lbl, ex), (name, b)


@pytest.mark.parametrize("seed", range(6))
def test_labels_sound_on_arbitrary_bounds(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(1, 700))
    m = _rand_mask(N, rng)
    for bq, bk in ((128, 128), (64, 128), (64, 64)):
        lbl = oracle.tile_labels(*_bounds(m), bq, bk)
        ex = oracle.tile_labels(*_bounds(m), bq, bk, exact=True)
        assert np.all(ex[lbl == 0] == 0)          # SKIP only where all is masked
        assert np.all(ex[lbl == 1] == 1)          # FULL only where nothing is masked
        assert np.all(lbl[ex == 0] != 1) and np.all(lbl[ex == 1] != 0)


def test_labels_sound_on_prefix_random():
    wl = W.FULL["prefix_random"]
    m = _mask_np(wl)
    lbl = oracle.tile_labels(*_bounds(m))
    ex = oracle.tile_labels(*_bounds(m), exact=True)
    assert np.all(ex[lbl == 0] == 0) and np.all(ex[lbl == 1] == 1)
    assert (lbl == 2).sum() > (lbl == 1).sum()    # the stress case is mostly partial tiles


def test_softmax_max_subtraction_identity():
    """FlashAttention article §二.2: subtracting the row max leaves softmax unchanged;
    the oracle's stabilised lse equals the naive log-sum-exp where that is finite."""
    rng = np.random.default_rng(5)
    N, d = 32, 8
    m = dict(lts=np.full((1, 1, N), N, np.int32), lte=np.full((1, 1, N), N, np.int32),
             uts=np.zeros((1, 1, N), np.int32), ute=np.arange(N, dtype=np.int32)[None, None])
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(1, 1, N, d, generator=g).to(torch.bfloat16) for _ in range(3))
    _, lse = oracle.forward(q, k, v, m, 0.5)
    s = 0.5 * (q[0, 0].double() @ k[0, 0].double().T).numpy()
    naive = np.log(np.array([np.exp(s[i, : i + 1]).sum() for i in range(N)]))
    np.testing.assert_allclose(lse[0, 0], naive, rtol=1e-13)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("which", ["lower", "upper"])
def test_labels_sound_with_one_random_range_per_column(seed, which):
    """Only one of the two ranges used, with random starts and ends: the rule
    must still never call a tile SKIP or FULL wrongly, and it must find some
    SKIP and FULL tiles (narrow random ranges leave whole tiles untouched)."""
    rng = np.random.default_rng(500 + seed)
    N = 700
    a = rng.integers(0, N + 1, size=N)
    w = rng.integers(0, 200, size=N)
    s0 = np.sort(a).astype(np.int32)                    # starts grow with the column
    e0 = np.minimum(s0 + w, N).astype(np.int32)
    empty_lo = (np.full(N, N, np.int32), np.full(N, N, np.int32))
    empty_up = (np.zeros(N, np.int32), np.zeros(N, np.int32))
    b = (s0, e0) + empty_up if which == "lower" else empty_lo + (s0, e0)
    for bq, bk in ((64, 64), (128, 128), (64, 128)):
        lbl = oracle.tile_labels(*b, bq, bk)
        ex = oracle.tile_labels(*b, bq, bk, exact=True)
        assert np.all(ex[lbl == 0] == 0) and np.all(ex[lbl == 1] == 1)
        assert (lbl == 1).any()


# ---- e4m3 (FP8 forward) --------------------------------------------------------
def test_e4m3_codes_of_the_format_definition():
    """Codes fixed by the format: sign | 4-bit exponent (bias 7) | 3-bit mantissa,
    subnormals in steps of 2^-9, largest finite 448, ties to even, saturation."""
    cases = [(1.0, 0x38), (2.0, 0x40), (0.5, 0x30), (1.125, 0x39), (448.0, 0x7E), (-448.0, 0xFE),
             (500.0, 0x7E), (1e9, 0x7E), (-1e9, 0xFE), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01),
             (7 * 2.0 ** -9, 0x07), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (1.0625, 0x38),
             (1.1875, 0x3A), (240.0, 0x77), (256.0, 0x78), (0.0, 0x00), (-0.0, 0x80)]
    for x, c in cases:
        assert int(oracle.e4m3_encode(np.array([x]))[0]) == c, x
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0) and pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_encode_matches_exhaustive_nearest_search():
    """Nearest grid value by brute force over the 127 non-negative codes, ties to
    the even code (an even mantissa), saturating at 448."""
    rng = np.random.default_rng(8)
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[1:] + grid[:-1]) / 2
    x = np.concatenate([np.exp2(rng.uniform(-12, 9.5, 4000)), mids, grid, [470.0, 455.0]])
    x = np.concatenate([x, -x[:500]])
    got = oracle.e4m3_encode(x)
    a = np.minimum(np.abs(x), 448.0)
    dist = np.abs(a[:, None] - grid[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist <= best                                   # one or two nearest codes
    code = np.array([np.flatnonzero(row)[0] if row.sum() == 1 else
                     [c for c in np.flatnonzero(row) if c % 2 == 0][0] for row in cand])
    want = (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
    assert np.array_equal(got, want)


def test_quantize_e4m3_scale_and_reduction_to_the_exact_path():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 2, 40, 16)).astype(np.float32)
    codes, ds = oracle.quantize_e4m3(x)
    assert ds == np.float32(np.abs(x).max() / np.float32(448.0))
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert codes[i] & 0x7F == 0x7E                        # the largest magnitude maps to +-448
    assert np.abs(oracle.e4m3_decode(codes) * ds - x).max() <= np.abs(x).max() / 448 * 16   # half a top-binade step
    # values already on the e4m3 grid with amax 448 are kept exactly (descale 1), so
    # the FP8 path reduces to the plain one
    g = oracle.e4m3_decode(rng.integers(0, 0x7F, size=(1, 2, 40, 16)).astype(np.uint8))
    g *= np.where(rng.random(g.shape) < 0.5, -1.0, 1.0)
    g.flat[0] = 448.0
    q8, dq = oracle.quantize_e4m3(g)
    assert dq == 1.0 and np.array_equal(oracle.e4m3_decode(q8), g)
    k8, dk = oracle.quantize_e4m3(g[:, :, ::-1].copy())
    vt8, dv = oracle.quantize_e4m3(g, transpose=True)
    assert vt8.shape == (1, 2, 16, 40)
    wl = W.Workload("c", 1, 1, 40, 16, "causal")
    m = _mask_np(wl)
    O8, L8 = oracle.forward_fp8(q8, k8, vt8, (dq, dk, dv), m, 0.1)
    O, L = oracle.forward(g.astype(np.float32), g[:, :, ::-1].astype(np.float32), g.astype(np.float32), m, 0.1)
    np.testing.assert_allclose(O8, O, rtol=0, atol=0)
    np.testing.assert_allclose(L8, L, rtol=0, atol=0)
