"""The C ABI library loads, exports every entry point of include/fm.h, and its
host-side logic (sizes, status strings, the row-to-column converter) is right.
No GPU is used: the converter is host code."""
import os
import re

import numpy as np
import pytest

import oracle
from long_context_fm_gb300 import build as fmbuild
from long_context_fm_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fm():
    fmbuild.build()
    from long_context_fm_gb300 import fm as mod
    return mod


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fm_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(fm):
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(fm._lib, n), n
    assert sorted(fm.EXPORTED) == names


def test_abi_version_and_status_strings(fm):
    assert fm.fm_abi_version() == 6
    for code in range(10):
        assert fm.fm_status_string(code) and "unknown" not in fm.fm_status_string(code)
    assert "unknown" in fm.fm_status_string(99)


def test_plan_bytes(fm):
    assert fm.fm_plan_bytes(1, 1, 256) > 0
    assert fm.fm_plan_bytes(1, 1, 256, 96, 128) == 0
    assert fm.fm_plan_bytes(0, 1, 256) == 0
    big = fm.fm_plan_bytes(1, 1, 131072)
    n = 1024
    assert big >= n * n * (1 + 4 + 4) and big < n * n * 10 + (1 << 20)
    assert fm.fm_bwd_workspace_bytes(1, 8, 131072, 128) >= 8 * 131072 * 128 * 4 + 8 * 131072 * 4
    assert fm.fm_bwd_workspace_bytes(1, 1, 10, 96) == 0


def _cols(m, b, hm):
    return [m[k][b, hm] for k in ("lts", "lte", "uts", "ute")]


@pytest.mark.parametrize("name", [n for n in list(W.SMALL) + ["tiny_causal", "doc_packing",
                                                             "sliding_window", "prefix_lm",
                                                             "long_packing_128k"]])
def test_converter_reproduces_generator_bounds(fm, name):
    wl = W.SMALL.get(name) or W.FULL[name]
    m = W.make_mask(wl)
    if m["rows"] is None:
        pytest.skip("no row form")
    lts, lte, uts, ute = fm.fm_mask_from_rows(*m["rows"])
    # the generator writes the same canonical form: bit-exact
    assert np.array_equal(lts, m["lts"]) and np.array_equal(lte, m["lte"])
    assert np.array_equal(uts, m["uts"]) and np.array_equal(ute, m["ute"])


def test_converter_golden_examples(fm):
    import json
    gd = json.load(open(os.path.join(ROOT, "tests", "golden", "causal_row_form.json")))
    cs = np.array(gd["col_start"], np.int32)[None, None]
    ce = np.array(gd["col_end"], np.int32)[None, None]
    got = fm.fm_mask_from_rows(cs, ce)
    for arr, key in zip(got, ("lts", "lte", "uts", "ute")):
        assert arr[0, 0].tolist() == gd["expect_columns"][key]
    gd = json.load(open(os.path.join(ROOT, "tests", "golden", "doc_packing_example.json")))["small"]
    got = fm.fm_mask_from_rows(np.array(gd["col_start"], np.int32)[None, None],
                               np.array(gd["col_end"], np.int32)[None, None])
    for arr, key in zip(got, ("lts", "lte", "uts", "ute")):
        assert arr[0, 0].tolist() == gd["expect_columns"][key]


def _masked_runs_per_column(M):
    """Number of maximal masked row runs in each column of a dense mask."""
    Mi = M.astype(np.int8)
    starts = (Mi[0] == 1).astype(int) + ((Mi[1:] == 1) & (Mi[:-1] == 0)).sum(0)
    return starts


@pytest.mark.parametrize("seed", range(12))
def test_converter_random_rows_against_dense_masks(fm, seed):
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 90))
    mode = seed % 3
    if mode == 0:       # arbitrary intervals: often unrepresentable
        a = rng.integers(0, N, size=N); b = rng.integers(0, N, size=N)
        cs, ce = np.minimum(a, b), np.maximum(a, b)
    elif mode == 1:     # monotone-ish (sliding structures): usually representable
        cs = np.sort(rng.integers(0, N, size=N)); ce = np.maximum(cs, np.sort(rng.integers(0, N, size=N)))
    else:               # with empty rows and full rows
        cs = rng.integers(0, N, size=N); ce = cs + rng.integers(-3, N, size=N)
        ce = np.minimum(ce, N - 1)
    cs = cs.astype(np.int32); ce = ce.astype(np.int32)
    Mr = oracle.dense_from_rows(cs, ce)
    representable = bool((_masked_runs_per_column(Mr) <= 2).all())
    try:
        got = fm.fm_mask_from_rows(cs[None, None], ce[None, None])
    except fm.FmError as e:
        assert e.code == fm.FM_ERR_UNREPRESENTABLE and not representable
        return
    assert representable
    Mc = oracle.dense_from_cols(*[g[0, 0] for g in got])
    assert np.array_equal(Mr, Mc)
    lts, lte, uts, ute = (g[0, 0] for g in got)
    assert np.all((lts < lte) | ((lts == N) & (lte == N)))      # canonical empty lower
    assert np.all((uts < ute) | ((uts == 0) & (ute == 0)))      # canonical empty upper


def test_converter_counts_representable_cases(fm):
    """Across many random masks both outcomes occur and always agree with brute force."""
    rng = np.random.default_rng(77)
    seen = {True: 0, False: 0}
    for _ in range(200):
        N = int(rng.integers(1, 40))
        cs = rng.integers(0, N, size=N).astype(np.int32)
        ce = (cs + rng.integers(-2, 12, size=N)).clip(max=N - 1).astype(np.int32)
        Mr = oracle.dense_from_rows(cs, ce)
        rep = bool((_masked_runs_per_column(Mr) <= 2).all())
        try:
            got = fm.fm_mask_from_rows(cs[None, None], ce[None, None])
            assert rep
            assert np.array_equal(Mr, oracle.dense_from_cols(*[g[0, 0] for g in got]))
        except fm.FmError as e:
            assert e.code == fm.FM_ERR_UNREPRESENTABLE and not rep
        seen[rep] += 1
    assert seen[True] > 20 and seen[False] > 20


def test_converter_rejects_bad_rows(fm):
    cs = np.array([[[0, 0, 5]]], np.int32)
    ce = np.array([[[0, 1, 7]]], np.int32)            # ce = 7 >= N = 3
    with pytest.raises(fm.FmError) as e:
        fm.fm_mask_from_rows(cs, ce)
    assert e.value.code == fm.FM_ERR_BAD_BOUNDS
    cs = np.array([[[-1, 0, 0]]], np.int32)
    ce = np.array([[[0, 1, 2]]], np.int32)
    with pytest.raises(fm.FmError) as e:
        fm.fm_mask_from_rows(cs, ce)
    assert e.value.code == fm.FM_ERR_BAD_BOUNDS
    # empty rows (cs > ce) are fine anywhere
    out = fm.fm_mask_from_rows(np.array([[[2, 0, 0]]], np.int32), np.array([[[1, 0, 2]]], np.int32))
    assert out[0].shape == (1, 1, 3)


def test_converter_batches_and_heads(fm):
    wl = W.SMALL["docs_small"].with_(Hm=1)
    m = W.make_mask(wl)
    cs, ce = m["rows"]
    cs2 = np.concatenate([cs, cs[:, :, ::-1] * 0], axis=1)      # second head: causal (cs = 0)
    ce2 = np.concatenate([ce, np.broadcast_to(np.arange(wl.N, dtype=np.int32), ce.shape)], axis=1)
    got = fm.fm_mask_from_rows(cs2, ce2)
    assert np.array_equal(got[0][:, :1], m["lts"]) and np.array_equal(got[3][:, :1], m["ute"])
    assert np.all(got[3][:, 1] == np.arange(wl.N)) and np.all(got[0][:, 1] == wl.N)


# ---- several intervals per row (blog "FlashMask技术" §6.1 item 1) -------------
@pytest.mark.parametrize("name", [n for n in list(W.SMALL) + ["tiny_causal", "doc_packing",
                                                             "sliding_window", "prefix_lm",
                                                             "sliding_window_sink"]])
def test_interval_converter_reproduces_generator_bounds(fm, name):
    wl = W.SMALL.get(name) or W.FULL[name]
    m = W.make_mask(wl)
    if m["row_intervals"] is None:
        pytest.skip("no row form")
    got = fm.fm_mask_from_row_intervals(*m["row_intervals"])
    for arr, key in zip(got, ("lts", "lte", "uts", "ute")):
        assert np.array_equal(arr, m[key]), key
    if m["rows"] is not None:                         # K = 1: same as the one-interval entry
        ref = fm.fm_mask_from_rows(*m["rows"])
        assert all(np.array_equal(a, b) for a, b in zip(got, ref))


def test_interval_converter_golden_example(fm):
    import json
    gd = json.load(open(os.path.join(ROOT, "tests", "golden", "multi_interval_example.json")))
    N = gd["N"]
    starts = np.ones((N, 2), np.int32)
    ends = np.zeros((N, 2), np.int32)
    for r, ivs in gd["rows"].items():
        for k, (a, b) in enumerate(ivs):
            starts[int(r), k], ends[int(r), k] = a, b
    got = fm.fm_mask_from_row_intervals(starts[None, None], ends[None, None])
    for j, want in gd["expect_columns"].items():
        assert [int(g[0, 0, int(j)]) for g in got] == want, j
    # slots in the other order, and a third slot that overlaps the first
    s2 = np.concatenate([starts[:, ::-1], starts[:, :1]], axis=1)
    e2 = np.concatenate([ends[:, ::-1], ends[:, :1]], axis=1)
    got2 = fm.fm_mask_from_row_intervals(s2[None, None], e2[None, None])
    assert all(np.array_equal(a, b) for a, b in zip(got, got2))


def _row_runs(M):
    """Attended runs of each row of a dense mask as inclusive (start, end) slots,
    padded with unused (1, 0) slots to the largest count."""
    N = M.shape[0]
    runs = []
    for i in range(N):
        a = np.concatenate([[0], (~M[i]).astype(np.int8), [0]])
        d = np.diff(a)
        runs.append(list(zip(np.flatnonzero(d == 1), np.flatnonzero(d == -1) - 1)))
    K = max(1, max(len(r) for r in runs))
    s = np.ones((N, K), np.int32)
    e = np.zeros((N, K), np.int32)
    for i, r in enumerate(runs):
        for k, (a, b) in enumerate(r):
            s[i, k], e[i, k] = a, b
    return s, e


@pytest.mark.parametrize("seed", range(6))
def test_interval_converter_round_trips_column_masks(fm, seed):
    """Any two-range column mask has a row form with several intervals per row;
    converting that back gives the same dense mask in canonical form."""
    wl = W.SMALL["random_cols_small"]
    m = W.make_mask(wl, seed)
    for b in range(wl.B):
        for hm in range(wl.Hm):
            Mc = oracle.dense_from_cols(*_cols(m, b, hm))
            s, e = _row_runs(Mc)
            assert s.shape[1] > 1
            got = fm.fm_mask_from_row_intervals(s[None, None], e[None, None])
            assert np.array_equal(oracle.dense_from_cols(*[g[0, 0] for g in got]), Mc)
            lts, lte, uts, ute = (g[0, 0] for g in got)
            N = wl.N
            assert np.all((lts < lte) | ((lts == N) & (lte == N)))
            assert np.all((uts < ute) | ((uts == 0) & (ute == 0)))


@pytest.mark.parametrize("seed", range(12))
def test_interval_converter_random_rows_against_dense_masks(fm, seed):
    rng = np.random.default_rng(2000 + seed)
    N = int(rng.integers(1, 80))
    K = int(rng.integers(1, 5))
    mode = seed % 3
    if mode == 0:       # arbitrary, overlapping, unsorted: often unrepresentable
        a = rng.integers(0, N, size=(N, K)); b = rng.integers(0, N, size=(N, K))
        s, e = np.minimum(a, b), np.maximum(a, b)
    elif mode == 1:     # a sliding structure per slot: usually representable
        base = np.sort(rng.integers(0, N, size=(N, K)), axis=0)
        s = base
        e = np.minimum(N - 1, base + rng.integers(0, 6, size=(1, K)))
    else:               # with unused slots
        s = rng.integers(0, N, size=(N, K)); e = s + rng.integers(-4, 8, size=(N, K))
        e = np.minimum(e, N - 1)
    s = s.astype(np.int32); e = e.astype(np.int32)
    Mr = oracle.dense_from_row_intervals(s, e)
    representable = bool((_masked_runs_per_column(Mr) <= 2).all())
    try:
        got = fm.fm_mask_from_row_intervals(s[None, None], e[None, None])
    except fm.FmError as err:
        assert err.code == fm.FM_ERR_UNREPRESENTABLE and not representable
        return
    assert representable
    assert np.array_equal(Mr, oracle.dense_from_cols(*[g[0, 0] for g in got]))


def test_interval_converter_rejects_bad_input(fm):
    s = np.array([[[[0, 2], [1, 5]]]], np.int32)      # [1, 1, 2, 2]: slot (5, ...) too far
    e = np.array([[[[0, 1], [1, 5]]]], np.int32)
    with pytest.raises(fm.FmError) as err:
        fm.fm_mask_from_row_intervals(s, e)
    assert err.value.code == fm.FM_ERR_BAD_BOUNDS
    s = np.array([[[[0, -1], [1, 3]]]], np.int32)
    e = np.array([[[[0, 0], [1, 2]]]], np.int32)      # (-1, 0) used with a negative start
    with pytest.raises(fm.FmError) as err:
        fm.fm_mask_from_row_intervals(s, e)
    assert err.value.code == fm.FM_ERR_BAD_BOUNDS
    z = np.zeros(4, np.int32)
    p = z.ctypes.data
    assert fm._lib.fm_mask_from_row_intervals(p, p, 0, 1, 1, 2, p, p, p, p) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_mask_from_row_intervals(None, p, 1, 1, 1, 2, p, p, p, p) == fm.FM_ERR_INVALID_ARG


def test_wait_test_hook_argument_checks(fm):
    """The test hook rejects unknown kernels and out-of-range bounds; -1 clears it."""
    assert fm._lib.fm_debug_wait_test(2, 1_000_000) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_debug_wait_test(0, 10) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_debug_wait_test(1, 10**12) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_debug_wait_test(-1, 0) == fm.FM_OK


def test_step_graph_null_arguments(fm):
    """Argument checks that need no GPU: no graph handle or no arguments."""
    import ctypes
    h = ctypes.c_void_p(1234)
    assert fm._lib.fm_step_graph_create(None, ctypes.byref(h)) == fm.FM_ERR_INVALID_ARG
    assert h.value is None                                   # cleared on failure
    assert fm._lib.fm_step_graph_create(ctypes.byref(fm.StepArgs()), None) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_step_graph_launch(None, None) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_step_graph_destroy(None) == fm.FM_ERR_INVALID_ARG
    assert ctypes.sizeof(fm.StepArgs) == 200                 # the C layout on LP64


def test_binding_fails_loudly_without_the_library():
    """No CPU fallback: importing the binding without libfm.so raises, naming the build step."""
    import subprocess
    import sys
    code = ("import os; real = os.path.exists; "
            "os.path.exists = lambda p: False if str(p).endswith('libfm.so') else real(p); "
            "import long_context_fm_gb300.fm")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "build" in r.stderr


def test_noalloc_shape_errors_match_the_workspace_backward(fm):
    """The allocation-free backward reports a bad shape with the same code as
    fm_attn_bwd (both return before any CUDA call, so no GPU is needed)."""
    import ctypes
    cases = [(70000, 1, 256, 128), (1, 70000, 256, 128), (1, 1, 256, 96), (0, 1, 256, 128), (1, 1, -5, 64)]
    for B, H, N, d in cases:
        bounds = fm.Bounds(None, None, None, None, B, 1, N)
        args = (None, None, None, None, 0, None, None, bounds, None, B, H, N, d, ctypes.c_float(0.1),
                None, None, None, 1, 0)
        want = fm._lib.fm_attn_bwd(*args, None, 0, None, None)
        got = fm._lib.fm_attn_bwd_noalloc(*args, None, None)
        assert got == want != fm.FM_OK, (B, H, N, d, got, want)
