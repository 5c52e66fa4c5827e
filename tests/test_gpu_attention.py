"""Forward and backward on the GPU against the oracle, element by element, on
sizes that span several tiles and a ragged tail; invariants; failure paths."""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_all, check_close, check_lse, run_fm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


@pytest.mark.parametrize("mode", ["standard", "precise"])
@pytest.mark.parametrize("name", list(W.SMALL))
def test_fwd_bwd_match_oracle(fm, name, mode):
    wl = W.SMALL[name]
    if mode == "standard" and wl.input_scale != 1.0:
        pytest.skip("x2-scaled inputs run in precise mode (bf16 P/dS operands exceed the max-abs bound)")
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    out = run_fm(fm, wl, m, q, k, v, dO, flags=1 if mode == "precise" else 0)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    check_all([("O", out["o"].cpu().numpy(), O), ("lse", out["lse"].cpu().numpy(), L),
               ("dQ", out["dq"].cpu().numpy(), g["dq"]), ("dK", out["dk"].cpu().numpy(), g["dk"]),
               ("dV", out["dv"].cpu().numpy(), g["dv"])])


@pytest.mark.parametrize("name", ["docs_small", "random_cols_d64", "causal_ragged"])
def test_bf16_outputs(fm, name):
    """bf16 outputs: the same values up to one bf16 rounding of each output."""
    wl = W.SMALL[name]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    out = run_fm(fm, wl, m, q, k, v, dO, o_dtype=torch.bfloat16, g_dtype=torch.bfloat16)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    check_close("O", out["o"].float().cpu().numpy(), O)
    check_lse(out["lse"].cpu().numpy(), L)
    for key in ("dq", "dk", "dv"):
        check_close(key, out[key].float().cpu().numpy(), g[key])


def test_full_ragged_multi_tile_causal_d128(fm):
    wl = W.Workload("causal_1000", B=2, H=3, N=1000, d=128, mask="causal")
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl, seed=4)
    out = run_fm(fm, wl, m, q, k, v, dO)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    check_close("O", out["o"].cpu().numpy(), O)
    check_lse(out["lse"].cpu().numpy(), L)
    for key in ("dq", "dk", "dv"):
        check_close(key, out[key].cpu().numpy(), g[key])


def test_single_row_and_tiny_n(fm):
    for N in (1, 7, 64, 129):
        wl = W.Workload(f"c{N}", B=1, H=1, N=N, d=64, mask="causal")
        m = W.make_mask(wl)
        q, k, v, dO = W.make_inputs(wl, seed=N)
        out = run_fm(fm, wl, m, q, k, v, dO)
        O, L = oracle.forward(q, k, v, m, wl.scale)
        g = oracle.backward(q, k, v, dO, m, wl.scale)
        check_close("O", out["o"].cpu().numpy(), O)
        check_lse(out["lse"].cpu().numpy(), L)
        for key in ("dq", "dk", "dv"):
            check_close(key, out[key].cpu().numpy(), g[key])


@pytest.mark.parametrize("precise", [False, True])
def test_constant_v_and_dead_rows(fm, precise):
    """Constant V returns V on every row that attends something; rows that
    attend nothing return O = 0 and lse = -inf; columns nobody attends get
    dK = dV = 0.  O = sum_j p^_j v / sum_j p_j: the product applies the bf16
    weights p^_j = p_j (1 + e_j), |e_j| <= 2^-9, so standard mode returns V
    within 2^-9 relative; precise mode (p^ = hi + lo) within ~2^-17."""
    N, d = 300, 128
    lts = np.full(N, N, np.int32); lte = np.full(N, N, np.int32)
    uts = np.zeros(N, np.int32); ute = np.maximum(np.arange(N), 150).astype(np.int32)
    ute[20:40] = 0; lts[20:40] = 100; lte[20:40] = 150      # rows < 100 see columns 20..39 only
    ute[-5:] = N                                            # last five columns: nobody
    m = {k: x[None, None] for k, x in zip(("lts", "lte", "uts", "ute"), (lts, lte, uts, ute))}
    wl = W.Workload("inv", B=1, H=2, N=N, d=d, mask="causal")
    g = torch.Generator().manual_seed(9)
    q, k, dO = (torch.randn(1, 2, N, d, generator=g).to(torch.bfloat16) for _ in range(3))
    vrow = torch.randn(d, generator=g).to(torch.bfloat16)
    v = vrow.expand(1, 2, N, d).contiguous()
    out = run_fm(fm, wl, m, q, k, v, dO, flags=fm.FM_FLAG_PRECISE if precise else 0)
    M = oracle.dense_from_cols(lts, lte, uts, ute)
    live = ~M.all(1)
    o = out["o"].cpu().numpy()[0]
    assert (~live).sum() == 50                               # rows 100..149 see nothing
    want = np.broadcast_to(vrow.float().numpy(), (2, live.sum(), d))
    np.testing.assert_allclose(o[:, live], want, rtol=(1e-5 if precise else 2.0 ** -9), atol=1e-6)
    assert np.all(o[:, ~live] == 0)
    assert np.all(out["lse"].cpu().numpy()[0, :, ~live] == -np.inf)
    assert np.all(out["dq"].cpu().numpy()[0, :, ~live] == 0)
    never = M.all(0)
    assert np.all(out["dk"].cpu().numpy()[0, :, never] == 0) and np.all(out["dv"].cpu().numpy()[0, :, never] == 0)


def test_single_attended_key(fm):
    """A row that attends one key returns that key's value row, lse = its score."""
    N, d = 256, 64
    lts = np.full(N, N, np.int32); lte = np.full(N, N, np.int32)
    uts = np.zeros(N, np.int32); ute = np.full(N, N, np.int32)   # everything masked ...
    ute[17] = 0; lts[17] = 200                                   # ... but column 17 for rows < 200
    m = {k: x[None, None] for k, x in zip(("lts", "lte", "uts", "ute"), (lts, lte, uts, ute))}
    wl = W.Workload("one", B=1, H=1, N=N, d=d, mask="causal")
    q, k, v, dO = W.make_inputs(wl.with_(N=N), seed=3)
    out = run_fm(fm, wl, m, q, k, v, dO)
    o = out["o"].cpu().numpy()[0, 0]
    np.testing.assert_allclose(o[:200], np.broadcast_to(v[0, 0, 17].float().numpy(), (200, d)), atol=1e-6)
    s = wl.scale * (q[0, 0, :200].double() @ k[0, 0, 17].double()).numpy()
    np.testing.assert_allclose(out["lse"].cpu().numpy()[0, 0, :200], s, atol=1e-3)


def test_deterministic_forward(fm):
    wl = W.SMALL["prefix_random_small"]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    a = run_fm(fm, wl, m, q, k, v)
    b = run_fm(fm, wl, m, q, k, v)
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])


def test_plan_mismatch_reported(fm):
    wl = W.SMALL["docs_small"]
    m = W.make_mask(wl)
    q, k, v, _ = W.make_inputs(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    plan64 = torch.empty(fm.fm_plan_bytes(wl.B, 1, wl.N, 64, 64), dtype=torch.uint8, device="cuda")
    fm.fm_tile_classify(att.bounds, plan64, att.status, 64, 64)
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    big = torch.empty(max(plan64.numel(), att.plan.numel()), dtype=torch.uint8, device="cuda")
    big[: plan64.numel()].copy_(plan64)
    fm.fm_attn_fwd(q.cuda(), k.cuda(), v.cuda(), att.bounds, big, wl.scale, o, lse, att.status)
    torch.cuda.synchronize()
    assert int(att.status.item()) == fm.FM_ERR_PLAN_MISMATCH


def test_host_rejects_bad_arguments(fm):
    wl = W.SMALL["causal_ragged"]
    m = W.make_mask(wl)
    q, k, v, _ = W.make_inputs(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    qd = q.cuda()
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_attn_fwd(qd, qd, qd, att.bounds, att.plan, -1.0, o, lse, att.status)
    assert e.value.code == fm.FM_ERR_INVALID_ARG
    q96 = torch.zeros((1, 1, 64, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_attn_fwd(q96, q96, q96, att.bounds, att.plan, 0.1, torch.empty_like(q96, dtype=torch.float32),
                       torch.empty((1, 1, 64), device="cuda"), att.status)
    assert e.value.code in (fm.FM_ERR_UNSUPPORTED, fm.FM_ERR_INVALID_ARG)
    with pytest.raises(fm.FmError) as e:
        ws = torch.empty(16, dtype=torch.uint8, device="cuda")
        g = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        fm.fm_attn_bwd(qd, qd, qd, o, lse, qd, att.bounds, att.plan, 0.1, g, g, g, ws, att.status)
    assert e.value.code == fm.FM_ERR_WORKSPACE


def test_bounded_wait_times_out_and_context_survives(fm):
    """A wait that nothing completes returns FM_ERR_TIMEOUT instead of hanging,
    and the GPU context keeps working afterwards."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fm.fm_selftest_wait_timeout(20_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == fm.FM_ERR_TIMEOUT
    wl = W.FULL["tiny_causal"]
    m = W.make_mask(wl)
    q, k, v, _ = W.make_inputs(wl)
    out = run_fm(fm, wl, m, q, k, v)
    O, _ = oracle.forward(q, k, v, m, wl.scale)
    check_close("O", out["o"].cpu().numpy(), O)


@pytest.mark.parametrize("kernel", ["forward", "backward"])
def test_real_kernel_wait_runs_out_and_context_survives(fm, kernel):
    """The real attention kernel's abort path: with the test hook armed, the
    first CTA of the launch withholds one tile load, the wait for it runs out
    after 2e6 cycles, the kernel reports FM_ERR_TIMEOUT (its other waits give
    up on the abort flag, it drains its copies and products and frees TMEM),
    and the context then still passes a parity case."""
    wl = W.Workload("unmasked_512", B=1, H=2, N=512, d=128, mask="full")   # every list has 4 tiles
    m = W.make_mask(wl)
    q, k, v, dO = (t.cuda() for t in W.make_inputs(wl))
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fm.fm_attn_fwd(q, k, v, att.bounds, att.plan, wl.scale, o, lse, att.status)
    torch.cuda.synchronize()
    assert int(att.status.item()) == 0
    g = [torch.empty(q.shape, dtype=torch.float32, device="cuda") for _ in range(3)]
    ws = torch.empty(fm.fm_bwd_workspace_bytes(*q.shape), dtype=torch.uint8, device="cuda")
    fm.fm_debug_wait_test(0 if kernel == "forward" else 1, 2_000_000)
    try:
        if kernel == "forward":
            fm.fm_attn_fwd(q, k, v, att.bounds, att.plan, wl.scale, o, lse, att.status)
        else:
            fm.fm_attn_bwd(q, k, v, o, lse, dO, att.bounds, att.plan, wl.scale, *g, ws, att.status)
        torch.cuda.synchronize()
    finally:
        fm.fm_debug_wait_test(-1, 0)
    assert int(att.status.item()) == fm.FM_ERR_TIMEOUT
    # the switch was consumed by that one launch; the context still works
    small = W.SMALL["docs_small"]
    ms = W.make_mask(small)
    qs, ks, vs, dOs = W.make_inputs(small)
    out = run_fm(fm, small, ms, qs, ks, vs, dOs)
    O, L = oracle.forward(qs, ks, vs, ms, small.scale)
    gr = oracle.backward(qs, ks, vs, dOs, ms, small.scale)
    check_all([("O", out["o"].cpu().numpy(), O), ("lse", out["lse"].cpu().numpy(), L),
               ("dQ", out["dq"].cpu().numpy(), gr["dq"]), ("dK", out["dk"].cpu().numpy(), gr["dk"]),
               ("dV", out["dv"].cpu().numpy(), gr["dv"])])


def test_profiler_records_every_launch(fm):
    """Every launch of a step, in order; fp32 gradients accumulate dQ in the
    caller's buffer directly (no postprocess), bf16 gradients go through the
    postprocess that scales and rounds the accumulator."""
    wl = W.SMALL["docs_small"]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    head = ["classify_minmax", "classify_lists", "classify_order", "fwd", "bwd_pre", "bwd"]
    for g_dtype, tail in ((torch.float32, []), (torch.bfloat16, ["bwd_post"])):
        fm.fm_profile_begin()
        run_fm(fm, wl, m, q, k, v, dO, g_dtype=g_dtype)
        rec = fm.fm_profile_end()
        assert [r[0] for r in rec] == head + tail, g_dtype
        assert all(ms > 0 for _, ms in rec)


def test_partial_tile_warp_summaries(fm):
    """A PARTIAL tile in which the first 32 rows (one softmax warp) are masked
    in every column, rows 64-95 in some columns and the other rows in none, so
    the forward's per-warp mask summary takes each of its three paths; another
    tile with a lower-triangle mask and one without any.  Element by element
    against the oracle, forward and backward."""
    B, H, N, d = 1, 2, 384, 128
    c = np.arange(N)
    lts, lte = np.zeros(N, np.int32), np.zeros(N, np.int32)
    uts, ute = np.zeros(N, np.int32), np.zeros(N, np.int32)
    t0 = c < 128
    lte[t0] = 32                                   # rows 0-31 in every column of KV tile 0
    uts[t0] = 64
    ute[t0] = 64 + c[t0] % 32                      # rows 64 .. 64 + c mod 32: mixed within rows 64-95
    t1 = (c >= 128) & (c < 256)
    lte[t1] = c[t1] - 128                          # KV tile 1: rows below c - 128
    m = {key: arr.reshape(1, 1, N).copy() for key, arr in (("lts", lts), ("lte", lte), ("uts", uts), ("ute", ute))}
    wl = W.Workload("warp_summaries", B=B, H=H, N=N, d=d, mask="full")
    q, k, v, dO = W.make_inputs(wl, seed=11)
    for flags in (0, 1):
        out = run_fm(fm, wl, m, q, k, v, dO, flags=flags)
        O, L = oracle.forward(q, k, v, m, wl.scale)
        g = oracle.backward(q, k, v, dO, m, wl.scale)
        check_all([("O", out["o"].cpu().numpy(), O), ("lse", out["lse"].cpu().numpy(), L),
                   ("dQ", out["dq"].cpu().numpy(), g["dq"]), ("dK", out["dk"].cpu().numpy(), g["dk"]),
                   ("dV", out["dv"].cpu().numpy(), g["dv"])])


def test_unaligned_bound_arrays_refused(fm):
    """Bound arrays must start on a 16-byte boundary (device pointers of the C
    ABI are 16-byte aligned; the forward reads four columns of each array per
    16-byte load).  Arrays 4 bytes past one are refused with
    FM_ERR_INVALID_ARG by the forward and the backward before any launch, and
    the same call with aligned copies of the same values then succeeds."""
    wl = W.SMALL["lognormal_small"]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    dev = torch.device("cuda")
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"], device=dev)
    views = []
    for key in ("lts", "lte", "uts", "ute"):
        src = torch.from_numpy(np.ascontiguousarray(m[key])).reshape(-1)
        buf = torch.zeros(src.numel() + 1, dtype=torch.int32, device=dev)
        buf[1:] = src.to(dev)
        views.append(buf[1:].view(m[key].shape))
    assert all(t.data_ptr() % 16 != 0 for t in views)
    bnd = fm.make_bounds(*views)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, dO))
    B, H, N, d = q.shape
    o = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    with pytest.raises(fm.FmError) as ei:
        fm.fm_attn_fwd(qd, kd, vd, bnd, att.plan, wl.scale, o, lse, att.status)
    assert ei.value.code == fm.FM_ERR_INVALID_ARG
    ws = torch.empty(fm.fm_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    gr = [torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev) for _ in range(3)]
    with pytest.raises(fm.FmError) as ei:
        fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, bnd, att.plan, wl.scale, *gr, ws, att.status)
    assert ei.value.code == fm.FM_ERR_INVALID_ARG
    fm.fm_attn_fwd(qd, kd, vd, att.bounds, att.plan, wl.scale, o, lse, att.status)
    torch.cuda.synchronize()
    att.check_status()
    O, L = oracle.forward(q, k, v, m, wl.scale)
    check_close("O", o.cpu().numpy(), O)
    check_lse(lse.cpu().numpy(), L)
