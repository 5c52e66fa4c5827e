"""Row windows on the GPU (the per-rank computation of context parallelism),
ranks emulated one after another on one device: each window's O, lse and dQ
match the oracle's rows of the whole mask, and the windows' dK, dV
contributions summed match the oracle's gradients, within the parity
tolerances; each window's O and lse are also the library's full call's rows
bit for bit (a Q tile's list of key tiles does not
depend on the window), dQ matches within the atomics' rounding, the dK, dV
contributions of the windows add up to the full gradients, the window's tile
labels are the oracle's rows, and key shards a window never attends get
exactly zero."""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import cp
from long_context_fm_gb300 import workloads as W
from parity import check_all, mode_for, run_fm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


def _costs(m):
    return (oracle.tile_labels_all(m, 128, 128) != oracle.SKIP).sum(axis=(0, 1, 3))


CASES = [("causal_1000", 3), ("docs_small", 2), ("window_sink_small", 3), ("random_cols_small", 2)]


@pytest.mark.parametrize("name,world", CASES)
def test_windows_reassemble_the_full_step(fm, name, world):
    wl = W.Workload("causal_1000", B=1, H=2, N=1000, d=128, mask="causal") if name == "causal_1000" else W.SMALL[name]
    m = W.make_mask(wl)
    flags = fm.FM_FLAG_PRECISE if mode_for(wl) else 0
    q, k, v, dO = (t.cuda() for t in W.make_inputs(wl))
    full = run_fm(fm, wl, m, q, k, v, dO, flags=flags)
    bounds = [torch.from_numpy(np.ascontiguousarray(m[x])).cuda() for x in ("lts", "lte", "uts", "ute")]
    splits = cp.balanced_splits(_costs(m), wl.N, world)
    local = cp.LibraryLocal(flags)
    qc, kc, vc, dOc = (t.cpu() for t in (q, k, v, dO))
    O_ref, L_ref = oracle.forward(qc, kc, vc, m, wl.scale)
    g_ref = oracle.backward(qc, kc, vc, dOc, m, wl.scale)
    dk_sum = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    dv_sum = torch.zeros_like(dk_sum)
    for r in range(world):
        r0, r1 = splits[r], splits[r + 1]
        qs, dOs = q[:, :, r0:r1].contiguous(), dO[:, :, r0:r1].contiguous()
        o, lse = local.forward(qs, k, v, bounds, r0, wl.scale)
        dq, dk, dv = local.backward(qs, k, v, o, lse, dOs, bounds, r0, wl.scale)
        # each window against the oracle's rows of the whole mask ...
        check_all([(f"O window {r}", o.cpu().numpy(), O_ref[:, :, r0:r1]),
                   ("lse", lse.cpu().numpy(), L_ref[:, :, r0:r1]),
                   (f"dQ window {r}", dq.cpu().numpy(), g_ref["dq"][:, :, r0:r1])])
        # ... and against the library's own whole-mask call
        assert torch.equal(o, full["o"][:, :, r0:r1]), r
        assert torch.equal(lse, full["lse"][:, :, r0:r1]), r
        torch.testing.assert_close(dq, full["dq"][:, :, r0:r1], rtol=1e-5, atol=1e-6)
        dk_sum += dk
        dv_sum += dv
    check_all([("dK summed over windows", dk_sum.cpu().numpy(), g_ref["dk"]),
               ("dV summed over windows", dv_sum.cpu().numpy(), g_ref["dv"])])
    torch.testing.assert_close(dk_sum, full["dk"], rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(dv_sum, full["dv"], rtol=1e-5, atol=1e-5)


def test_window_labels_are_the_oracles_rows(fm):
    wl = W.SMALL["window_sink_small"]
    m = W.make_mask(wl)
    ref = oracle.tile_labels_all(m, 64, 128)                   # [B, Hm, n_q, n_k]
    bt = [torch.from_numpy(np.ascontiguousarray(m[x])).cuda() for x in ("lts", "lte", "uts", "ute")]
    bnd = fm.make_bounds(*bt)          # raw pointers: bt keeps the tensors alive
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for q_row0, Nq in ((0, wl.N), (192, 300), (640, wl.N - 640), (64, 1)):
        plan = torch.empty(fm.fm_plan_bytes_rows(wl.B, wl.Hm, wl.N, q_row0, Nq, 64, 128), dtype=torch.uint8,
                           device="cuda")
        n_q = -(-Nq // 64)
        labels = torch.empty((wl.B, wl.Hm, n_q, ref.shape[3]), dtype=torch.uint8, device="cuda")
        fm.fm_tile_classify_rows(bnd, q_row0, Nq, plan, status, bq=64, bk=128, labels=labels)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        want = oracle.tile_labels(*[m[x][0, 0] for x in ("lts", "lte", "uts", "ute")], 64, 128)
        # a ragged last window tile covers fewer rows than the whole-mask tile of the same index
        lbl = labels.cpu().numpy()[0, 0]
        t0 = q_row0 // 64
        full_rows = lbl[:-1] if (q_row0 + Nq) % 64 and q_row0 + Nq < wl.N else lbl
        assert np.array_equal(full_rows, want[t0:t0 + full_rows.shape[0]]), (q_row0, Nq)


def test_causal_window_skips_later_key_shards(fm):
    """Rows [0, 384) of a causal mask attend keys [0, 384) only: the window's
    dK, dV contribution is exactly zero for every later key."""
    wl = W.Workload("c", B=1, H=2, N=1024, d=64, mask="causal")
    m = W.make_mask(wl)
    q, k, v, dO = (t.cuda() for t in W.make_inputs(wl))
    bounds = [torch.from_numpy(np.ascontiguousarray(m[x])).cuda() for x in ("lts", "lte", "uts", "ute")]
    local = cp.LibraryLocal()
    qs, dOs = q[:, :, :384].contiguous(), dO[:, :, :384].contiguous()
    o, lse = local.forward(qs, k, v, bounds, 0, wl.scale)
    dq, dk, dv = local.backward(qs, k, v, o, lse, dOs, bounds, 0, wl.scale)
    assert torch.count_nonzero(dk[:, :, 384:]) == 0 and torch.count_nonzero(dv[:, :, 384:]) == 0
    assert torch.count_nonzero(dk[:, :, :384]) > 0
    # the window's rows against the oracle
    O, L = oracle.forward(q.cpu(), k.cpu(), v.cpu(), m, wl.scale, rows=np.arange(384))
    check_all([("O window", o.cpu().numpy(), O)])


def test_window_argument_errors(fm):
    wl = W.SMALL["causal_ragged"]
    m = W.make_mask(wl)
    bt = [torch.from_numpy(np.ascontiguousarray(m[x])).cuda() for x in ("lts", "lte", "uts", "ute")]
    bnd = fm.make_bounds(*bt)          # raw pointers: bt keeps the tensors alive
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fm.fm_plan_bytes_rows(1, 1, wl.N, 100, 50) == 0                 # not tile aligned
    assert fm.fm_plan_bytes_rows(1, 1, wl.N, 256, wl.N) == 0               # past the end
    plan = torch.empty(fm.fm_plan_bytes_rows(1, 1, wl.N, 128, 100), dtype=torch.uint8, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_tile_classify_rows(bnd, 100, 50, plan, status)
    assert e.value.code == fm.FM_ERR_INVALID_ARG
    fm.fm_tile_classify_rows(bnd, 128, 100, plan, status)
    q, k, v, _ = (t.cuda() for t in W.make_inputs(wl))
    qs = q[:, :, 0:100].contiguous()
    o = torch.empty(qs.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(qs.shape[:3], dtype=torch.float32, device="cuda")
    fm.fm_attn_fwd_rows(qs, k, v, bnd, plan, 0, wl.scale, o, lse, status)  # plan of rows [128, 228)
    torch.cuda.synchronize()
    assert int(status.item()) == fm.FM_ERR_PLAN_MISMATCH
