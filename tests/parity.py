"""Shared helpers of the parity tests: running the CUDA path through the C ABI
and comparing with the oracle under the stated tolerances.

Tolerances (fixed by the method's target; outputs in fp32 so that output
rounding is not counted):
  O, dQ, dK, dV : max |x - ref| <= 2e-2  and  ||x - ref||_2 / ||ref||_2 <= 1e-2
  lse           : max |x - ref| <= 1e-3 on finite entries; -inf entries match
                  exactly; no NaN anywhere.
"""
import numpy as np
import torch

ATOL = 2e-2
RTOL_L2 = 1e-2
LSE_ATOL = 1e-3


def check_close(name, got, ref, atol=ATOL, rl2=RTOL_L2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert not np.isnan(got).any(), f"{name}: NaN in output"
    err = np.abs(got - ref).max() if got.size else 0.0
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got - ref)
    assert err <= atol and rel <= rl2, f"{name}: max-abs {err:.3e} (<= {atol}), rel-L2 {rel:.3e} (<= {rl2})"
    return err, rel


def check_all(items):
    """check_close on every (name, got, ref) and the lse check on ("lse", got, ref);
    every output is checked and all failures are reported together."""
    msgs, report = [], []
    for name, got, ref in items:
        try:
            if name == "lse":
                check_lse(got, ref)
                report.append("lse ok")
            else:
                err, rel = check_close(name, got, ref)
                report.append(f"{name} {err:.2e}/{rel:.2e}")
        except AssertionError as e:
            msgs.append(str(e))
    print("; ".join(report))
    assert not msgs, " | ".join(msgs)


def check_lse(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert not np.isnan(got).any(), "lse: NaN"
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "lse: -inf pattern differs"
    assert np.all(got[~fin] == -np.inf)
    if fin.any():
        err = np.abs(got[fin] - ref[fin]).max()
        assert err <= LSE_ATOL, f"lse: max-abs {err:.3e} (<= {LSE_ATOL})"


def to_dev_mask(m, device="cuda"):
    return [torch.from_numpy(np.ascontiguousarray(m[k])).to(device) for k in ("lts", "lte", "uts", "ute")]


def mode_for(wl):
    """Precision mode of the parity runs: the x2-scaled prefix workloads have
    gradients of tens, where one bf16 rounding of P and dS exceeds the max-abs
    bound, so they run in precise mode; every other workload runs in the
    standard mode that bench.py times."""
    return 1 if wl.input_scale != 1.0 else 0


def run_fm(fm, wl, m, q, k, v, dO=None, o_dtype=torch.float32, g_dtype=torch.float32, flags=None):
    """Classify + forward (+ backward) through the C ABI.  Outputs are
    NaN-poisoned first so that an element the kernels never write fails."""
    flags = mode_for(wl) if flags is None else flags
    dev = torch.device("cuda")
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"], device=dev)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    B, H, N, d = q.shape
    o = torch.full(q.shape, float("nan"), dtype=o_dtype, device=dev)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    fm.fm_attn_fwd(qd, kd, vd, att.bounds, att.plan, wl.scale, o, lse, att.status, flags=flags)
    out = dict(att=att, o=o, lse=lse)
    torch.cuda.synchronize()
    code = int(att.status.item())
    assert code == 0, f"forward: device status {code} ({fm.fm_status_string(code)})"
    if dO is not None:
        dod = dO.to(dev)
        ws = torch.full((fm.fm_bwd_workspace_bytes(B, H, N, d),), 0xFF, dtype=torch.uint8, device=dev)
        g = [torch.full(q.shape, float("nan"), dtype=g_dtype, device=dev) for _ in range(3)]
        fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, att.bounds, att.plan, wl.scale, *g, ws, att.status,
                       flags=flags)
        out.update(dq=g[0], dk=g[1], dv=g[2])
    torch.cuda.synchronize()
    att.check_status()
    return out
