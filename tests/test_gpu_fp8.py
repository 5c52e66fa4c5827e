"""FP8 (e4m3) forward on the GPU.

* The quantizer's codes and descale equal the oracle's bit for bit (plain and
  transposed layouts): the division and the rounding are the same fp32
  operation on both sides.
* The forward on those codes matches the oracle's exact attention on the
  oracle's own codes.  The kernel rounds P to e4m3 for the P V product
  (relative error <= 2^-4 per weight) and normalises by the fp32 sum of the
  unrounded P, so |O - O_exact| <= 2^-4 max|V| for every element (a sound
  bound).  A row's error is a weighted mean of its weights' relative rounding
  errors, whose RMS is at most 2^-4 / sqrt(3) (uniform rounding within half a
  step; fewer than that when a row has one dominant weight, which is exact at
  P = 1): rel-L2 <= 2^-4 / sqrt(3) ~ 0.036 whatever the number of keys a row
  attends.  lse comes from fp32 sums of the unrounded P: within 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


CASES = {
    "fp8_causal": W.Workload("fp8_causal", B=1, H=2, N=624, d=128, mask="causal"),
    "fp8_docs": W.Workload("fp8_docs", B=2, H=2, N=1008, d=128, mask="docs_uniform", params=dict(lo=16, hi=300)),
    "random_cols_small": W.SMALL["random_cols_small"],
    "prefix_small": W.SMALL["prefix_small"],
    "fp8_sink": W.Workload("fp8_sink", B=1, H=2, N=768, d=128, mask="window_sink", params=dict(window=100, sink=10)),
}


@pytest.mark.parametrize("name", ["fp8_causal", "prefix_small"])
def test_quantizer_matches_oracle_codes(fm, name):
    wl = CASES[name]
    q, k, v, _ = W.make_inputs(wl)
    for x, transpose in ((q, False), (v, True), (k, False)):
        codes, ds = fm.fm_quantize_fp8(x.cuda(), transpose=transpose)
        ref, ref_ds = oracle.quantize_e4m3(x, transpose=transpose)
        torch.cuda.synchronize()
        assert np.float32(ds.item()) == ref_ds
        got = codes.cpu().numpy()
        assert got.shape == ref.shape
        assert np.array_equal(got, ref), f"{(got != ref).sum()} codes differ"


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_forward_matches_oracle(fm, name):
    wl = CASES[name]
    m = W.make_mask(wl)
    q, k, v, _ = W.make_inputs(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    q8, dq = fm.fm_quantize_fp8(q.cuda())
    k8, dk = fm.fm_quantize_fp8(k.cuda())
    vt8, dv = fm.fm_quantize_fp8(v.cuda(), transpose=True)
    descale = torch.cat([dq, dk, dv])
    o = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    fm.fm_attn_fwd_fp8(q8, k8, vt8, descale, att.bounds, att.plan, wl.scale, o, lse, att.status)
    torch.cuda.synchronize()
    att.check_status()
    rq, rdq = oracle.quantize_e4m3(q)
    rk, rdk = oracle.quantize_e4m3(k)
    rvt, rdv = oracle.quantize_e4m3(v, transpose=True)
    O, L = oracle.forward_fp8(rq, rk, rvt, (rdq, rdk, rdv), m, wl.scale)
    got = o.cpu().numpy()
    assert np.isfinite(got).all()
    vmax = float(np.abs(oracle.e4m3_decode(rvt)).max() * rdv)
    assert np.abs(got - O).max() <= 2.0 ** -4 * vmax + 1e-6
    rel = np.linalg.norm(got - O) / max(np.linalg.norm(O), 1e-30)
    assert rel <= 2.0 ** -4 / np.sqrt(3), rel
    check_lse(lse.cpu().numpy(), L)


def test_fp8_bf16_output_and_argument_errors(fm):
    wl = CASES["fp8_causal"]
    m = W.make_mask(wl)
    q, k, v, _ = W.make_inputs(wl)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    q8, dq = fm.fm_quantize_fp8(q.cuda())
    k8, dk = fm.fm_quantize_fp8(k.cuda())
    vt8, dv = fm.fm_quantize_fp8(v.cuda(), transpose=True)
    descale = torch.cat([dq, dk, dv])
    o32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    o16 = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fm.fm_attn_fwd_fp8(q8, k8, vt8, descale, att.bounds, att.plan, wl.scale, o32, lse, att.status)
    fm.fm_attn_fwd_fp8(q8, k8, vt8, descale, att.bounds, att.plan, wl.scale, o16, lse, att.status)
    torch.cuda.synchronize()
    att.check_status()
    assert torch.equal(o16, o32.to(torch.bfloat16))
    # d = 64 and N not a multiple of 16 are not supported
    x = torch.zeros(1, 1, 40, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_quantize_fp8(x, transpose=True)
    assert e.value.code == fm.FM_ERR_UNSUPPORTED
    wl64 = W.Workload("c64", B=1, H=1, N=128, d=64, mask="causal")
    m64 = W.make_mask(wl64)
    att64 = fm.MaskedAttention(m64["lts"], m64["lte"], m64["uts"], m64["ute"])
    z8 = torch.zeros(1, 1, 128, 64, dtype=torch.uint8, device="cuda")
    o = torch.empty(1, 1, 128, 64, dtype=torch.float32, device="cuda")
    l64 = torch.empty(1, 1, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_attn_fwd_fp8(z8, z8, z8.view(1, 1, 64, 128), descale, att64.bounds, att64.plan, 0.1, o, l64,
                           att64.status)
    assert e.value.code == fm.FM_ERR_UNSUPPORTED
