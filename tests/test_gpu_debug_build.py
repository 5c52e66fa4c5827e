"""The FM_DEBUG build: the same kernels with device-side checks that record
FM_ERR_DEBUG_CHECK in the status word instead of trapping (plan entries
within range with a FULL or PARTIAL label, the TMEM allocation at column 0,
and at the end of every CTA each pipeline mbarrier's phase parity against the
tiles, halves and units the CTA processed).  The parity cases run through it
in both precision modes, plus the FP8 forward: every check must pass (status
0) and the results must still match the oracle.  Only valid inputs are used;
failure reporting without a GPU fault is covered by the wait-limit tests."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))
import torch
import oracle
from long_context_fm_gb300 import fm
from long_context_fm_gb300 import workloads as W
from parity import check_all, check_close, check_lse, run_fm

assert fm._LIB_PATH.endswith("libfm_debug.so"), fm._LIB_PATH
for name in ["causal_ragged", "docs_small", "window_small", "prefix_small", "random_cols_d64",
             "lognormal_small", "window_sink_small", "all_masked_small"]:
    wl = W.SMALL[name]
    m = W.make_mask(wl)
    q, k, v, dO = W.make_inputs(wl)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    g = oracle.backward(q, k, v, dO, m, wl.scale)
    for flags in ((1,) if wl.input_scale != 1.0 else (0, 1)):
        out = run_fm(fm, wl, m, q, k, v, dO, flags=flags)   # asserts status 0 after each launch
        check_all([("O", out["o"].cpu().numpy(), O), ("lse", out["lse"].cpu().numpy(), L),
                   ("dQ", out["dq"].cpu().numpy(), g["dq"]), ("dK", out["dk"].cpu().numpy(), g["dk"]),
                   ("dV", out["dv"].cpu().numpy(), g["dv"])])
        print("ok", name, flags, flush=True)

# FP8 forward (d = 128, N a multiple of 16): status 0 with the debug checks.
wl = W.SMALL["lognormal_small"]
m = W.make_mask(wl)
q, k, v, dO = W.make_inputs(wl)
att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"], device=torch.device("cuda"))
q8, dq8 = fm.fm_quantize_fp8(q.cuda())
k8, dk8 = fm.fm_quantize_fp8(k.cuda())
vt8, dv8 = fm.fm_quantize_fp8(v.cuda(), transpose=True)
o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
fm.fm_attn_fwd_fp8(q8, k8, vt8, torch.cat([dq8, dk8, dv8]), att.bounds, att.plan, wl.scale, o, lse, att.status)
torch.cuda.synchronize()
att.check_status()
print("DEBUG-BUILD-OK", flush=True)
"""


def test_debug_build_checks_pass_and_results_match_oracle():
    from long_context_fm_gb300 import build

    lib = build.build(debug=True)
    env = dict(os.environ, FM_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", "import os\nROOT = %r\n" % ROOT + SCRIPT], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0 and "DEBUG-BUILD-OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
