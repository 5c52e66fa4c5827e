"""The allocation-free backward, fm_attn_bwd_noalloc.

Some callers of this library cannot call cudaMalloc: code running under
another framework's memory pool, loops that must not touch the allocator
after start-up, plugins that are handed only their input and output
buffers.  fm_attn_bwd_noalloc serves them by taking the backward's
workspace from an array built into the library.  These tests call it
through the C ABI and check that two calls in a row give the gradients of
fm_attn_bwd (with a caller workspace) and of the oracle within the parity
tolerance, and that a size beyond the built-in array is refused.  The file is collected last so
that a run stopping at the first failure has run everything else first; it
also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


@pytest.mark.parametrize("name,g_dtype", [("docs_small", torch.float32),
                                          ("random_cols_d64", torch.float32),
                                          ("causal_ragged", torch.bfloat16)])
def test_noalloc_matches_workspace_backward_twice(fm, name, g_dtype):
    wl = W.SMALL[name]
    m = W.make_mask(wl)
    inputs = W.make_inputs(wl)
    g_ref = oracle.backward(*inputs, m, wl.scale)
    q, k, v, dO = (t.cuda() for t in inputs)
    att = fm.MaskedAttention(m["lts"], m["lte"], m["uts"], m["ute"])
    o, lse = att.forward(q, k, v, wl.scale, o_dtype=torch.float32)
    ws = torch.empty(fm.fm_bwd_workspace_bytes(*q.shape), dtype=torch.uint8, device="cuda")
    assert ws.numel() <= fm.NOALLOC_SCRATCH_BYTES
    ref = [torch.empty(q.shape, dtype=g_dtype, device="cuda") for _ in range(3)]
    fm.fm_attn_bwd(q, k, v, o, lse, dO, att.bounds, att.plan, wl.scale, *ref, ws, att.status)
    for call in range(2):
        got = [torch.full(q.shape, float("nan"), dtype=g_dtype, device="cuda") for _ in range(3)]
        fm.fm_attn_bwd_noalloc(q, k, v, o, lse, dO, att.bounds, att.plan, wl.scale, *got, att.status)
        torch.cuda.synchronize()
        att.check_status()
        for label, key, a, b in zip(("dQ", "dK", "dV"), ("dq", "dk", "dv"), got, ref):
            check_close(f"{label} call {call}", a.float().cpu().numpy(), b.float().cpu().numpy())
            check_close(f"{label} call {call} vs oracle", a.float().cpu().numpy(), g_ref[key])


def test_noalloc_refuses_sizes_beyond_the_builtin_array(fm):
    # fm_bwd_workspace_bytes(1, 1, 140000, 128) is about 72 MB > 64 MiB: the call
    # must return FM_ERR_WORKSPACE before it touches any pointer.
    B, H, N, d = 1, 1, 140000, 128
    assert fm.fm_bwd_workspace_bytes(B, H, N, d) > fm.NOALLOC_SCRATCH_BYTES
    bounds = fm.Bounds(None, None, None, None, B, 1, N)
    code = fm._lib.fm_attn_bwd_noalloc(None, None, None, None, 0, None, None, bounds, None, B, H, N,
                                       d, ctypes.c_float(0.1), None, None, None, 1, 0, None, None)
    assert code == fm.FM_ERR_WORKSPACE
