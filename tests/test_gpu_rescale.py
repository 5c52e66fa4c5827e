"""Forward parity when the running row max rises from KV tile to KV tile, so
that the online softmax's lazy rescale of O runs on many tiles: the two
softmax warpgroups take alternate tiles and hand the running max on, and the
owner of a tile that raises it beyond the band rescales O after the previous
tile's P V.  The exact softmax does not depend on any of this (FlashAttention
article §二.2: the max-subtracted softmax), so O and lse must match the oracle.

Inputs: standard-normal bf16 Q, K, V, with Q[..., 0] = 4 and K[j, 0] =
beta * (j // 128), so that the scores of KV tile t sit about
t * step_log2 (base 2, after the softmax scale) above those of tile 0.  Under
a causal mask the Q tile t walks KV tiles 0..t, every one raising its rows'
maximum: with a step of 40 beyond the bf16 path's band of 2^32 on every tile,
with 20 on every other tile.  Only the forward is compared: the backward uses
the exact lse (no lazy rescale) and, with K entries in the hundreds, its dQ is
outside the absolute bound for reasons unrelated to this path."""
import numpy as np
import pytest
import torch

import oracle
from long_context_fm_gb300 import workloads as W
from parity import check_close, check_lse, run_fm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    from long_context_fm_gb300 import fm as mod
    return mod


def rising_inputs(wl, step_log2, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (wl.B, wl.H, wl.N, wl.d)
    q = torch.randn(shape, generator=g)
    k = torch.randn(shape, generator=g)
    v = torch.randn(shape, generator=g)
    beta = step_log2 / (4.0 * wl.scale * np.log2(np.e))
    q[..., 0] = 4.0
    k[..., 0] = beta * (torch.arange(wl.N) // 128).float()
    return q.bfloat16(), k.bfloat16(), v.bfloat16()


@pytest.mark.parametrize("precise", [False, True])
@pytest.mark.parametrize("step_log2", [20.0, 40.0])
def test_rising_row_max_matches_oracle(fm, step_log2, precise):
    wl = W.Workload("rising_causal", B=1, H=2, N=1024, d=128, mask="causal")
    m = W.make_mask(wl)
    q, k, v = rising_inputs(wl, step_log2, seed=11)
    out = run_fm(fm, wl, m, q, k, v, flags=1 if precise else 0)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    # The scores really do rise by the step from tile to tile.
    s = (q[0, 0, -1].double() @ k[0, 0].double().T) * wl.scale * np.log2(np.e)
    tile_max = s.reshape(-1, 128).max(dim=1).values
    assert float((tile_max[1:] - tile_max[:-1]).min()) > 0.8 * step_log2
    check_close("O", out["o"].cpu().numpy(), O)
    check_lse(out["lse"].cpu().numpy(), L)


def test_rising_row_max_ragged_d64(fm):
    """The same on d = 64 with a ragged last tile (N = 1000)."""
    wl = W.Workload("rising_causal_d64", B=1, H=2, N=1000, d=64, mask="causal")
    m = W.make_mask(wl)
    q, k, v = rising_inputs(wl, 40.0, seed=12)
    out = run_fm(fm, wl, m, q, k, v, flags=0)
    O, L = oracle.forward(q, k, v, m, wl.scale)
    check_close("O", out["o"].cpu().numpy(), O)
    check_lse(out["lse"].cpu().numpy(), L)
