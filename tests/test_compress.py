"""Compressed column bounds (blog "FlashMask技术" §6.2 item 2: differential
encoding with 8-bit offsets), host side: the library's encoder output is
decoded here with an independent reader of the documented format and must
give the bounds back exactly; structured masks compress about 3.5-3.8x;
argument errors."""
import ctypes
import struct

import numpy as np
import pytest

from long_context_fm_gb300 import build as fmbuild
from long_context_fm_gb300 import workloads as W


@pytest.fixture(scope="module")
def fm():
    fmbuild.build()
    from long_context_fm_gb300 import fm as mod
    return mod


def decode(buf):
    """Reader of the compressed format: header (magic "FMC1", B, Hm, N, n_blk,
    pad, int64 payload bytes), directory of (offset << 1 | mode) per (b*Hm+hm,
    block, array), payload blocks (mode 0: int32 base + int8 deltas; mode 1:
    int32 values)."""
    buf = bytes(buf)
    magic, B, Hm, N, n_blk, _pad, payload_bytes = struct.unpack_from("<IiiiiiQ", buf, 0)
    assert magic == 0x31434D46 and n_blk == -(-N // 128)
    S = B * Hm
    dir_off = 32
    pay_off = dir_off + S * n_blk * 16
    assert pay_off + payload_bytes == len(buf)
    out = np.zeros((4, S, N), np.int64)
    for s in range(S):
        for blk in range(n_blk):
            ncol = min(128, N - blk * 128)
            for q in range(4):
                (e,) = struct.unpack_from("<I", buf, dir_off + ((s * n_blk + blk) * 4 + q) * 4)
                mode, off = e & 1, e >> 1
                p = pay_off + off
                if mode == 1:
                    vals = np.frombuffer(buf, np.int32, ncol, p).astype(np.int64)
                else:
                    (base,) = struct.unpack_from("<i", buf, p)
                    d = np.frombuffer(buf, np.int8, ncol - 1, p + 4).astype(np.int64)
                    vals = base + np.concatenate([[0], np.cumsum(d)])
                out[q, s, blk * 128: blk * 128 + ncol] = vals
    return [out[q].reshape(B, Hm, N) for q in range(4)]


CASES = list(W.SMALL) + ["tiny_causal", "doc_packing", "sliding_window", "sliding_window_sink", "prefix_lm",
                         "prefix_random", "long_packing_128k"]


@pytest.mark.parametrize("name", CASES)
def test_round_trip_through_the_format(fm, name):
    wl = W.SMALL.get(name) or W.FULL[name]
    m = W.make_mask(wl)
    c = fm.fm_bounds_compress(m["lts"], m["lte"], m["uts"], m["ute"])
    got = decode(c)
    for q, key in enumerate(("lts", "lte", "uts", "ute")):
        assert np.array_equal(got[q], m[key]), key


@pytest.mark.parametrize("name,ratio", [("long_packing_128k", 3.5), ("sliding_window", 3.5),
                                        ("doc_packing", 3.3), ("prefix_random", 2.0)])
def test_compression_ratio(fm, name, ratio):
    m = W.make_mask(W.FULL[name])
    c = fm.fm_bounds_compress(m["lts"], m["lte"], m["uts"], m["ute"])
    assert 16 * m["lts"].size / c.size >= ratio


def test_incompressible_and_ragged_bounds(fm):
    rng = np.random.default_rng(5)
    for N in (1, 127, 128, 129, 1000):
        arr = [rng.integers(0, N + 1, size=(2, 3, N)).astype(np.int32) for _ in range(4)]
        arr[1][0, 0, :] = np.arange(N)                    # one differential block family
        c = fm.fm_bounds_compress(*arr)
        got = decode(c)
        for q in range(4):
            assert np.array_equal(got[q], arr[q])


def test_argument_errors(fm):
    z = np.zeros((1, 1, 64), np.int32)
    p = z.ctypes.data_as(ctypes.c_void_p)
    n = fm._lib.fm_bounds_compressed_bytes(p, p, p, p, 1, 1, 64)
    assert n > 0
    out = np.zeros(n, np.uint8)
    po = out.ctypes.data_as(ctypes.c_void_p)
    assert fm._lib.fm_bounds_compress(p, p, p, p, 1, 1, 64, po, n - 1) == fm.FM_ERR_WORKSPACE
    assert fm._lib.fm_bounds_compress(p, p, p, p, 1, 1, 64, None, n) == fm.FM_ERR_WORKSPACE
    assert fm._lib.fm_bounds_compress(None, p, p, p, 1, 1, 64, po, n) == fm.FM_ERR_INVALID_ARG
    assert fm._lib.fm_bounds_compressed_bytes(p, p, p, p, 0, 1, 64) == 0
    assert fm._lib.fm_bounds_compress(p, p, p, p, 1, 1, 64, po, n) == fm.FM_OK
