"""Oracle for FlashMask-style masked attention (fp64, CPU).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library under
``long_context_fm_gb300`` never does, and this package never imports it.

The arithmetic lives in ``oracle.c`` (plain loops, fp64, OpenMP); this module
only builds it with gcc, marshals numpy arrays and loops over (batch, head).
Definitions and the pages' passages they follow are in the header comment of
``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lib = None

SKIP, FULL, PARTIAL = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (-O2, OpenMP, IEEE fp64: no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _configure(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_dense_from_cols.argtypes = [P, P, P, P, I64, P]
    lib.oracle_dense_from_rows.argtypes = [P, P, I64, P]
    lib.oracle_dense_from_row_intervals.argtypes = [P, P, I64, I64, P]
    lib.oracle_attended_pairs.argtypes = [P, P, P, P, I64]
    lib.oracle_attended_pairs.restype = I64
    lib.oracle_fwd_rows.argtypes = [P, P, P, P, P, P, P, I64, ctypes.c_int, ctypes.c_double,
                                    P, I64, P, P]
    lib.oracle_bwd_rows.argtypes = [P, P, P, P, P, P, P, P, I64, ctypes.c_int, ctypes.c_double,
                                    P, I64, P, P, P]
    lib.oracle_bwd_cols.argtypes = [P, P, P, P, P, P, P, P, I64, ctypes.c_int, ctypes.c_double,
                                    P, P, P, I64, P, P]
    lib.oracle_tile_labels.argtypes = [P, P, P, P, I64, ctypes.c_int, ctypes.c_int, P]
    lib.oracle_tile_labels_exact.argtypes = [P, P, P, P, I64, ctypes.c_int, ctypes.c_int, P]
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _f32(t):
    """bf16/fp32 torch tensor or numpy array -> contiguous float32 numpy."""
    if hasattr(t, "detach"):
        import torch
        t = t.detach().to("cpu", torch.float32).numpy()
    return np.ascontiguousarray(t, dtype=np.float32)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _bounds_of(mask, b, hm):
    return tuple(_i32(mask[key][b, hm]) for key in ("lts", "lte", "uts", "ute"))


# ---- masks -------------------------------------------------------------------
def dense_from_cols(lts, lte, uts, ute) -> np.ndarray:
    """Dense boolean mask (True = masked) of one head from the column rule."""
    lts, lte, uts, ute = map(_i32, (lts, lte, uts, ute))
    N = lts.shape[0]
    M = np.empty((N, N), np.uint8)
    _load().oracle_dense_from_cols(_p(lts), _p(lte), _p(uts), _p(ute), N, _p(M))
    return M.astype(bool)


def dense_from_rows(cs, ce) -> np.ndarray:
    """Dense boolean mask (True = masked) of one head from the row rule."""
    cs, ce = _i32(cs), _i32(ce)
    N = cs.shape[0]
    M = np.empty((N, N), np.uint8)
    _load().oracle_dense_from_rows(_p(cs), _p(ce), N, _p(M))
    return M.astype(bool)


def dense_from_row_intervals(starts, ends) -> np.ndarray:
    """Dense boolean mask (True = masked) of one head from K inclusive
    intervals per row (int32 [N, K])."""
    starts, ends = _i32(starts), _i32(ends)
    N, K = starts.shape
    M = np.empty((N, N), np.uint8)
    _load().oracle_dense_from_row_intervals(_p(starts), _p(ends), N, K, _p(M))
    return M.astype(bool)


def attended_pairs(lts, lte, uts, ute) -> int:
    lts, lte, uts, ute = map(_i32, (lts, lte, uts, ute))
    return int(_load().oracle_attended_pairs(_p(lts), _p(lte), _p(uts), _p(ute), lts.shape[0]))


# ---- attention ---------------------------------------------------------------
def forward(q, k, v, mask, scale, rows=None, heads=None):
    """O [B,H,R,d] and lse [B,H,R] in fp64 for rows ``rows`` (default: all).

    ``mask`` holds ``lts, lte, uts, ute`` int32 [B, Hm, N]; head h uses mask
    head ``h`` when Hm == H, else 0.  ``heads`` restricts to a list of
    (b, h) pairs; the outputs then have shape [len(heads), R, ...]."""
    lib = _load()
    qf, kf, vf = _f32(q), _f32(k), _f32(v)
    B, H, N, d = qf.shape
    Hm = mask["lts"].shape[1]
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    O = np.zeros((len(pairs), rows.size, d))
    lse = np.zeros((len(pairs), rows.size))
    for n, (b, h) in enumerate(pairs):
        bd = _bounds_of(mask, b, h if Hm == H else 0)
        Ob = np.zeros((rows.size, d))
        lb = np.zeros(rows.size)
        lib.oracle_fwd_rows(_p(np.ascontiguousarray(qf[b, h])), _p(np.ascontiguousarray(kf[b, h])),
                            _p(np.ascontiguousarray(vf[b, h])), *map(_p, bd), N, d, float(scale),
                            _p(rows), rows.size, _p(Ob), _p(lb))
        O[n], lse[n] = Ob, lb
    if heads is None:
        return O.reshape(B, H, rows.size, d), lse.reshape(B, H, rows.size)
    return O, lse


def backward(q, k, v, dO, mask, scale, rows=None, cols=None, heads=None):
    """dQ for ``rows`` and dK, dV for ``cols`` (default: all) in fp64.

    Returns dict(dq, dk, dv, lse, D) where lse and D are for ``rows``."""
    lib = _load()
    qf, kf, vf, dof = _f32(q), _f32(k), _f32(v), _f32(dO)
    B, H, N, d = qf.shape
    Hm = mask["lts"].shape[1]
    rows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, np.int64)
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    P = len(pairs)
    dq = np.zeros((P, rows.size, d)); lse = np.zeros((P, rows.size)); D = np.zeros((P, rows.size))
    dk = np.zeros((P, cols.size, d)); dv = np.zeros((P, cols.size, d))
    for n, (b, h) in enumerate(pairs):
        bd = _bounds_of(mask, b, h if Hm == H else 0)
        qh, kh = np.ascontiguousarray(qf[b, h]), np.ascontiguousarray(kf[b, h])
        vh, doh = np.ascontiguousarray(vf[b, h]), np.ascontiguousarray(dof[b, h])
        dqb = np.zeros((rows.size, d)); lb = np.zeros(rows.size); Db = np.zeros(rows.size)
        lib.oracle_bwd_rows(_p(qh), _p(kh), _p(vh), _p(doh), *map(_p, bd), N, d, float(scale),
                            _p(rows), rows.size, _p(dqb), _p(lb), _p(Db))
        dq[n], lse[n], D[n] = dqb, lb, Db
        if cols.size:
            # Row statistics for every row that attends a listed column.
            need = _rows_attending(bd, cols, N)
            lse_full = np.zeros(N); D_full = np.zeros(N)
            if need.size:
                tmp = np.zeros((need.size, d)); ln = np.zeros(need.size); Dn = np.zeros(need.size)
                lib.oracle_bwd_rows(_p(qh), _p(kh), _p(vh), _p(doh), *map(_p, bd), N, d,
                                    float(scale), _p(need), need.size, _p(tmp), _p(ln), _p(Dn))
                lse_full[need] = ln
                D_full[need] = Dn
            dkb = np.zeros((cols.size, d)); dvb = np.zeros((cols.size, d))
            lib.oracle_bwd_cols(_p(qh), _p(kh), _p(vh), _p(doh), *map(_p, bd), N, d, float(scale),
                                _p(lse_full), _p(D_full), _p(cols), cols.size, _p(dkb), _p(dvb))
            dk[n], dv[n] = dkb, dvb
    out = dict(dq=dq, dk=dk, dv=dv, lse=lse, D=D)
    if heads is None:
        out = {key: val.reshape((B, H) + val.shape[1:]) for key, val in out.items()}
    return out


def _rows_attending(bd, cols, N):
    """Rows that attend at least one of ``cols`` (column rule, per element)."""
    lts, lte, uts, ute = bd
    i = np.arange(N, dtype=np.int64)
    need = np.zeros(N, bool)
    for j in cols:
        masked = ((lts[j] <= i) & (i < lte[j])) | ((uts[j] <= i) & (i < ute[j]))
        need |= ~masked
    return np.nonzero(need)[0].astype(np.int64)


# ---- tile labels -------------------------------------------------------------
def tile_labels(lts, lte, uts, ute, bq=128, bk=128, exact=False) -> np.ndarray:
    """uint8 [n_q, n_k] labels of one mask head (0 skip, 1 full, 2 partial)."""
    lts, lte, uts, ute = map(_i32, (lts, lte, uts, ute))
    N = lts.shape[0]
    n_q, n_k = -(-N // bq), -(-N // bk)
    out = np.empty((n_q, n_k), np.uint8)
    fn = _load().oracle_tile_labels_exact if exact else _load().oracle_tile_labels
    fn(_p(lts), _p(lte), _p(uts), _p(ute), N, bq, bk, _p(out))
    return out


def tile_labels_all(mask, bq=128, bk=128, exact=False) -> np.ndarray:
    """uint8 [B, Hm, n_q, n_k]."""
    B, Hm, _ = mask["lts"].shape
    return np.stack([np.stack([tile_labels(*_bounds_of(mask, b, hm), bq, bk, exact)
                               for hm in range(Hm)]) for b in range(B)])


# ---- FP8 (e4m3) --------------------------------------------------------------
# The e4m3 format of the FP8 path (sign, 4 exponent bits with bias 7, 3 mantissa
# bits; subnormals below 2^-6 in steps of 2^-9; no infinities; 0x7F / 0xFF are
# NaN, so the largest finite value is 448 = 0x7E).  Per-tensor scaling (blog
# "FlashMask技术" §4.2, FP8 compute mode on TMA/tensor-core hardware; the scale
# rule is the plainest one): descale = amax / 448 in fp32 (1 when amax = 0),
# code = e4m3(x / descale), the division in fp32, rounding to nearest even,
# saturating at +-448.

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of e4m3 codes (uint8); NaN codes give NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e4m3_encode(x) -> np.ndarray:
    """Round finite values to the nearest e4m3 code (ties to even), saturating."""
    y = np.asarray(x, dtype=np.float64)
    a = np.abs(y)
    sign = np.where(np.signbit(y), 0x80, 0).astype(np.int64)
    a = np.minimum(a, E4M3_MAX)
    # exponent of the binade holding a (normal range), clamped at the subnormal one
    E = np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64)
    E = np.clip(E, -6, 8)
    step = 2.0 ** (E - 3)                     # spacing of the 8 mantissa steps of the binade
    q = np.rint(a / step)                     # nearest multiple of the spacing, ties to even
    # q in [8, 16] for normal binades (16: carried into the next binade), [0, 8] for E = -6
    val = q * step
    val = np.minimum(val, E4M3_MAX)
    code = np.zeros(a.shape, np.int64)
    nz = val > 0
    Ev = np.floor(np.log2(np.where(nz, val, 1.0))).astype(np.int64)
    sub = nz & (Ev < -6)
    code = np.where(sub, np.rint(val / 2.0 ** -9).astype(np.int64), code)
    nrm = nz & ~sub
    mant = np.rint((val / 2.0 ** Ev - 1.0) * 8).astype(np.int64)
    code = np.where(nrm, ((Ev + 7) << 3) | mant, code)
    return (code | sign).astype(np.uint8)


def quantize_e4m3(x, transpose=False):
    """Per-tensor e4m3 quantization of a [B, H, N, d] tensor: (codes uint8, descale
    float32).  transpose=True returns the codes as [B, H, d, N]."""
    xf = _f32(x)
    amax = np.float32(np.max(np.abs(xf))) if xf.size else np.float32(0)
    descale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    y = (xf / descale).astype(np.float32)               # fp32 division, as the device does it
    codes = e4m3_encode(y)
    if transpose:
        codes = np.ascontiguousarray(np.swapaxes(codes, 2, 3))
    return codes, descale


def forward_fp8(q8, k8, vt8, descale, mask, scale, rows=None):
    """Attention on e4m3 inputs (q8, k8: [B, H, N, d] codes; vt8: [B, H, d, N]),
    exactly: s_ij = scale * dq * dk * sum_c q_ic k_jc on the decoded values,
    O = dv * sum_j P_ij v_j.  descale = (dq, dk, dv)."""
    dq, dk, dv = (float(x) for x in descale)
    qv = e4m3_decode(q8).astype(np.float32)             # e4m3 values are exact in fp32
    kv = e4m3_decode(k8).astype(np.float32)
    vv = np.ascontiguousarray(np.swapaxes(e4m3_decode(vt8), 2, 3)).astype(np.float32)
    O, L = forward(qv, kv, vv, mask, scale * dq * dk, rows=rows)
    return O * dv, L
