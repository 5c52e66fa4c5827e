"""Python binding of ``libfm.so`` (include/fm.h): the same entry points, with
torch tensors and numpy arrays marshalled to pointers.  Every step of the
computation runs inside the library; this module only checks types,
allocates caller-owned buffers with torch where a helper says so, and
forwards.  Importing it fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

# FM_LIBRARY selects another build of the same library (the FM_DEBUG build of
# build.build(debug=True)); by default the in-tree release build.
_LIB_PATH = os.environ.get("FM_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libfm.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
_lib = ctypes.CDLL(_LIB_PATH)

FM_OK, FM_ERR_INVALID_ARG, FM_ERR_UNSUPPORTED, FM_ERR_UNREPRESENTABLE = 0, 1, 2, 3
FM_ERR_BAD_BOUNDS, FM_ERR_PLAN_MISMATCH, FM_ERR_WORKSPACE, FM_ERR_CUDA, FM_ERR_TIMEOUT = 4, 5, 6, 7, 8
FM_ERR_DEBUG_CHECK = 9
FM_TILE_SKIP, FM_TILE_FULL, FM_TILE_PARTIAL = 0, 1, 2
FM_DT_BF16, FM_DT_F32 = 0, 1
FM_FLAG_PRECISE = 1
KERNEL_NAMES = ["classify_minmax", "classify_lists", "fwd", "bwd_pre", "bwd", "bwd_post",
                "classify_order", "fp8_amax", "fp8_convert"]

EXPORTED = ["fm_status_string", "fm_abi_version", "fm_mask_from_rows", "fm_mask_from_row_intervals",
            "fm_plan_bytes", "fm_tile_classify", "fm_fwd_workspace_bytes", "fm_attn_fwd", "fm_bwd_workspace_bytes",
            "fm_attn_bwd", "fm_profile_begin", "fm_profile_end", "fm_selftest_wait_timeout",
            "fm_attn_bwd_noalloc", "fm_step_graph_create", "fm_step_graph_launch", "fm_step_graph_destroy",
            "fm_plan_bytes_rows", "fm_tile_classify_rows", "fm_attn_fwd_rows", "fm_attn_bwd_rows",
            "fm_quantize_fp8", "fm_attn_fwd_fp8", "fm_debug_wait_test", "fm_bounds_compressed_bytes",
            "fm_bounds_compress", "fm_bounds_decompress"]
# Size of the library's built-in backward workspace (FM_NOALLOC_SCRATCH_BYTES in fm.h).
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class FmError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        super().__init__(f"{where}: {fm_status_string(code)} ({code})")


class Bounds(ctypes.Structure):
    _fields_ = [("lts", ctypes.c_void_p), ("lte", ctypes.c_void_p), ("uts", ctypes.c_void_p),
                ("ute", ctypes.c_void_p), ("B", ctypes.c_int32), ("Hm", ctypes.c_int32),
                ("N", ctypes.c_int32)]


class StepArgs(ctypes.Structure):
    """fm_step_args of include/fm.h (field order and C layout)."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("dO", ctypes.c_void_p), ("mask", Bounds), ("plan", ctypes.c_void_p),
                ("plan_bytes", ctypes.c_size_t), ("o", ctypes.c_void_p), ("o_dtype", ctypes.c_int),
                ("lse", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p),
                ("dv", ctypes.c_void_p), ("grad_dtype", ctypes.c_int), ("ws", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t), ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("scale", ctypes.c_float), ("flags", ctypes.c_int),
                ("dev_status", ctypes.c_void_p)]


class KernelTime(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("ms", ctypes.c_float)]


_P, _I, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_lib.fm_status_string.restype = ctypes.c_char_p
_lib.fm_status_string.argtypes = [_I]
_lib.fm_abi_version.restype = _I
_lib.fm_mask_from_rows.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P]
_lib.fm_mask_from_row_intervals.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P]
_lib.fm_plan_bytes.restype = _SZ
_lib.fm_plan_bytes.argtypes = [_I, _I, _I, _I, _I]
_lib.fm_tile_classify.argtypes = [Bounds, _I, _I, _P, _SZ, _P, _P, _P]
_lib.fm_fwd_workspace_bytes.restype = _SZ
_lib.fm_fwd_workspace_bytes.argtypes = [_I, _I, _I, _I]
_lib.fm_attn_fwd.argtypes = [_P, _P, _P, Bounds, _P, _I, _I, _I, _I, _F, _P, _I, _P, _P, _SZ, _I, _P, _P]
_lib.fm_bwd_workspace_bytes.restype = _SZ
_lib.fm_bwd_workspace_bytes.argtypes = [_I, _I, _I, _I]
_lib.fm_attn_bwd.argtypes = [_P, _P, _P, _P, _I, _P, _P, Bounds, _P, _I, _I, _I, _I, _F, _P, _P, _P,
                             _I, _I, _P, _SZ, _P, _P]
_lib.fm_attn_bwd_noalloc.argtypes = [_P, _P, _P, _P, _I, _P, _P, Bounds, _P, _I, _I, _I, _I, _F, _P,
                                     _P, _P, _I, _I, _P, _P]
_lib.fm_profile_begin.argtypes = []
_lib.fm_profile_end.restype = _I
_lib.fm_profile_end.argtypes = [_P, _I]
_lib.fm_selftest_wait_timeout.argtypes = [ctypes.c_longlong, _P, _P]
_lib.fm_debug_wait_test.argtypes = [ctypes.c_int, ctypes.c_longlong]
_lib.fm_bounds_compressed_bytes.argtypes = [_P, _P, _P, _P, _I, _I, _I]
_lib.fm_bounds_compressed_bytes.restype = _SZ
_lib.fm_bounds_compress.argtypes = [_P, _P, _P, _P, _I, _I, _I, _P, _SZ]
_lib.fm_bounds_decompress.argtypes = [_P, _SZ, Bounds, _P, _P]
_lib.fm_plan_bytes_rows.restype = _SZ
_lib.fm_plan_bytes_rows.argtypes = [_I, _I, _I, _I, _I, _I, _I]
_lib.fm_tile_classify_rows.argtypes = [Bounds, _I, _I, _I, _I, _P, _SZ, _P, _P, _P]
_lib.fm_attn_fwd_rows.argtypes = [_P, _P, _P, Bounds, _P, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P, _P, _SZ, _I,
                                  _P, _P]
_lib.fm_attn_bwd_rows.argtypes = [_P, _P, _P, _P, _I, _P, _P, Bounds, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                  _P, _I, _I, _P, _SZ, _P, _P]
_lib.fm_quantize_fp8.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _P]
_lib.fm_attn_fwd_fp8.argtypes = [_P, _P, _P, _P, Bounds, _P, _I, _I, _I, _I, _F, _P, _I, _P, _P, _P]
_lib.fm_step_graph_create.argtypes = [ctypes.POINTER(StepArgs), ctypes.POINTER(ctypes.c_void_p)]
_lib.fm_step_graph_launch.argtypes = [_P, _P]
_lib.fm_step_graph_destroy.argtypes = [_P]


def _check(code, where):
    if code != FM_OK:
        raise FmError(code, where)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _dt(t):
    if t.dtype == torch.bfloat16:
        return FM_DT_BF16
    if t.dtype == torch.float32:
        return FM_DT_F32
    raise TypeError(f"unsupported output dtype {t.dtype}")


def fm_status_string(code: int) -> str:
    return _lib.fm_status_string(int(code)).decode()


def fm_abi_version() -> int:
    return _lib.fm_abi_version()


def make_bounds(lts, lte, uts, ute) -> Bounds:
    """fm_bounds from four device int32 tensors [B, Hm, N]."""
    for n, t in zip(("lts", "lte", "uts", "ute"), (lts, lte, uts, ute)):
        _dev(t, torch.int32, n)
        if t.dim() != 3 or t.shape != lts.shape:
            raise ValueError(f"{n} must be [B, Hm, N] like lts")
    B, Hm, N = lts.shape
    return Bounds(lts.data_ptr(), lte.data_ptr(), uts.data_ptr(), ute.data_ptr(), B, Hm, N)


def fm_mask_from_rows(cs, ce):
    """Host conversion of row intervals (int32 [B, Hm, N]) to column bounds."""
    cs = np.ascontiguousarray(cs, dtype=np.int32)
    ce = np.ascontiguousarray(ce, dtype=np.int32)
    if cs.ndim != 3 or cs.shape != ce.shape:
        raise ValueError("cs and ce must be int32 [B, Hm, N]")
    B, Hm, N = cs.shape
    out = [np.empty_like(cs) for _ in range(4)]
    code = _lib.fm_mask_from_rows(cs.ctypes.data, ce.ctypes.data, B, Hm, N,
                                  *[o.ctypes.data for o in out])
    _check(code, "fm_mask_from_rows")
    return tuple(out)


def fm_mask_from_row_intervals(starts, ends):
    """Host conversion of K inclusive intervals per row (int32 [B, Hm, N, K];
    start > end marks an unused slot) to column bounds [B, Hm, N]."""
    starts = np.ascontiguousarray(starts, dtype=np.int32)
    ends = np.ascontiguousarray(ends, dtype=np.int32)
    if starts.ndim != 4 or starts.shape != ends.shape:
        raise ValueError("starts and ends must be int32 [B, Hm, N, K]")
    B, Hm, N, K = starts.shape
    out = [np.empty((B, Hm, N), np.int32) for _ in range(4)]
    code = _lib.fm_mask_from_row_intervals(starts.ctypes.data, ends.ctypes.data, K, B, Hm, N,
                                           *[o.ctypes.data for o in out])
    _check(code, "fm_mask_from_row_intervals")
    return tuple(out)


def fm_plan_bytes(B, Hm, N, bq=128, bk=128) -> int:
    return int(_lib.fm_plan_bytes(B, Hm, N, bq, bk))


def fm_tile_classify(bounds: Bounds, plan, dev_status, bq=128, bk=128, labels=None, stream=None):
    _dev(plan, torch.uint8, "plan")
    _dev(dev_status, torch.int32, "dev_status")
    if labels is not None:
        _dev(labels, torch.uint8, "labels")
    code = _lib.fm_tile_classify(bounds, bq, bk, _ptr(plan), plan.numel(), _ptr(labels),
                                 _ptr(dev_status), _stream(stream))
    _check(code, "fm_tile_classify")


def fm_fwd_workspace_bytes(B, H, N, d) -> int:
    return int(_lib.fm_fwd_workspace_bytes(B, H, N, d))


def fm_attn_fwd(q, k, v, bounds: Bounds, plan, scale, o, lse, dev_status, ws=None, stream=None,
                flags=0):
    for n, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, torch.bfloat16, n)
    B, H, N, d = q.shape
    if k.shape != q.shape or v.shape != q.shape or o.shape != q.shape:
        raise ValueError("q, k, v, o must share the shape [B, H, N, d]")
    _dev(o, o.dtype, "o")
    _dev(lse, torch.float32, "lse")
    _dev(plan, torch.uint8, "plan")
    _dev(dev_status, torch.int32, "dev_status")
    code = _lib.fm_attn_fwd(_ptr(q), _ptr(k), _ptr(v), bounds, _ptr(plan), B, H, N, d, float(scale),
                            _ptr(o), _dt(o), _ptr(lse), _ptr(ws), 0 if ws is None else ws.numel(),
                            int(flags), _ptr(dev_status), _stream(stream))
    _check(code, "fm_attn_fwd")


def fm_bwd_workspace_bytes(B, H, N, d) -> int:
    return int(_lib.fm_bwd_workspace_bytes(B, H, N, d))


def fm_attn_bwd(q, k, v, o, lse, dO, bounds: Bounds, plan, scale, dq, dk, dv, ws, dev_status,
                stream=None, flags=0):
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _dev(t, torch.bfloat16, n)
    B, H, N, d = q.shape
    for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        _dev(t, t.dtype, n)
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q")
    if not (dq.dtype == dk.dtype == dv.dtype):
        raise TypeError("dq, dk, dv must share one dtype")
    _dev(lse, torch.float32, "lse")
    _dev(ws, torch.uint8, "ws")
    code = _lib.fm_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o), _ptr(lse), _ptr(dO), bounds,
                            _ptr(plan), B, H, N, d, float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                            _dt(dq), int(flags), _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream))
    _check(code, "fm_attn_bwd")


def fm_attn_bwd_noalloc(q, k, v, o, lse, dO, bounds: Bounds, plan, scale, dq, dk, dv, dev_status,
                        stream=None, flags=0):
    """fm_attn_bwd without a caller workspace: for callers that cannot
    allocate device memory; the library's fixed built-in array is used
    instead (see fm.h for the size limit and the rules on overlapping calls)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _dev(t, torch.bfloat16, n)
    B, H, N, d = q.shape
    for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        _dev(t, t.dtype, n)
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q")
    if not (dq.dtype == dk.dtype == dv.dtype):
        raise TypeError("dq, dk, dv must share one dtype")
    _dev(lse, torch.float32, "lse")
    code = _lib.fm_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o), _ptr(lse), _ptr(dO),
                                    bounds, _ptr(plan), B, H, N, d, float(scale), _ptr(dq), _ptr(dk),
                                    _ptr(dv), _dt(dq), int(flags), _ptr(dev_status), _stream(stream))
    _check(code, "fm_attn_bwd_noalloc")


def fm_profile_begin():
    _check(_lib.fm_profile_begin(), "fm_profile_begin")


def fm_profile_end(max_entries=4096):
    """[(kernel name, ms)] of every launch since fm_profile_begin."""
    buf = (KernelTime * max_entries)()
    n = _lib.fm_profile_end(buf, max_entries)
    if n < 0:
        raise FmError(FM_ERR_CUDA, "fm_profile_end")
    return [(KERNEL_NAMES[buf[i].kernel], float(buf[i].ms)) for i in range(n)]


def fm_bounds_compress(lts, lte, uts, ute):
    """Host int32 [B, Hm, N] bounds -> the compressed form (numpy uint8)."""
    arr = [np.ascontiguousarray(x, dtype=np.int32) for x in (lts, lte, uts, ute)]
    if not all(a.shape == arr[0].shape and a.ndim == 3 for a in arr):
        raise ValueError("bounds must be int32 [B, Hm, N], all of one shape")
    B, Hm, N = arr[0].shape
    p = [a.ctypes.data_as(ctypes.c_void_p) for a in arr]
    n = _lib.fm_bounds_compressed_bytes(*p, B, Hm, N)
    if n == 0:
        raise FmError(FM_ERR_INVALID_ARG, "fm_bounds_compressed_bytes")
    out = np.zeros(n, np.uint8)
    _check(_lib.fm_bounds_compress(*p, B, Hm, N, out.ctypes.data_as(ctypes.c_void_p), n), "fm_bounds_compress")
    return out


def fm_bounds_decompress(cbounds, bounds: Bounds, dev_status, stream=None):
    """Device uint8 compressed buffer -> the device int32 arrays of `bounds`."""
    _dev(cbounds, torch.uint8, "cbounds")
    _dev(dev_status, torch.int32, "dev_status")
    _check(_lib.fm_bounds_decompress(_ptr(cbounds), cbounds.numel(), bounds, _ptr(dev_status), _stream(stream)),
           "fm_bounds_decompress")


def fm_debug_wait_test(kernel, limit_cycles):
    """Test hook: the next forward (kernel=0) or backward (kernel=1) launch runs
    with every device-side wait bounded by limit_cycles and its first CTA
    withholds one tile load, so it must end with FM_ERR_TIMEOUT in dev_status."""
    _check(_lib.fm_debug_wait_test(int(kernel), int(limit_cycles)), "fm_debug_wait_test")


def fm_selftest_wait_timeout(limit_cycles, dev_status, stream=None):
    _dev(dev_status, torch.int32, "dev_status")
    _check(_lib.fm_selftest_wait_timeout(int(limit_cycles), _ptr(dev_status), _stream(stream)),
           "fm_selftest_wait_timeout")


# ---------------------------------------------------------------------------
# Convenience layer: allocates the caller-owned buffers with torch and calls
# the entry points above.
# ---------------------------------------------------------------------------
def fm_plan_bytes_rows(B, Hm, N, q_row0, Nq, bq=128, bk=128) -> int:
    return int(_lib.fm_plan_bytes_rows(B, Hm, N, q_row0, Nq, bq, bk))


def fm_tile_classify_rows(bounds: Bounds, q_row0, Nq, plan, dev_status, bq=128, bk=128, labels=None, stream=None):
    _dev(plan, torch.uint8, "plan")
    _dev(dev_status, torch.int32, "dev_status")
    if labels is not None:
        _dev(labels, torch.uint8, "labels")
    code = _lib.fm_tile_classify_rows(bounds, int(q_row0), int(Nq), bq, bk, _ptr(plan), plan.numel(),
                                      _ptr(labels), _ptr(dev_status), _stream(stream))
    _check(code, "fm_tile_classify_rows")


def fm_attn_fwd_rows(q, k, v, bounds: Bounds, plan, q_row0, scale, o, lse, dev_status, stream=None, flags=0):
    """Q rows [q_row0, q_row0 + Nq) (q: [B, H, Nq, d]) against all N keys (k, v: [B, H, N, d])."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, torch.bfloat16, n)
    B, H, Nq, d = q.shape
    N = k.shape[2]
    if k.shape != (B, H, N, d) or v.shape != k.shape or o.shape != q.shape:
        raise ValueError("q, o: [B, H, Nq, d]; k, v: [B, H, N, d]")
    _dev(o, o.dtype, "o")
    _dev(lse, torch.float32, "lse")
    _dev(plan, torch.uint8, "plan")
    _dev(dev_status, torch.int32, "dev_status")
    code = _lib.fm_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), bounds, _ptr(plan), B, H, N, int(q_row0), Nq, d,
                                 float(scale), _ptr(o), _dt(o), _ptr(lse), None, 0, int(flags), _ptr(dev_status),
                                 _stream(stream))
    _check(code, "fm_attn_fwd_rows")


def fm_attn_bwd_rows(q, k, v, o, lse, dO, bounds: Bounds, plan, q_row0, scale, dq, dk, dv, ws, dev_status,
                     stream=None, flags=0):
    """dQ of the window's rows; dK, dV receive the window's contribution (all N rows)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _dev(t, torch.bfloat16, n)
    B, H, Nq, d = q.shape
    N = k.shape[2]
    for n, t, shp in (("o", o, q.shape), ("dq", dq, q.shape), ("dO", dO, q.shape), ("dk", dk, k.shape),
                      ("dv", dv, k.shape)):
        _dev(t, t.dtype, n)
        if t.shape != shp:
            raise ValueError(f"{n} has the wrong shape")
    if not (dq.dtype == dk.dtype == dv.dtype):
        raise TypeError("dq, dk, dv must share one dtype")
    _dev(lse, torch.float32, "lse")
    _dev(ws, torch.uint8, "ws")
    code = _lib.fm_attn_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o), _ptr(lse), _ptr(dO), bounds,
                                 _ptr(plan), B, H, N, int(q_row0), Nq, d, float(scale), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _dt(dq), int(flags), _ptr(ws), ws.numel(), _ptr(dev_status),
                                 _stream(stream))
    _check(code, "fm_attn_bwd_rows")


def fm_quantize_fp8(x, transpose=False, out=None, descale=None, stream=None):
    """Per-tensor e4m3 codes (uint8) of a bf16 [B, H, N, d] tensor and its
    descale (device float32 [1]); transpose=True gives the [B, H, d, N] layout."""
    _dev(x, torch.bfloat16, "x")
    B, H, N, d = x.shape
    shape = (B, H, d, N) if transpose else (B, H, N, d)
    out = torch.empty(shape, dtype=torch.uint8, device=x.device) if out is None else _dev(out, torch.uint8, "out")
    descale = torch.empty(1, dtype=torch.float32, device=x.device) if descale is None else descale
    _dev(descale, torch.float32, "descale")
    _check(_lib.fm_quantize_fp8(_ptr(x), B, H, N, d, int(bool(transpose)), _ptr(out), _ptr(descale),
                                _stream(stream)), "fm_quantize_fp8")
    return out, descale


def fm_attn_fwd_fp8(q8, k8, vt8, descale, bounds: Bounds, plan, scale, o, lse, dev_status, stream=None):
    """Forward on e4m3 q8, k8 [B, H, N, d] and vt8 [B, H, d, N]; descale: device
    float32 [3] (Q, K, V)."""
    for n, t in (("q8", q8), ("k8", k8), ("vt8", vt8)):
        _dev(t, torch.uint8, n)
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or vt8.shape != (B, H, d, N) or o.shape != q8.shape:
        raise ValueError("q8, k8, o: [B, H, N, d]; vt8: [B, H, d, N]")
    _dev(descale, torch.float32, "descale")
    if descale.numel() != 3:
        raise ValueError("descale holds the Q, K and V descales")
    _dev(o, o.dtype, "o")
    _dev(lse, torch.float32, "lse")
    _dev(plan, torch.uint8, "plan")
    _dev(dev_status, torch.int32, "dev_status")
    code = _lib.fm_attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(descale), bounds, _ptr(plan), B, H, N, d,
                                float(scale), _ptr(o), _dt(o), _ptr(lse), _ptr(dev_status), _stream(stream))
    _check(code, "fm_attn_fwd_fp8")


def fm_step_graph_create(q, k, v, dO, bounds: Bounds, plan, scale, o, lse, dev_status, dq=None, dk=None,
                         dv=None, ws=None, flags=0):
    """Capture classify + forward (+ backward when dO is given) for these
    buffers; returns the opaque handle (an int)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, torch.bfloat16, n)
    B, H, N, d = q.shape
    a = StepArgs()
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.dO = None if dO is None else _dev(dO, torch.bfloat16, "dO").data_ptr()
    a.mask = bounds
    a.plan, a.plan_bytes = _dev(plan, torch.uint8, "plan").data_ptr(), plan.numel()
    a.o, a.o_dtype = _dev(o, o.dtype, "o").data_ptr(), _dt(o)
    a.lse = _dev(lse, torch.float32, "lse").data_ptr()
    if dO is not None:
        if not (dq.dtype == dk.dtype == dv.dtype):
            raise TypeError("dq, dk, dv must share one dtype")
        a.dq, a.dk, a.dv = (_dev(t, t.dtype, n).data_ptr() for n, t in (("dq", dq), ("dk", dk), ("dv", dv)))
        a.grad_dtype = _dt(dq)
        a.ws, a.ws_bytes = _dev(ws, torch.uint8, "ws").data_ptr(), ws.numel()
    a.B, a.H, a.N, a.d = B, H, N, d
    a.scale, a.flags = float(scale), int(flags)
    a.dev_status = _dev(dev_status, torch.int32, "dev_status").data_ptr()
    h = ctypes.c_void_p()
    _check(_lib.fm_step_graph_create(ctypes.byref(a), ctypes.byref(h)), "fm_step_graph_create")
    return h.value


def fm_step_graph_launch(graph, stream=None):
    _check(_lib.fm_step_graph_launch(ctypes.c_void_p(graph), _stream(stream)), "fm_step_graph_launch")


def fm_step_graph_destroy(graph):
    _check(_lib.fm_step_graph_destroy(ctypes.c_void_p(graph)), "fm_step_graph_destroy")


class StepGraph:
    """One captured step over fixed buffers (keeps them referenced while the
    graph lives); refill the inputs in place and call launch()."""

    def __init__(self, q, k, v, dO, att: "MaskedAttention", scale, o, lse, dq=None, dk=None, dv=None, ws=None,
                 flags=0):
        self._keep = (q, k, v, dO, att, o, lse, dq, dk, dv, ws)
        self.handle = fm_step_graph_create(q, k, v, dO, att.bounds, att.plan, scale, o, lse, att.status,
                                           dq, dk, dv, ws, flags)

    def launch(self, stream=None):
        fm_step_graph_launch(self.handle, stream)

    def close(self):
        if self.handle is not None:
            fm_step_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MaskedAttention:
    """Holds the device bounds, plan and status word of one mask."""

    def __init__(self, lts, lte, uts, ute, device="cuda", stream=None):
        t = [torch.as_tensor(np.ascontiguousarray(x), dtype=torch.int32).to(device) for x in
             (lts, lte, uts, ute)]
        self.lts, self.lte, self.uts, self.ute = t
        self.bounds = make_bounds(*t)
        self.B, self.Hm, self.N = self.lts.shape
        self.plan = torch.empty(fm_plan_bytes(self.B, self.Hm, self.N), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.stream = stream
        fm_tile_classify(self.bounds, self.plan, self.status, stream=stream)

    def labels(self, bq=128, bk=128):
        """Labels uint8 [B, Hm, n_q, n_k] (a separate plan of tile size bq x bk)."""
        n_q, n_k = -(-self.N // bq), -(-self.N // bk)
        out = torch.empty((self.B, self.Hm, n_q, n_k), dtype=torch.uint8, device=self.plan.device)
        plan = torch.empty(fm_plan_bytes(self.B, self.Hm, self.N, bq, bk), dtype=torch.uint8,
                           device=self.plan.device)
        fm_tile_classify(self.bounds, plan, self.status, bq, bk, labels=out, stream=self.stream)
        return out

    def forward(self, q, k, v, scale=None, o_dtype=torch.bfloat16, flags=0):
        B, H, N, d = q.shape
        scale = 1.0 / d ** 0.5 if scale is None else scale
        o = torch.empty(q.shape, dtype=o_dtype, device=q.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        fm_attn_fwd(q, k, v, self.bounds, self.plan, scale, o, lse, self.status, stream=self.stream,
                    flags=flags)
        return o, lse

    def backward(self, q, k, v, o, lse, dO, scale=None, grad_dtype=torch.float32, ws=None, flags=0):
        B, H, N, d = q.shape
        scale = 1.0 / d ** 0.5 if scale is None else scale
        if ws is None:
            ws = torch.empty(fm_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
        dq, dk, dv = (torch.empty(q.shape, dtype=grad_dtype, device=q.device) for _ in range(3))
        fm_attn_bwd(q, k, v, o, lse, dO, self.bounds, self.plan, scale, dq, dk, dv, ws, self.status,
                    stream=self.stream, flags=flags)
        return dq, dk, dv

    def check_status(self):
        code = int(self.status.item())
        if code != 0:
            raise FmError(code, "device")
