"""Thin ctypes binding of liblbq.so (include/lbq.h).

Argument marshalling only: every step of the computation runs in the C++/CUDA
library.  Host entry points take and return numpy arrays; device entry points
take torch CUDA tensors (or raw device addresses) and the current torch
stream.  If the library has not been built this module raises on first use;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblbq.so")

LBQ_F16 = 0
LBQ_F32 = 1
LBQ_KIND_W4 = 0
LBQ_KIND_W2CB = 1
LBQ_FLAG_PDL = 1
LBQ_MAX_GROUP = 32

STATUS = {
    0: "LBQ_OK", 1: "LBQ_ERR_NULL", 2: "LBQ_ERR_SHAPE", 3: "LBQ_ERR_ALIGN", 4: "LBQ_ERR_OUTLIER_IDX",
    5: "LBQ_ERR_BUFFER_TOO_SMALL", 6: "LBQ_ERR_FORMAT", 7: "LBQ_ERR_CUDA", 8: "LBQ_ERR_TIMEOUT",
    9: "LBQ_ERR_VALUE", 10: "LBQ_ERR_UNSUPPORTED",
}

# every symbol include/lbq.h declares
EXPORTS = (
    "lbq_version", "lbq_format_version", "lbq_status_string", "lbq_blob_layout",
    "lbq_w4_packed_bytes", "lbq_w2cb_packed_bytes", "lbq_select_outliers_w4",
    "lbq_select_outliers_impact", "lbq_pack_w4", "lbq_pack_w2cb", "lbq_gemv_w4a16",
    "lbq_gemv_w2cb_outlier", "lbq_gemm_w4a16_smallM", "lbq_gemv_w4a16_ex",
    "lbq_gemv_w2cb_outlier_ex", "lbq_gemm_w4a16_smallM_ex", "lbq_gemm_w2cb_outlier_smallM",
    "lbq_gemm_w2cb_outlier_smallM_ex", "lbq_gemv_grouped", "lbq_gemv_grouped_launches",
    "lbq_selftest_wait_timeout", "lbq_device_error", "lbq_refine_packed_bytes", "lbq_pack_refine",
    "lbq_dequant_host", "lbq_refine_selected_count", "lbq_refine_select", "lbq_refine_apply",
    "lbq_refine_noalloc", "lbq_embed_gather", "lbq_kv_record_bytes", "lbq_kv_quantize", "lbq_kv_dequant",
    "lbq_refine_select_grouped", "lbq_gemv_grouped_refined",
)


class LbqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, STATUS.get(status, "status %d" % status)))


class Layout(ctypes.Structure):
    _fields_ = [("area_offset", ctypes.c_uint64), ("row_block_bytes", ctypes.c_uint64),
                ("record_bytes", ctypes.c_uint64), ("records", ctypes.c_uint64),
                ("outlier_record_bytes", ctypes.c_uint64), ("outlier_records", ctypes.c_uint64),
                ("idx_offset", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64)]


class SelectProblem(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("K", ctypes.c_int64), ("k", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("idx", ctypes.c_void_p), ("refine", ctypes.c_void_p), ("N", ctypes.c_int64)]


class Refinement(ctypes.Structure):
    _fields_ = [("refine", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("n_sel", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class Problem(ctypes.Structure):
    """lbq_problem: one problem of a grouped launch (device pointers)."""
    _fields_ = [("packed", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("n_out", ctypes.c_int32), ("reserved", ctypes.c_int32), ("x", ctypes.c_void_p),
                ("ldx", ctypes.c_int64), ("y", ctypes.c_void_p), ("ldy", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()

c_i64, c_i32, c_u32, c_vp, c_sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t


def lib():
    """Load liblbq.so (once).  Raises ImportError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError("liblbq.so is not built (%s); run `python -c \"import __graft_entry__ as g; "
                              "g.build()\"`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "lbq_version": (ctypes.c_int, []),
            "lbq_format_version": (ctypes.c_int, []),
            "lbq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "lbq_blob_layout": (ctypes.c_int, [ctypes.c_int, c_i64, c_i64, c_i32, ctypes.POINTER(Layout)]),
            "lbq_w4_packed_bytes": (c_sz, [c_i64, c_i64, c_i32]),
            "lbq_w2cb_packed_bytes": (c_sz, [c_i64, c_i64, c_i32]),
            "lbq_select_outliers_w4": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_i32, ctypes.POINTER(c_i32)]),
            "lbq_select_outliers_impact": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_i32, ctypes.c_double,
                                                          c_vp, c_i32, ctypes.POINTER(c_i32)]),
            "lbq_pack_w4": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_i32, c_vp, c_sz]),
            "lbq_pack_w2cb": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_i32, c_vp, c_sz]),
            "lbq_gemv_w4a16": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, ctypes.c_int, c_vp]),
            "lbq_gemv_w2cb_outlier": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, ctypes.c_int, c_vp]),
            "lbq_gemm_w4a16_smallM": (ctypes.c_int, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_i64, c_vp, c_i64,
                                                     ctypes.c_int, c_vp]),
            "lbq_gemv_w4a16_ex": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, ctypes.c_int, c_vp, c_u32]),
            "lbq_gemv_w2cb_outlier_ex": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, ctypes.c_int,
                                                        c_vp, c_u32]),
            "lbq_gemm_w4a16_smallM_ex": (ctypes.c_int, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_i64, c_vp,
                                                        c_i64, ctypes.c_int, c_vp, c_u32]),
            "lbq_gemm_w2cb_outlier_smallM": (ctypes.c_int, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_i64, c_vp,
                                                            c_i64, ctypes.c_int, c_vp]),
            "lbq_gemm_w2cb_outlier_smallM_ex": (ctypes.c_int, [c_vp, c_i32, c_i64, c_i64, c_i32, c_vp, c_i64,
                                                               c_vp, c_i64, ctypes.c_int, c_vp, c_u32]),
            "lbq_gemv_grouped": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(Problem), c_i32, c_i32, ctypes.c_int,
                                                c_vp, c_u32]),
            "lbq_gemv_grouped_launches": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(Problem), c_i32, c_i32,
                                                         ctypes.c_int, ctypes.POINTER(c_i32)]),
            "lbq_selftest_wait_timeout": (ctypes.c_int, [c_u32, c_vp]),
            "lbq_device_error": (ctypes.c_int, [c_vp]),
            "lbq_refine_packed_bytes": (c_sz, [c_i64, c_i64]),
            "lbq_pack_refine": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_sz]),
            "lbq_dequant_host": (ctypes.c_int, [c_vp, c_sz, c_vp]),
            "lbq_refine_selected_count": (c_i64, [c_i64, c_i32]),
            "lbq_refine_select": (ctypes.c_int, [c_vp, c_i64, c_i32, c_vp, c_vp]),
            "lbq_refine_apply": (ctypes.c_int, [c_vp, c_i64, c_i64, c_vp, c_vp, c_i32, c_vp, ctypes.c_int, c_vp]),
            "lbq_refine_noalloc": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, ctypes.c_int, c_vp]),
            "lbq_embed_gather": (ctypes.c_int, [ctypes.c_int, c_vp, c_i64, c_i64, c_i32, c_vp, c_i32, c_vp,
                                                ctypes.c_int, c_vp]),
            "lbq_kv_record_bytes": (c_sz, [c_i64]),
            "lbq_kv_quantize": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_vp]),
            "lbq_kv_dequant": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_vp]),
            "lbq_refine_select_grouped": (ctypes.c_int, [ctypes.POINTER(SelectProblem), c_i32, c_vp]),
            "lbq_gemv_grouped_refined": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(Problem),
                                                        ctypes.POINTER(Refinement), c_i32, ctypes.c_int, c_vp, c_u32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise LbqError(st, where)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ------------------------------------------------------------------ host side

def blob_layout(kind: int, N: int, K: int, n_out: int) -> dict:
    L = Layout()
    _check(lib().lbq_blob_layout(kind, N, K, n_out, ctypes.byref(L)), "lbq_blob_layout")
    return {"area": L.area_offset, "rb_bytes": L.row_block_bytes, "rec_bytes": L.record_bytes, "recs": L.records,
            "out_rec_bytes": L.outlier_record_bytes, "out_recs": L.outlier_records, "idx": L.idx_offset,
            "total": L.total_bytes}


def _as_f32(W) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.float32)
    assert W.ndim == 2
    return W


def _as_idx(idx) -> np.ndarray:
    if idx is None:
        return np.zeros(0, np.int32)
    return np.ascontiguousarray(idx, dtype=np.int32).reshape(-1)


def select_outliers_w4(W) -> np.ndarray:
    W = _as_f32(W)
    N, K = W.shape
    cap = K
    idx = np.zeros(cap, np.int32)
    n = c_i32(0)
    _check(lib().lbq_select_outliers_w4(_ptr(W), N, K, _ptr(idx), cap, ctypes.byref(n)), "lbq_select_outliers_w4")
    return idx[:n.value].copy()


def select_outliers_impact(W, Xprof, frac: float = 0.035) -> np.ndarray:
    W = _as_f32(W)
    N, K = W.shape
    X = np.ascontiguousarray(Xprof, dtype=np.float16).reshape(-1, K)
    idx = np.zeros(K, np.int32)
    n = c_i32(0)
    _check(lib().lbq_select_outliers_impact(_ptr(W), N, K, _ptr(X), X.shape[0], float(frac), _ptr(idx), K,
                                            ctypes.byref(n)), "lbq_select_outliers_impact")
    return idx[:n.value].copy()


def pack_w4(W, idx=None) -> np.ndarray:
    W = _as_f32(W)
    idx = _as_idx(idx)
    N, K = W.shape
    nb = lib().lbq_w4_packed_bytes(N, K, idx.size)
    if nb == 0:
        raise LbqError(2, "lbq_w4_packed_bytes")
    out = np.empty(nb, np.uint8)
    _check(lib().lbq_pack_w4(_ptr(W), N, K, _ptr(idx) if idx.size else None, idx.size, _ptr(out), nb), "lbq_pack_w4")
    return out


def pack_w2cb(W, idx=None) -> np.ndarray:
    W = _as_f32(W)
    idx = _as_idx(idx)
    N, K = W.shape
    nb = lib().lbq_w2cb_packed_bytes(N, K, idx.size)
    if nb == 0:
        raise LbqError(2, "lbq_w2cb_packed_bytes")
    out = np.empty(nb, np.uint8)
    _check(lib().lbq_pack_w2cb(_ptr(W), N, K, _ptr(idx) if idx.size else None, idx.size, _ptr(out), nb),
           "lbq_pack_w2cb")
    return out


def pack_refine(R) -> np.ndarray:
    """Refinement blob of an N x K residual (column records, see include/lbq.h)."""
    R = _as_f32(R)
    N, K = R.shape
    nb = lib().lbq_refine_packed_bytes(N, K)
    if nb == 0:
        raise LbqError(2, "lbq_refine_packed_bytes")
    out = np.empty(nb, np.uint8)
    _check(lib().lbq_pack_refine(_ptr(R), N, K, _ptr(out), nb), "lbq_pack_refine")
    return out


def dequant_host(blob) -> np.ndarray:
    """The N x K FP32 matrix a resident blob applies (outlier columns exact)."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8).reshape(-1)
    # the library's own checks, made before the output is sized from the header:
    # shorter than the header or than the header says -> LBQ_ERR_BUFFER_TOO_SMALL,
    # not a blob of this format -> LBQ_ERR_FORMAT
    kinds = {b"LBQW4G32": LBQ_KIND_W4, b"LBQW2C32": LBQ_KIND_W2CB}
    if blob.size < 128:
        raise LbqError(5, "lbq_dequant_host")
    if bytes(blob[:8]) not in kinds:
        raise LbqError(6, "lbq_dequant_host")
    N = int(blob[16:24].view("<i8")[0])
    K = int(blob[24:32].view("<i8")[0])
    n_out = int(blob[32:36].view("<i4")[0])
    L = Layout()
    if lib().lbq_blob_layout(kinds[bytes(blob[:8])], N, K, n_out, ctypes.byref(L)) != 0:
        raise LbqError(6, "lbq_dequant_host")
    if L.total_bytes > blob.size:
        raise LbqError(5, "lbq_dequant_host")
    out = np.empty((N, K), np.float32)
    _check(lib().lbq_dequant_host(_ptr(blob), blob.size, _ptr(out)), "lbq_dequant_host")
    return out


def refine_selected_count(K: int, k: int) -> int:
    return int(lib().lbq_refine_selected_count(K, k))


# ---------------------------------------------------------------- device side

def _dev_ptr(t) -> int:
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device entry points take CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ydtype(y) -> int:
    import torch
    if y.dtype == torch.float16:
        return LBQ_F16
    if y.dtype == torch.float32:
        return LBQ_F32
    raise ValueError("y must be float16 or float32")


def gemv_w4a16(packed, N: int, K: int, n_out: int, x, y, stream=None, pdl: bool = False, y_dtype: int | None = None):
    yd = _ydtype(y) if y_dtype is None else y_dtype
    _check(lib().lbq_gemv_w4a16_ex(_dev_ptr(packed), N, K, n_out, _dev_ptr(x), _dev_ptr(y), yd, _stream(stream),
                                   LBQ_FLAG_PDL if pdl else 0), "lbq_gemv_w4a16")


def gemv_w2cb_outlier(packed, N: int, K: int, n_out: int, x, y, stream=None, pdl: bool = False,
                      y_dtype: int | None = None):
    yd = _ydtype(y) if y_dtype is None else y_dtype
    _check(lib().lbq_gemv_w2cb_outlier_ex(_dev_ptr(packed), N, K, n_out, _dev_ptr(x), _dev_ptr(y), yd,
                                          _stream(stream), LBQ_FLAG_PDL if pdl else 0), "lbq_gemv_w2cb_outlier")


def gemm_w4a16_smallM(packed, M: int, N: int, K: int, n_out: int, X, ldx: int, Y, ldy: int, stream=None,
                      pdl: bool = False, y_dtype: int | None = None):
    yd = _ydtype(Y) if y_dtype is None else y_dtype
    _check(lib().lbq_gemm_w4a16_smallM_ex(_dev_ptr(packed), M, N, K, n_out, _dev_ptr(X), ldx, _dev_ptr(Y), ldy, yd,
                                          _stream(stream), LBQ_FLAG_PDL if pdl else 0), "lbq_gemm_w4a16_smallM")


def gemm_w2cb_outlier_smallM(packed, M: int, N: int, K: int, n_out: int, X, ldx: int, Y, ldy: int, stream=None,
                             pdl: bool = False, y_dtype: int | None = None):
    yd = _ydtype(Y) if y_dtype is None else y_dtype
    _check(lib().lbq_gemm_w2cb_outlier_smallM_ex(_dev_ptr(packed), M, N, K, n_out, _dev_ptr(X), ldx, _dev_ptr(Y),
                                                 ldy, yd, _stream(stream), LBQ_FLAG_PDL if pdl else 0),
           "lbq_gemm_w2cb_outlier_smallM")


def refine_select(x, K: int, k: int, idx, stream=None):
    """S(x) of a device FP16 vector into the device int32 buffer idx."""
    _check(lib().lbq_refine_select(_dev_ptr(x), K, k, _dev_ptr(idx), _stream(stream)), "lbq_refine_select")


def refine_apply(refine, N: int, K: int, x, idx, n_sel: int, y, stream=None, y_dtype: int | None = None):
    """y += sum over the n_sel selected channels of x_i C[:, i] (device buffers)."""
    yd = _ydtype(y) if y_dtype is None else y_dtype
    _check(lib().lbq_refine_apply(_dev_ptr(refine), N, K, _dev_ptr(x), _dev_ptr(idx) if n_sel else None, n_sel,
                                  _dev_ptr(y), yd, _stream(stream)), "lbq_refine_apply")


def refine_select_grouped(problems, stream=None):
    """Several selections in one launch.  problems: sequence of (x, K, k, idx) or
    (x, K, k, idx, refine, N) (refine: blob whose chosen columns are prefetched
    into L2); device buffers."""
    arr = (SelectProblem * len(problems))()
    for i, p in enumerate(problems):
        x, K, k, idx = p[:4]
        refine, N = (p[4], p[5]) if len(p) > 4 else (None, 0)
        arr[i] = SelectProblem(_dev_ptr(x), K, k, 0, _dev_ptr(idx), _dev_ptr(refine) if refine is not None else None, N)
    _check(lib().lbq_refine_select_grouped(arr, len(problems), _stream(stream)), "lbq_refine_select_grouped")


def gemv_grouped_refined(kind: int, problems, refinements, stream=None, pdl: bool = False,
                         y_dtype: int | None = None):
    """gemv_grouped (M = 1) with selective refinement in the same kernel.
    refinements: one entry per problem, None or (refine, idx, n_sel) device buffers."""
    arr, yd = _problems(problems, y_dtype)
    ref = (Refinement * len(problems))()
    for i, r in enumerate(refinements):
        if r is not None:
            ref[i] = Refinement(_dev_ptr(r[0]), _dev_ptr(r[1]) if r[2] else None, r[2], 0)
    _check(lib().lbq_gemv_grouped_refined(kind, arr, ref, len(problems), yd, _stream(stream),
                                          LBQ_FLAG_PDL if pdl else 0), "lbq_gemv_grouped_refined")


def refine_noalloc(refine, N: int, K: int, k: int, x, y, stream=None, y_dtype: int | None = None):
    """Select + apply with the library's static index scratch (calls must not overlap)."""
    yd = _ydtype(y) if y_dtype is None else y_dtype
    _check(lib().lbq_refine_noalloc(_dev_ptr(refine), N, K, k, _dev_ptr(x), _dev_ptr(y), yd, _stream(stream)),
           "lbq_refine_noalloc")


def embed_gather(kind: int, packed, V: int, D: int, n_out: int, ids, out, stream=None, out_dtype: int | None = None):
    """Rows ids of a packed V x D table into out (T x D), dequantised (device buffers)."""
    od = _ydtype(out) if out_dtype is None else out_dtype
    T = ids.numel() if hasattr(ids, "numel") else int(np.asarray(ids).size)
    _check(lib().lbq_embed_gather(kind, _dev_ptr(packed), V, D, n_out, _dev_ptr(ids) if T else None, T,
                                  _dev_ptr(out) if T else None, od, _stream(stream)), "lbq_embed_gather")


def kv_record_bytes(width: int) -> int:
    return int(lib().lbq_kv_record_bytes(width))


def kv_quantize(x, rows: int, width: int, cache, first_row: int, ldx: int | None = None, stream=None):
    """Quantise rows of FP16 states (device) into records of the device cache."""
    _check(lib().lbq_kv_quantize(_dev_ptr(x), ldx or width, rows, width, _dev_ptr(cache), first_row,
                                 _stream(stream)), "lbq_kv_quantize")


def kv_dequant(cache, first_row: int, rows: int, width: int, out, ldo: int | None = None, stream=None):
    """Read cache records back as FP16 rows (device)."""
    _check(lib().lbq_kv_dequant(_dev_ptr(cache), first_row, rows, width, _dev_ptr(out), ldo or width,
                                _stream(stream)), "lbq_kv_dequant")


def _problems(problems, y_dtype):
    arr = (Problem * len(problems))()
    yd = y_dtype
    for i, p in enumerate(problems):
        if len(p) == 6:
            packed, N, K, n_out, x, y = p
            ldx, ldy = K, N
        else:
            packed, N, K, n_out, x, ldx, y, ldy = p
        if yd is None:
            yd = _ydtype(y)
        arr[i] = Problem(_dev_ptr(packed), N, K, n_out, 0, _dev_ptr(x), ldx, _dev_ptr(y), ldy)
    return arr, yd


def gemv_grouped(kind: int, problems, M: int = 1, stream=None, pdl: bool = False, y_dtype: int | None = None):
    """One launch over independent problems.  problems: sequence of
    (packed, N, K, n_out, x, y) or (packed, N, K, n_out, x, ldx, y, ldy); x / y
    are CUDA tensors or device addresses; ldx defaults to K, ldy to N."""
    arr, yd = _problems(problems, y_dtype)
    _check(lib().lbq_gemv_grouped(kind, arr, len(problems), M, yd, _stream(stream), LBQ_FLAG_PDL if pdl else 0),
           "lbq_gemv_grouped")


def gemv_grouped_launches(kind: int, problems, M: int = 1, y_dtype: int | None = None) -> int:
    """Kernels gemv_grouped would launch for the same arguments."""
    arr, yd = _problems(problems, y_dtype)
    n = c_i32(0)
    _check(lib().lbq_gemv_grouped_launches(kind, arr, len(problems), M, yd, ctypes.byref(n)),
           "lbq_gemv_grouped_launches")
    return n.value


def selftest_wait_timeout(limit_us: int, stream=None):
    _check(lib().lbq_selftest_wait_timeout(limit_us, _stream(stream)), "lbq_selftest_wait_timeout")


def device_error(stream=None) -> int:
    return int(lib().lbq_device_error(_stream(stream)))
