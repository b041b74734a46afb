"""CPU oracle for the sparse-attention prefill indexer (fp64, exact top-k).

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never imports, links or calls it, and it shares no code with the library.

The arithmetic lives in ``oracle.c`` (plain C11, compiled here with gcc); this
module only builds it and marshals numpy arrays.  What it computes is stated in
the header of ``oracle.c``:

* ``scores_row``      s[r,j] = k_scale[j] * sum_h w[r,h] * ReLU(q[r,h,:].k[j,:])
                      in fp64 over the visible keys of row r.
* ``select_row``      top-k by (score desc, key index asc), returned as
                      ascending row-relative indices padded with -1.
* ``score_topk``      both, for a list of rows, on host threads.
* ``topk_from_scores``the selection applied to given fp32 scores.
* ``page_transform``  row-relative positions -> physical KV slots of a paged
                      cache (page size P): table[t, p // P] * P + p % P, -1 kept.

Input formats: bf16, e4m3 and MXFP4 (e2m1 elements packed two per byte with
one e8m0 scale per 32 elements; ``q_sf`` / ``k_sf`` on the input set).

``IDX_ORACLE_LIB`` names an already built oracle library to load instead of
building ``oracle.c``; the mutation tests use it to run the pins against
copies of the oracle with planted mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, E4M3, MXFP4 = 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, no GPU)."""
    override = os.environ.get("IDX_ORACLE_LIB")
    if override:
        return override
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O3", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_longlong
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint32]
        lib.orc_e4m3_to_f64.restype = ctypes.c_double
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint32]
        lib.orc_bf16_to_f64.restype = ctypes.c_double
        lib.orc_e2m1_to_f64.argtypes = [ctypes.c_uint32]
        lib.orc_e2m1_to_f64.restype = ctypes.c_double
        lib.orc_e8m0_to_f64.argtypes = [ctypes.c_uint32]
        lib.orc_e8m0_to_f64.restype = ctypes.c_double
        lib.orc_scores_row.argtypes = [P, P, P, P, i32, P, P, i32, i32, i64, i64, i64, P]
        lib.orc_scores_row.restype = i32
        lib.orc_select_row.argtypes = [P, i64, i32, P]
        lib.orc_select_row.restype = i32
        lib.orc_score_topk.argtypes = [P, P, P, P, i32, P, P, P, P, i32, i32, P, i32, i32, P,
                                       P, i64, i32]
        lib.orc_score_topk.restype = i32
        lib.orc_topk_from_scores.argtypes = [P, i64, P, P, P, i32, i32, P, i32]
        lib.orc_topk_from_scores.restype = i32
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _np(x, dtype=None):
    """torch tensor or array -> C-contiguous numpy array (raw bytes kept)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            elif t.dtype == torch.float8_e4m3fn:
                t = t.view(torch.uint8)
            x = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if dtype is not None and a.dtype != dtype:
        a = np.ascontiguousarray(a.astype(dtype))
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(q) -> int:
    name = str(getattr(q, "dtype", ""))
    if "bfloat16" in name or name == "int16" or name == "uint16":
        return BF16
    if "float8_e4m3" in name or name == "uint8":
        return E4M3
    raise ValueError(f"unsupported q/k dtype {name}")


def e4m3_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint32).ravel()
    return np.array([lib.orc_e4m3_to_f64(int(v)) for v in c], dtype=np.float64)


def bf16_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint32).ravel()
    return np.array([lib.orc_bf16_to_f64(int(v)) for v in c], dtype=np.float64)


def e2m1_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint32).ravel()
    return np.array([lib.orc_e2m1_to_f64(int(v)) for v in c], dtype=np.float64)


def e8m0_to_f64(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint32).ravel()
    return np.array([lib.orc_e8m0_to_f64(int(v)) for v in c], dtype=np.float64)


class _Indexer:
    """Raw views of an indexer input set (q, k, k_scale, w, ks, ke, and the
    block scales q_sf, k_sf of MXFP4 inputs)."""

    def __init__(self, q, k, k_scale, w, ks, ke, q_sf=None, k_sf=None):
        mx = q_sf is not None or k_sf is not None
        self.dtype = MXFP4 if mx else _dtype_code(q)
        self.q = _np(q, np.uint8 if mx else None)
        self.k = _np(k, np.uint8 if mx else None)
        self.k_scale = _np(k_scale, np.float32)
        self.w = _np(w, np.float32)
        self.ks = _np(ks, np.int32)
        self.ke = _np(ke, np.int32)
        self.rows, self.H, dq = self.q.shape
        self.D = 2 * dq if mx else dq
        if mx:
            self.q_sf = _np(q_sf, np.uint8)
            self.k_sf = _np(k_sf, np.uint8)
            if (self.D % 32 or self.k.shape[1] * 2 != self.D
                    or self.q_sf.shape != (self.rows, self.H, self.D // 32)
                    or self.k_sf.shape != (self.k.shape[0], self.D // 32)):
                raise ValueError("inconsistent MXFP4 input shapes")
        else:
            self.q_sf = self.k_sf = None
        if self.w.shape != (self.rows, self.H) or (not mx and self.k.shape[1] != self.D):
            raise ValueError("inconsistent indexer input shapes")

    def sf_ptrs(self):
        if self.q_sf is None:
            return None, None
        return _ptr(self.q_sf), _ptr(self.k_sf)


def _indexer(inp) -> _Indexer:
    return _Indexer(inp.q, inp.k, inp.k_scale, inp.w, inp.ks, inp.ke,
                    getattr(inp, "q_sf", None), getattr(inp, "k_sf", None))


def scores_row(inp, r: int) -> np.ndarray:
    """fp64 scores of row r over its visible keys (length ke - ks)."""
    X = _indexer(inp) if not isinstance(inp, _Indexer) else inp
    ks, ke = int(X.ks[r]), int(X.ke[r])
    out = np.zeros(max(ke - ks, 0), dtype=np.float64)
    if out.size:
        qsf, ksf = X.sf_ptrs()
        e = _load().orc_scores_row(_ptr(X.q), qsf, _ptr(X.k), ksf, X.dtype, _ptr(X.k_scale),
                                   _ptr(X.w), X.H, X.D, r, ks, ke, _ptr(out))
        if e:
            raise MemoryError("oracle scores_row failed")
    return out


def select_row(s, topk: int) -> np.ndarray:
    """Ascending row-relative top-k indices of s (fp64), -1 padded."""
    s = _np(s, np.float64)
    out = np.empty(topk, dtype=np.int32)
    if _load().orc_select_row(_ptr(s), s.size, topk, _ptr(out)):
        raise MemoryError("oracle select_row failed")
    return out


def score_topk(inp, rows=None, nthreads: int | None = None, want_scores: bool = False):
    """Exact top-k for `rows` (default: all).  Returns out [len(rows), topk]
    int32, and with want_scores also the fp64 scores [len(rows), max_len]."""
    X = _indexer(inp)
    topk = int(inp.topk)
    rows = np.arange(X.rows, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    rows = np.ascontiguousarray(rows)
    out = np.empty((rows.size, topk), dtype=np.int32)
    lens = (X.ke.astype(np.int64) - X.ks.astype(np.int64)).clip(min=0)
    sstride = int(lens[rows].max()) if (want_scores and rows.size) else 0
    sc = np.zeros((rows.size, max(sstride, 1)), dtype=np.float64) if want_scores else None
    qsf, ksf = X.sf_ptrs()
    e = _load().orc_score_topk(_ptr(X.q), qsf, _ptr(X.k), ksf, X.dtype, _ptr(X.k_scale),
                               _ptr(X.w), _ptr(X.ks), _ptr(X.ke), X.H, X.D, _ptr(rows),
                               rows.size, topk, _ptr(out), _ptr(sc) if want_scores else None,
                               max(sstride, 1), nthreads or default_threads())
    if e:
        raise MemoryError("oracle score_topk failed")
    return (out, sc) if want_scores else out


def topk_from_scores(scores, ks, ke, topk: int, rows=None, nthreads: int | None = None):
    """Exact top-k of given fp32 scores [rows_total, stride]."""
    S = _np(scores, np.float32)
    ks_a, ke_a = _np(ks, np.int32), _np(ke, np.int32)
    rows = np.arange(S.shape[0], dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    rows = np.ascontiguousarray(rows)
    out = np.empty((rows.size, topk), dtype=np.int32)
    e = _load().orc_topk_from_scores(_ptr(S), S.shape[1], _ptr(ks_a), _ptr(ke_a), _ptr(rows),
                                     rows.size, topk, _ptr(out), nthreads or default_threads())
    if e:
        raise MemoryError("oracle topk_from_scores failed")
    return out


def page_transform(idx, table, page_size: int = 64, row_map=None, table_rows=None):
    """Page-table transform of idx [rows, topk] (a new array) and the number
    of positions set to -1 because their page lies outside the table row or
    their table row (row_map entry) outside the table's first `table_rows`
    rows (default: all of them)."""
    ix = _np(idx, np.int32)
    tb = _np(table, np.int32)
    table_rows = tb.shape[0] if table_rows is None else int(table_rows)
    if not 0 <= table_rows <= tb.shape[0]:
        raise ValueError("oracle page_transform: table_rows outside the table")
    rows, topk = ix.shape
    rm = None if row_map is None else _np(row_map, np.int32)
    out = np.empty_like(ix)
    lib = _load()
    fn = lib.orc_page_transform
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    fn.argtypes = [P, i32, i32, P, i64, i64, P, i32, P]
    fn.restype = i64
    bad = fn(_ptr(ix), rows, topk, _ptr(tb), table_rows, tb.shape[1],
             None if rm is None else _ptr(rm), page_size, _ptr(out))
    if bad < 0:
        raise ValueError("oracle page_transform: bad arguments")
    return out, int(bad)
