"""Python binding of libidx, the GB300 (sm_103a) sparse-attention prefill indexer.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libidx.so`` (built from ``csrc/`` by ``build.py``).  PyTorch
provides device memory and the current stream.  There is no CPU path: when the
library is missing or the GPU is not an sm_103 part, the calls raise.

Entry points (same names as the C ABI in ``include/idx.h``):
  idx_score_topk            fused score + exact top-k (no [rows, keys] logits)
  idx_score_topk_host       the same on host-memory inputs and output (copies overlap the compute)
  idx_topk_from_scores      exact radix top-k of given fp32 scores
  idx_score_materialise     the two-pass baseline's score pass
  idx_score_topk_mxfp4, idx_score_materialise_mxfp4, idx_mxfp4_to_e4m3
                            the same on MXFP4 inputs (expanded exactly to e4m3)
  idx_score_topk_workspace, idx_topk_workspace, idx_status_string
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "IdxError", "Options", "Stats", "load", "idx_score_topk", "idx_score_topk_workspace",
    "idx_score_topk_host", "idx_score_topk_host_workspace",
    "idx_topk_from_scores", "idx_topk_workspace", "idx_score_materialise",
    "idx_status_string", "DTYPES", "STAT_FIELDS", "StageEvents", "idx_launch_count",
    "idx_score_topk_noalloc", "idx_page_table_transform", "idx_route_fused",
    "idx_score_topk_routed", "idx_score_topk_routed_workspace", "idx_mxfp4_to_e4m3",
    "idx_score_topk_mxfp4", "idx_score_materialise_mxfp4",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libidx.so")

IDX_BF16, IDX_FP8_E4M3, IDX_MXFP4 = 1, 2, 3
DTYPES = {torch.bfloat16: IDX_BF16, torch.float8_e4m3fn: IDX_FP8_E4M3}
STAT_FIELDS = ("emit_all_rows", "overflow_rows", "short_rows", "fallback_rows", "max_count",
               "split_rows", "tie_rescan_rows", "reserved")


class IdxError(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed: {text} (status {code})")
        self.code = code


class Options(ctypes.Structure):
    """Mirror of idx_options."""
    _fields_ = [("cap_factor", ctypes.c_float), ("target_factor", ctypes.c_float),
                ("sample_stride", ctypes.c_int), ("row_split", ctypes.c_int),
                ("d_status", ctypes.c_void_p), ("d_stats", ctypes.c_void_p),
                ("relative_rows", ctypes.c_int), ("test_stall_us", ctypes.c_int),
                ("stage_events", ctypes.c_void_p)]


class Stats:
    """Device counters (idx_stats) plus the device status word."""

    def __init__(self, device=None):
        dev = device or torch.device("cuda", torch.cuda.current_device())
        self.buf = torch.zeros(len(STAT_FIELDS) + 1, dtype=torch.int32, device=dev)

    def reset(self):
        self.buf.zero_()

    @property
    def stats_ptr(self) -> int:
        return self.buf.data_ptr()

    @property
    def status_ptr(self) -> int:
        return self.buf.data_ptr() + 4 * len(STAT_FIELDS)

    def read(self) -> dict:
        v = self.buf.cpu().tolist()
        d = dict(zip(STAT_FIELDS, v[:len(STAT_FIELDS)]))
        d["status"] = v[-1]
        return d


_lib = None


def load(path: str | None = None):
    """Load libidx.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libidx.so not found at {p}; run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(p)
    P, I, LL, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    lib.idx_score_topk_workspace.argtypes = [I, LL, LL, I, I, I, I, P]
    lib.idx_score_topk_workspace.restype = SZ
    lib.idx_score_topk.argtypes = [P, P, P, P, P, P, I, LL, LL, I, I, I, I, P, P, SZ, P, P]
    lib.idx_score_topk.restype = I
    lib.idx_score_topk_host_workspace.argtypes = [I, LL, LL, I, I, I, I, P]
    lib.idx_score_topk_host_workspace.restype = SZ
    lib.idx_score_topk_host.argtypes = [P, P, P, P, P, P, I, LL, LL, I, I, I, I, P, P, SZ, P, P]
    lib.idx_score_topk_host.restype = I
    lib.idx_topk_workspace.argtypes = [I, LL, I, P]
    lib.idx_topk_workspace.restype = SZ
    lib.idx_topk_from_scores.argtypes = [P, LL, P, P, I, I, P, P, SZ, P, P]
    lib.idx_topk_from_scores.restype = I
    lib.idx_score_materialise.argtypes = [P, P, P, P, P, P, I, LL, I, I, I, P, LL, P, P]
    lib.idx_score_materialise.restype = I
    lib.idx_route_fused.argtypes = [I, LL, I]
    lib.idx_route_fused.restype = I
    lib.idx_score_topk_routed_workspace.argtypes = [I, LL, LL, I, I, I, I, P]
    lib.idx_score_topk_routed_workspace.restype = SZ
    lib.idx_score_topk_routed.argtypes = [P, P, P, P, P, P, I, LL, LL, I, I, I, I, P, P, SZ, P,
                                          P]
    lib.idx_score_topk_routed.restype = I
    lib.idx_page_table_transform.argtypes = [P, I, I, P, I, LL, P, I, P, P]
    lib.idx_page_table_transform.restype = I
    lib.idx_mxfp4_to_e4m3.argtypes = [P, P, LL, I, P, P, P]
    lib.idx_mxfp4_to_e4m3.restype = I
    lib.idx_score_topk_mxfp4_workspace.argtypes = [I, LL, LL, I, I, I, P]
    lib.idx_score_topk_mxfp4_workspace.restype = SZ
    lib.idx_score_topk_mxfp4.argtypes = [P, P, P, P, P, P, P, P, I, LL, LL, I, I, I, P, P, SZ,
                                         P, P]
    lib.idx_score_topk_mxfp4.restype = I
    lib.idx_score_materialise_mxfp4_workspace.argtypes = [I, LL, I, I]
    lib.idx_score_materialise_mxfp4_workspace.restype = SZ
    lib.idx_score_materialise_mxfp4.argtypes = [P, P, P, P, P, P, P, P, I, LL, I, I, P, LL, P,
                                                SZ, P, P]
    lib.idx_score_materialise_mxfp4.restype = I
    lib.idx_status_string.argtypes = [I]
    lib.idx_status_string.restype = ctypes.c_char_p
    lib.idx_version.argtypes = []
    lib.idx_version.restype = I
    lib.idx_last_cuda_error.argtypes = []
    lib.idx_last_cuda_error.restype = ctypes.c_char_p
    lib.idx_launch_count.argtypes = []
    lib.idx_launch_count.restype = ctypes.c_ulonglong
    _lib = lib
    return lib


def idx_launch_count() -> int:
    """Kernels launched by libidx in this process so far."""
    return int(load().idx_launch_count())


class StageEvents:
    """CUDA events the library records at its stage boundaries
    (options.stage_events); elapsed(i, j) in ms after a synchronize."""

    def __init__(self, n: int = 5):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in self.events:
            e.record()  # torch creates its events lazily, on the first record
        self._arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in self.events])

    @property
    def ptr(self) -> int:
        return ctypes.cast(self._arr, ctypes.c_void_p).value

    def elapsed(self, i: int, j: int) -> float:
        return self.events[i].elapsed_time(self.events[j])


def idx_status_string(code: int) -> str:
    return load().idx_status_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != 0:
        text = idx_status_string(code)
        cuda = load().idx_last_cuda_error().decode() if code in (4, 5) else ""
        raise IdxError(fn, code, f"{text} ({cuda})" if cuda else text)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dev(*ts):
    """Check that every tensor is a contiguous CUDA tensor and that all of them
    live on one device; returns that device."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("idx: every tensor must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("idx: tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"idx: tensors on different devices ({dev} and {t.device})")
    return dev


def make_options(options: Options | dict | None, stats: Stats | None = None) -> Options | None:
    if options is None and stats is None:
        return None
    o = options if isinstance(options, Options) else Options(**(options or {}))
    if stats is not None:
        o.d_stats = stats.stats_ptr
        o.d_status = stats.status_ptr
    return o


def _opt_ref(o: Options | None):
    return None if o is None else ctypes.byref(o)


def idx_score_topk_workspace(rows: int, keys: int, max_len: int, H: int, D: int, topk: int,
                             dtype, options=None) -> int:
    dt = DTYPES[dtype] if not isinstance(dtype, int) else dtype
    o = make_options(options)
    return int(load().idx_score_topk_workspace(rows, keys, max_len, H, D, topk, dt, _opt_ref(o)))


def idx_score_topk(q, k, k_scale, w, ks, ke, topk: int, *, max_len: int = 0, out=None, ws=None,
                   options=None, stats: Stats | None = None, stream=None):
    """Exact top-k indices [rows, topk] int32 (ascending, -1 padded)."""
    dev = _dev(q, k, k_scale, w, ks, ke, out, ws)
    with torch.cuda.device(dev):
        rows, H, D = q.shape
        keys = k.shape[0]
        dt = DTYPES[q.dtype]
        o = make_options(options, stats)
        need = idx_score_topk_workspace(rows, keys, max_len, H, D, topk, dt, o)
        if out is None:
            out = torch.empty(rows, topk, dtype=torch.int32, device=q.device)
        if ws is None:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        _check("idx_score_topk", load().idx_score_topk(
            _ptr(q), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke), rows, keys, max_len, H, D,
            topk, dt, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _opt_ref(o),
            _stream(stream)))
        return out


def idx_score_topk_host_workspace(rows: int, keys: int, max_len: int, H: int, D: int, topk: int,
                                  dtype, options=None) -> int:
    dt = DTYPES[dtype] if not isinstance(dtype, int) else dtype
    return int(load().idx_score_topk_host_workspace(rows, keys, max_len, H, D, topk, dt,
                                                    _opt_ref(make_options(options))))


def idx_score_topk_host(q, k, k_scale, w, ks, ke, topk: int, *, max_len: int = 0, out=None,
                        ws=None, device=None, options=None, stats: Stats | None = None,
                        stream=None):
    """idx_score_topk on inputs in host memory (CPU tensors; pinned ones let the
    copies overlap the compute): returns the indices [rows, topk] int32 in host
    memory, complete once `stream` is synchronised.  ws is a device uint8
    tensor (allocated on `device`, default the current one, when None)."""
    for t in (q, k, k_scale, w, ks, ke, out):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("idx_score_topk_host: inputs and out are contiguous CPU tensors")
    dev = ws.device if ws is not None else torch.device("cuda", torch.cuda.current_device()) \
        if device is None else torch.device(device)
    if not dev.type == "cuda":
        raise ValueError("idx_score_topk_host: the workspace lives on a CUDA device")
    with torch.cuda.device(dev):
        rows, H, D = q.shape
        keys = k.shape[0]
        dt = DTYPES[q.dtype]
        o = make_options(options, stats)
        need = idx_score_topk_host_workspace(rows, keys, max_len, H, D, topk, dt, o)
        if out is None:
            out = torch.empty(rows, topk, dtype=torch.int32, pin_memory=True)
        if ws is None:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _check("idx_score_topk_host", load().idx_score_topk_host(
            _ptr(q), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke), rows, keys, max_len, H,
            D, topk, dt, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _opt_ref(o),
            _stream(stream)))
        return out


def idx_topk_workspace(rows: int, row_stride: int, topk: int, options=None) -> int:
    return int(load().idx_topk_workspace(rows, row_stride, topk, _opt_ref(make_options(options))))


def idx_topk_from_scores(scores, ks, ke, topk: int, *, out=None, ws=None, options=None,
                         stats: Stats | None = None, stream=None):
    """Exact top-k of fp32 scores [rows, row_stride]; ks may be None."""
    dev = _dev(scores, ks, ke, out, ws)
    with torch.cuda.device(dev):
        if scores.dtype != torch.float32:
            raise ValueError("idx_topk_from_scores: scores must be float32")
        rows, stride = scores.shape
        o = make_options(options, stats)
        need = int(load().idx_topk_workspace(rows, stride, topk, _opt_ref(o)))
        if out is None:
            out = torch.empty(rows, topk, dtype=torch.int32, device=scores.device)
        if ws is None and need:
            ws = torch.empty(need, dtype=torch.uint8, device=scores.device)
        nbytes = 0 if ws is None else ws.numel() * ws.element_size()
        _check("idx_topk_from_scores", load().idx_topk_from_scores(
            _ptr(scores), stride, _ptr(ks), _ptr(ke), rows, topk, _ptr(out), _ptr(ws), nbytes,
            _opt_ref(o), _stream(stream)))
        return out


def idx_score_materialise(q, k, k_scale, w, ks, ke, *, out=None, row_stride: int | None = None,
                          options=None, stats: Stats | None = None, stream=None):
    """fp32 scores [rows, row_stride]; row r's key j at column j - ks[r]."""
    dev = _dev(q, k, k_scale, w, ks, ke, out)
    with torch.cuda.device(dev):
        rows, H, D = q.shape
        keys = k.shape[0]
        if out is None:
            stride = row_stride or keys
            out = torch.empty(rows, stride, dtype=torch.float32, device=q.device)
        stride = out.shape[1]
        o = make_options(options, stats)
        _check("idx_score_materialise", load().idx_score_materialise(
            _ptr(q), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke), rows, keys, H, D,
            DTYPES[q.dtype], _ptr(out), stride, _opt_ref(o), _stream(stream)))
        return out


def _mx_shapes(q, q_sf, k, k_sf):
    """rows, H, D of MXFP4 q [rows, H, D/2] uint8 with q_sf [rows, H, D/32] and k
    [keys, D/2] with k_sf [keys, D/32]."""
    for t in (q, q_sf, k, k_sf):
        if t.dtype != torch.uint8:
            raise ValueError("MXFP4 elements and scales are uint8 tensors")
    rows, H, half = q.shape
    D = 2 * half
    if q_sf.shape != (rows, H, D // 32) or k.shape[1] != half or \
            k_sf.shape != (k.shape[0], D // 32):
        raise ValueError("inconsistent MXFP4 shapes")
    return rows, H, D


def idx_mxfp4_to_e4m3(x, sf, *, out=None, options=None, stats: Stats | None = None,
                      stream=None):
    """MXFP4 rows x [n, D/2] + sf [n, D/32] -> e4m3 [n, D] (exact within the
    e4m3 range, else IDX_DEV_RANGE)."""
    dev = _dev(x, sf, out)
    with torch.cuda.device(dev):
        n, half = x.shape[0], x.shape[-1]
        D = 2 * half
        if out is None:
            out = torch.empty(*x.shape[:-1], D, dtype=torch.float8_e4m3fn, device=x.device)
        o = make_options(options, stats)
        _check("idx_mxfp4_to_e4m3", load().idx_mxfp4_to_e4m3(
            _ptr(x), _ptr(sf), x.numel() // half, D, _ptr(out), _opt_ref(o), _stream(stream)))
        return out


def idx_score_topk_mxfp4(q, q_sf, k, k_sf, k_scale, w, ks, ke, topk: int, *, max_len: int = 0,
                         out=None, ws=None, options=None, stats: Stats | None = None,
                         stream=None):
    """idx_score_topk on MXFP4 q/k (with their e8m0 block scales)."""
    dev = _dev(q, q_sf, k, k_sf, k_scale, w, ks, ke, out, ws)
    with torch.cuda.device(dev):
        rows, H, D = _mx_shapes(q, q_sf, k, k_sf)
        keys = k.shape[0]
        o = make_options(options, stats)
        need = int(load().idx_score_topk_mxfp4_workspace(rows, keys, max_len, H, D, topk,
                                                         _opt_ref(o)))
        if out is None:
            out = torch.empty(rows, topk, dtype=torch.int32, device=q.device)
        if ws is None:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        _check("idx_score_topk_mxfp4", load().idx_score_topk_mxfp4(
            _ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke),
            rows, keys, max_len, H, D, topk, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
            _opt_ref(o), _stream(stream)))
        return out


def idx_score_materialise_mxfp4(q, q_sf, k, k_sf, k_scale, w, ks, ke, *, out=None,
                                row_stride: int | None = None, ws=None, options=None,
                                stats: Stats | None = None, stream=None):
    """idx_score_materialise on MXFP4 q/k (with their e8m0 block scales)."""
    dev = _dev(q, q_sf, k, k_sf, k_scale, w, ks, ke, out, ws)
    with torch.cuda.device(dev):
        rows, H, D = _mx_shapes(q, q_sf, k, k_sf)
        keys = k.shape[0]
        if out is None:
            out = torch.empty(rows, row_stride or keys, dtype=torch.float32, device=q.device)
        need = int(load().idx_score_materialise_mxfp4_workspace(rows, keys, H, D))
        if ws is None:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        o = make_options(options, stats)
        _check("idx_score_materialise_mxfp4", load().idx_score_materialise_mxfp4(
            _ptr(q), _ptr(q_sf), _ptr(k), _ptr(k_sf), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke),
            rows, keys, H, D, _ptr(out), out.shape[1], _ptr(ws), ws.numel() * ws.element_size(),
            _opt_ref(o), _stream(stream)))
        return out


def idx_score_topk_noalloc(q, k, k_scale, w, ks, ke, topk: int, *, max_len: int = 0, out=None,
                           options=None, stats: Stats | None = None, stream=None):
    """idx_score_topk on the library's built-in scratch array (no workspace,
    no allocation by the library; out is allocated here when not given)."""
    dev = _dev(q, k, k_scale, w, ks, ke, out)
    with torch.cuda.device(dev):
        lib = load()
        fn = lib.idx_score_topk_noalloc
        P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        fn.argtypes = [P, P, P, P, P, P, I, LL, LL, I, I, I, I, P, P, P]
        fn.restype = I
        rows, H, D = q.shape
        if out is None:
            out = torch.empty(rows, topk, dtype=torch.int32, device=q.device)
        o = make_options(options, stats)
        _check("idx_score_topk_noalloc", fn(
            _ptr(q), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke), rows, k.shape[0], max_len,
            H, D, topk, DTYPES[q.dtype], _ptr(out), _opt_ref(o), _stream(stream)))
        return out


def idx_page_table_transform(idx, table, page_size: int = 64, *, row_map=None, options=None,
                             stats: Stats | None = None, stream=None):
    """In place: every position p >= 0 of idx [rows, topk] int32 becomes
    table[t, p // page_size] * page_size + p % page_size (t = row_map[r] or r);
    -1 entries stay.  Returns idx."""
    dev = _dev(idx, table, row_map)
    with torch.cuda.device(dev):
        if idx.dtype != torch.int32 or table.dtype != torch.int32:
            raise ValueError("idx_page_table_transform: idx and table must be int32")
        if row_map is not None and row_map.dtype != torch.int32:
            raise ValueError("idx_page_table_transform: row_map must be int32")
        rows, topk = idx.shape
        o = make_options(options, stats)
        _check("idx_page_table_transform", load().idx_page_table_transform(
            _ptr(idx), rows, topk, _ptr(table), table.shape[0], table.shape[1], _ptr(row_map),
            page_size, _opt_ref(o), _stream(stream)))
        return idx


def idx_route_fused(rows: int, max_len: int, topk: int) -> bool:
    """The routing gate: True when a call of `rows` rows whose longest row sees
    max_len keys takes the fused path."""
    return bool(load().idx_route_fused(rows, max_len, topk))


def idx_score_topk_routed_workspace(rows: int, keys: int, max_len: int, H: int, D: int,
                                    topk: int, dtype, options=None) -> int:
    dt = DTYPES[dtype] if not isinstance(dtype, int) else dtype
    o = make_options(options)
    return int(load().idx_score_topk_routed_workspace(rows, keys, max_len, H, D, topk, dt,
                                                      _opt_ref(o)))


def idx_score_topk_routed(q, k, k_scale, w, ks, ke, topk: int, *, max_len: int = 0, out=None,
                          ws=None, options=None, stats: Stats | None = None, stream=None):
    """idx_score_topk by the faster path for the longest row (fused, or the
    logits then their top-k); the same indices either way."""
    dev = _dev(q, k, k_scale, w, ks, ke, out, ws)
    with torch.cuda.device(dev):
        rows, H, D = q.shape
        keys = k.shape[0]
        dt = DTYPES[q.dtype]
        o = make_options(options, stats)
        need = int(load().idx_score_topk_routed_workspace(rows, keys, max_len, H, D, topk, dt,
                                                          _opt_ref(o)))
        if out is None:
            out = torch.empty(rows, topk, dtype=torch.int32, device=q.device)
        if ws is None:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        _check("idx_score_topk_routed", load().idx_score_topk_routed(
            _ptr(q), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(ks), _ptr(ke), rows, keys, max_len, H, D,
            topk, dt, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _opt_ref(o),
            _stream(stream)))
        return out
