"""Thin ctypes binding of libhogwild (include/hogwild.h): argument marshalling only.

Every function maps one-to-one to a C entry point of the same name without the
``hw_`` prefix.  Tensors are passed as device pointers (``tensor.data_ptr()``);
all computation happens in the library's CUDA kernels.  If the library has not
been built this module raises on first use: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libhogwild.so")

HW_OK = 0
HW_F32, HW_BF16, HW_FP8_E4M3 = 0, 1, 2
HW_DESC_VIEW_LIMITS = 1
HW_DESC_EARLY_LOADS = 2
STATUS = {0: "HW_OK", -1: "HW_ERR_INVALID", -2: "HW_ERR_UNSUPPORTED", -3: "HW_ERR_WORKSPACE",
          -4: "HW_ERR_CAPACITY", -5: "HW_ERR_OVERLAP", -6: "HW_ERR_CUDA", -7: "HW_ERR_DEVICE"}
DEV_FLAGS = {1: "HW_DEV_BAD_BLOCK", 2: "HW_DEV_BAD_RANGE", 4: "HW_DEV_BAD_HEADMAP",
             8: "HW_DEV_TOO_MANY_REFS", 16: "HW_DEV_TIMEOUT", 32: "HW_DEV_BAD_PLAN"}

# every symbol the header declares
EXPORTS = ["hw_attn_decode_workspace_size", "hw_workspace_init", "hw_attn_decode",
           "hw_attn_plan", "hw_attn_decode_planned", "hw_attn_decode_planned_fp8", "hw_attn_plan_limited", "hw_attn_plan_append",
           "hw_attn_append_decode_planned_fp8",
           "hw_attn_append_decode_planned", "hw_plan_export", "hw_attn_decode_noalloc",
           "hw_block_commit", "hw_block_commit_many", "hw_workspace_status", "hw_views_combined",
           "hw_views", "hw_views_chunked", "hw_last_cuda_error", "hw_status_string",
           "hw_test_set_merge_wait_limit", "hw_noalloc_status", "hw_trace_read", "hw_trace_clear"]
HW_LAYOUT_COMBINED, HW_LAYOUT_INTERLEAVED, HW_LAYOUT_CONTIGUOUS = 0, 1, 2
LAYOUTS = {"combined": HW_LAYOUT_COMBINED, "interleaved": HW_LAYOUT_INTERLEAVED,
           "contiguous": HW_LAYOUT_CONTIGUOUS}
HW_MAX_COMMITS = 64


class HwError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)} ({status})")


class AttnDesc(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("n_blocks", ctypes.c_int32),
        ("max_view_blocks", ctypes.c_int32),
        ("cache_capacity", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("rope_theta", ctypes.c_double),
        ("scale", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_lib = None


def lib(path: Optional[str] = None):
    """Load libhogwild.so (built by ``concurrent_shared_kv_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libhogwild.so not found at {p}: build it with "
                           "`python -m concurrent_shared_kv_gb300.build` (no fallback path exists)")
    L = ctypes.CDLL(p)
    L.hw_attn_decode_workspace_size.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(ctypes.c_size_t)]
    L.hw_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
    L.hw_attn_decode.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 12 + [ctypes.c_size_t, _P]
    L.hw_attn_plan.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 7 + [ctypes.c_size_t, _P]
    L.hw_attn_decode_planned.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 6 + [ctypes.c_size_t, _P]
    L.hw_attn_decode_planned_fp8.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 8 + [ctypes.c_size_t, _P]
    L.hw_attn_plan_limited.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 8 + [ctypes.c_size_t, _P]
    L.hw_attn_plan_append.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 9 + [ctypes.c_size_t, _P]
    L.hw_attn_append_decode_planned.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 8 + [ctypes.c_size_t, _P]
    L.hw_attn_append_decode_planned_fp8.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 10 + [
        ctypes.c_size_t, _P]
    L.hw_plan_export.argtypes = [ctypes.POINTER(AttnDesc), _P, ctypes.c_size_t, _P, ctypes.c_int32,
                                 ctypes.POINTER(ctypes.c_int32), _P]
    L.hw_attn_decode_noalloc.argtypes = [ctypes.POINTER(AttnDesc)] + [_P] * 12
    L.hw_trace_read.argtypes = [_P]
    L.hw_trace_clear.argtypes = []
    L.hw_block_commit.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_double, _P, _P, ctypes.c_int64, ctypes.c_int32,
                                  ctypes.c_int32, _P, _P, ctypes.c_int64, ctypes.c_int32,
                                  ctypes.c_int32, _P]
    L.hw_block_commit_many.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_double, _P, _P, ctypes.c_int64, _P, _P,
                                       ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P, _P]
    L.hw_workspace_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), _P]
    L.hw_views_combined.argtypes = [ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]
    L.hw_views.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]
    L.hw_views_chunked.argtypes = [ctypes.c_int32] * 4 + [_P] * 5
    L.hw_last_cuda_error.argtypes = []
    L.hw_test_set_merge_wait_limit.argtypes = [ctypes.c_int64]
    L.hw_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int32), _P]
    L.hw_status_string.argtypes = [ctypes.c_int]
    L.hw_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "hw_status_string":
            getattr(L, name).restype = ctypes.c_int
    if path is None:
        _lib = L
    return L


def use_library(path: str):
    """Make the library at `path` the process's (e.g. the HW_TRACE build);
    before any other call."""
    global _lib
    _lib = lib(path)
    return _lib


def _ptr(x) -> Optional[int]:
    """Device/host pointer of a tensor, numpy array or int (None stays NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(stream) -> Optional[int]:
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream or None
        except Exception:
            return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check(fn: str, st: int):
    if st != HW_OK:
        raise HwError(fn, st)


def make_desc(n_rows, n_q_heads, n_kv_heads, head_dim, n_blocks, max_view_blocks, cache_capacity,
              dtype, rope_theta, scale, flags=0) -> AttnDesc:
    return AttnDesc(int(n_rows), int(n_q_heads), int(n_kv_heads), int(head_dim), int(n_blocks),
                    int(max_view_blocks), int(cache_capacity), int(dtype), float(rope_theta),
                    float(scale), int(flags))


def attn_decode_workspace_size(desc: AttnDesc) -> int:
    n = ctypes.c_size_t(0)
    _check("hw_attn_decode_workspace_size", lib().hw_attn_decode_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def workspace_init(workspace, nbytes: int, stream=None):
    _check("hw_workspace_init", lib().hw_workspace_init(_ptr(workspace), int(nbytes), _stream(stream)))


def attn_decode(desc: AttnDesc, q, k_cache, v_cache, block_start, block_len, view_block,
                view_offset, q_pos, out, lse, workspace, workspace_bytes: int, q_to_kv=None,
                stream=None) -> int:
    """hw_attn_decode; returns the status (raises on failure)."""
    st = lib().hw_attn_decode(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                              _ptr(block_start), _ptr(block_len), _ptr(view_block),
                              _ptr(view_offset), _ptr(q_pos), _ptr(q_to_kv), _ptr(out), _ptr(lse),
                              _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("hw_attn_decode", st)
    return st


def attn_plan(desc: AttnDesc, block_start, block_len, view_block, view_offset, q_pos, workspace,
              workspace_bytes: int, q_to_kv=None, stream=None) -> int:
    """hw_attn_plan: the step's metadata planned once into the workspace."""
    st = lib().hw_attn_plan(ctypes.byref(desc), _ptr(block_start), _ptr(block_len), _ptr(view_block),
                            _ptr(view_offset), _ptr(q_pos), _ptr(q_to_kv), _ptr(workspace),
                            int(workspace_bytes), _stream(stream))
    _check("hw_attn_plan", st)
    return st


def attn_decode_planned(desc: AttnDesc, q, k_cache, v_cache, out, lse, workspace,
                        workspace_bytes: int, stream=None) -> int:
    """hw_attn_decode_planned: one layer against the plan in the workspace."""
    st = lib().hw_attn_decode_planned(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                      _stream(stream))
    _check("hw_attn_decode_planned", st)
    return st


def attn_decode_planned_fp8(desc: AttnDesc, q, k_cache, v_cache, k_scale, v_scale, out, lse,
                            workspace, workspace_bytes: int, stream=None) -> int:
    """hw_attn_decode_planned_fp8: one layer over E4M3 caches with per-kv-head
    scales, against the plan in the workspace."""
    st = lib().hw_attn_decode_planned_fp8(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse),
                                          _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("hw_attn_decode_planned_fp8", st)
    return st


def attn_append_decode_planned_fp8(desc: AttnDesc, q, k_new, v_new, k_cache, v_cache, k_scale,
                                   v_scale, out, lse, workspace, workspace_bytes: int,
                                   stream=None) -> int:
    """hw_attn_append_decode_planned_fp8: the layer's new tokens written into
    E4M3 caches (divided by the head scales, rounded), then the layer decoded."""
    st = lib().hw_attn_append_decode_planned_fp8(
        ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
        _stream(stream))
    _check("hw_attn_append_decode_planned_fp8", st)
    return st


def attn_plan_limited(desc: AttnDesc, block_start, block_len, view_block, view_offset, view_limit,
                      q_pos, workspace, workspace_bytes: int, q_to_kv=None, stream=None) -> int:
    """hw_attn_plan_limited: the step planned with a token limit per view
    entry (view_limit[r][v]: row r attends the first view_limit[r][v] tokens
    of block view_block[r][v]; negative = all of them)."""
    st = lib().hw_attn_plan_limited(ctypes.byref(desc), _ptr(block_start), _ptr(block_len),
                                    _ptr(view_block), _ptr(view_offset), _ptr(view_limit),
                                    _ptr(q_pos), _ptr(q_to_kv), _ptr(workspace),
                                    int(workspace_bytes), _stream(stream))
    _check("hw_attn_plan_limited", st)
    return st


def attn_plan_append(desc: AttnDesc, block_start, block_len, view_block, view_offset, q_pos,
                     append_block, append_pos, workspace, workspace_bytes: int, q_to_kv=None,
                     stream=None) -> int:
    """hw_attn_plan_append: the step planned with each row's new token
    (append_block[r], append_pos[r]; -1 = none)."""
    st = lib().hw_attn_plan_append(ctypes.byref(desc), _ptr(block_start), _ptr(block_len),
                                   _ptr(view_block), _ptr(view_offset), _ptr(q_pos), _ptr(q_to_kv),
                                   _ptr(append_block), _ptr(append_pos), _ptr(workspace),
                                   int(workspace_bytes), _stream(stream))
    _check("hw_attn_plan_append", st)
    return st


def attn_append_decode_planned(desc: AttnDesc, q, k_new, v_new, k_cache, v_cache, out, lse,
                               workspace, workspace_bytes: int, stream=None) -> int:
    """hw_attn_append_decode_planned: the layer's new tokens written, then the
    layer decoded, in one launch."""
    st = lib().hw_attn_append_decode_planned(ctypes.byref(desc), _ptr(q), _ptr(k_new), _ptr(v_new),
                                             _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse),
                                             _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("hw_attn_append_decode_planned", st)
    return st


def plan_export(desc: AttnDesc, workspace, workspace_bytes: int, max_ctas: int = 1024, stream=None):
    """hw_plan_export: the plan's per-CTA work split as an int64 array [ctas][15]
    (u0, u1, n_first, first rows x3, kv heads x3, segment flags x3, column
    groups x3)."""
    out = np.zeros((max_ctas, 15), np.int64)
    n = ctypes.c_int32(0)
    st = lib().hw_plan_export(ctypes.byref(desc), _ptr(workspace), int(workspace_bytes),
                              out.ctypes.data, int(max_ctas), ctypes.byref(n), _stream(stream))
    _check("hw_plan_export", st)
    return out[:n.value]


def attn_decode_noalloc(desc: AttnDesc, q, k_cache, v_cache, block_start, block_len, view_block,
                        view_offset, q_pos, out, lse, q_to_kv=None, stream=None) -> int:
    """hw_attn_decode_noalloc: the decode without a caller workspace, for code
    that cannot allocate device memory (it uses the library's fixed scratch)."""
    st = lib().hw_attn_decode_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(block_start), _ptr(block_len), _ptr(view_block),
                                      _ptr(view_offset), _ptr(q_pos), _ptr(q_to_kv), _ptr(out),
                                      _ptr(lse), _stream(stream))
    _check("hw_attn_decode_noalloc", st)
    return st


def block_commit(dtype: int, n_layers: int, n_kv_heads: int, head_dim: int, rope_theta: float,
                 k_src, v_src, src_capacity: int, src_begin: int, n_tokens: int, k_dst, v_dst,
                 dst_capacity: int, dst_offset: int, pos_delta: int, stream=None) -> int:
    st = lib().hw_block_commit(int(dtype), int(n_layers), int(n_kv_heads), int(head_dim),
                               float(rope_theta), _ptr(k_src), _ptr(v_src), int(src_capacity),
                               int(src_begin), int(n_tokens), _ptr(k_dst), _ptr(v_dst),
                               int(dst_capacity), int(dst_offset), int(pos_delta), _stream(stream))
    _check("hw_block_commit", st)
    return st


def block_commit_many(dtype: int, n_layers: int, n_kv_heads: int, head_dim: int, rope_theta: float,
                      k_src, v_src, src_capacity: int, k_dst, v_dst, dst_capacity: int,
                      src_begin, n_tokens, dst_offset, pos_delta, stream=None) -> int:
    """Several commits in one launch; the four per-commit sequences are host ints."""
    arrs = [np.ascontiguousarray(x, dtype=np.int32) for x in (src_begin, n_tokens, dst_offset, pos_delta)]
    n = len(arrs[0])
    if any(len(x) != n for x in arrs):
        raise ValueError("per-commit sequences of different lengths")
    st = lib().hw_block_commit_many(int(dtype), int(n_layers), int(n_kv_heads), int(head_dim),
                                    float(rope_theta), _ptr(k_src), _ptr(v_src), int(src_capacity),
                                    _ptr(k_dst), _ptr(v_dst), int(dst_capacity), int(n),
                                    *[x.ctypes.data for x in arrs], _stream(stream))
    _check("hw_block_commit_many", st)
    return st


def workspace_status(workspace, stream=None) -> int:
    """Device error bits (HW_DEV_*) since the last read; synchronises the stream."""
    f = ctypes.c_int32(0)
    _check("hw_workspace_status", lib().hw_workspace_status(_ptr(workspace), ctypes.byref(f), _stream(stream)))
    return int(f.value)


def views_combined(block_len, n_problems: int, n_workers: int):
    """Host helper: (view_block, view_offset, q_pos) int32 arrays of the combined layout."""
    bl = np.ascontiguousarray(block_len, dtype=np.int32)
    rows, V = n_problems * n_workers, n_workers + 1
    vb = np.empty((rows, V), np.int32)
    vo = np.empty((rows, V), np.int32)
    qp = np.empty(rows, np.int32)
    _check("hw_views_combined", lib().hw_views_combined(int(n_problems), int(n_workers), bl.ctypes.data,
                                                        vb.ctypes.data, vo.ctypes.data, qp.ctypes.data))
    return vb, vo, qp


def views(layout, block_len, n_problems: int, n_workers: int):
    """Host helper: (view_block, view_offset, q_pos) of a cache layout ("combined",
    "interleaved", "contiguous" or its HW_LAYOUT_* value)."""
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    bl = np.ascontiguousarray(block_len, dtype=np.int32)
    rows, V = n_problems * n_workers, n_workers + 1
    vb = np.empty((rows, V), np.int32)
    vo = np.empty((rows, V), np.int32)
    qp = np.empty(rows, np.int32)
    _check("hw_views", lib().hw_views(lay, int(n_problems), int(n_workers), bl.ctypes.data,
                                      vb.ctypes.data, vo.ctypes.data, qp.ctypes.data))
    return vb, vo, qp


def views_chunked(layout, block_len, n_problems: int, n_workers: int, chunk: int):
    """Host helper: (view_block, view_offset, view_limit, q_pos) of T-token
    query chunks (T = chunk) in a cache layout; row (p, w, t) at index
    (p*W + w)*T + t."""
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    bl = np.ascontiguousarray(block_len, dtype=np.int32)
    rows, V = n_problems * n_workers * chunk, n_workers + 1
    vb = np.empty((rows, V), np.int32)
    vo = np.empty((rows, V), np.int32)
    vl = np.empty((rows, V), np.int32)
    qp = np.empty(rows, np.int32)
    _check("hw_views_chunked", lib().hw_views_chunked(lay, int(n_problems), int(n_workers), int(chunk),
                                                      bl.ctypes.data, vb.ctypes.data, vo.ctypes.data,
                                                      vl.ctypes.data, qp.ctypes.data))
    return vb, vo, vl, qp


def status_string(st: int) -> str:
    return lib().hw_status_string(int(st)).decode()


def last_cuda_error() -> int:
    return int(lib().hw_last_cuda_error())


def noalloc_status(stream=None) -> int:
    """hw_noalloc_status: the no-allocation calls' device error bits (read and cleared)."""
    f = ctypes.c_int32(0)
    _check("hw_noalloc_status", lib().hw_noalloc_status(ctypes.byref(f), _stream(stream)))
    return int(f.value)


def test_set_merge_wait_limit(cycles: int):
    """hw_test_set_merge_wait_limit: the merge's wait bound (SM cycles) for the
    calls that follow; 0 restores the default."""
    _check("hw_test_set_merge_wait_limit", lib().hw_test_set_merge_wait_limit(int(cycles)))


TRACE_SHAPE = (8, 160, 24)  # calls (mod 8), CTAs, points: see hw_trace_read


def trace_read() -> np.ndarray:
    """hw_trace_read: the layer timeline of an HW_TRACE build (uint64 ns)."""
    out = np.zeros(TRACE_SHAPE, np.uint64)
    _check("hw_trace_read", lib().hw_trace_read(out.ctypes.data))
    return out


def trace_clear() -> None:
    _check("hw_trace_clear", lib().hw_trace_clear())
