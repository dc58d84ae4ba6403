"""Sliding-window attention on GB300 (sm_103a): thin Python binding of libswa.so.

The functions here marshal torch tensors into the C ABI of ``include/swa.h``
(``swa_fwd``, ``swa_decode``, ``swa_cache_append``, ``swa_decode_append``,
``swa_prefill_chunk`` and their workspace queries) and call it on the current
CUDA stream.  Every step of the computation runs in the library's
kernels; there is no fallback path.  If the library has not been built, the
first call raises (``build()`` compiles it in-tree with nvcc).

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build_mod

__all__ = [
    "SwaError", "build", "load_library", "library_path",
    "swa_fwd", "swa_decode", "swa_fwd_workspace_size", "swa_decode_workspace_size",
    "swa_check_device_error", "swa_status_string", "swa_abi_version",
    "SwaFwdParams", "SwaDecodeParams", "GLOBAL_FULL", "GLOBAL_SINK",
    "SwaCacheParams", "SwaChunkParams", "swa_cache_append", "swa_decode_append", "swa_prefill_chunk",
    "SwaDeviceErrors", "SwaDebugFaults", "swa_read_device_errors", "swa_debug_set_faults",
]

_c_i64x3 = ctypes.c_int64 * 3


class SwaFwdParams(ctypes.Structure):
    """Mirror of ``swa_fwd_params`` in include/swa.h."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_strides", _c_i64x3), ("k_strides", _c_i64x3), ("v_strides", _c_i64x3),
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
        ("d_h", ctypes.c_int32), ("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
        ("scale", ctypes.c_float), ("global_idx", ctypes.c_void_p), ("n_global", ctypes.c_int32),
        ("o", ctypes.c_void_p), ("o_strides", _c_i64x3), ("lse", ctypes.c_void_p), ("row_counts", ctypes.c_void_p),
        ("global_mode", ctypes.c_int32), ("q_g", ctypes.c_void_p), ("k_g", ctypes.c_void_p), ("v_g", ctypes.c_void_p),
        ("qg_strides", _c_i64x3), ("kg_strides", _c_i64x3), ("vg_strides", _c_i64x3),
        ("dilation", ctypes.POINTER(ctypes.c_int32)),
    ]


class SwaDecodeParams(ctypes.Structure):
    """Mirror of ``swa_decode_params`` in include/swa.h."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("slot_pos", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
        ("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("d_h", ctypes.c_int32),
        ("W", ctypes.c_int32), ("scale", ctypes.c_float),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("row_counts", ctypes.c_void_p),
        ("window", ctypes.c_int32), ("n_sink", ctypes.c_int32),
    ]


class SwaCacheParams(ctypes.Structure):
    """Mirror of ``swa_cache_params`` in include/swa.h."""

    _fields_ = [
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("slot_pos", ctypes.c_void_p),
        ("B", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("d_h", ctypes.c_int32), ("n_slots", ctypes.c_int32),
        ("n_sink", ctypes.c_int32),
    ]


class SwaChunkParams(ctypes.Structure):
    """Mirror of ``swa_chunk_params`` in include/swa.h."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("p0", ctypes.c_void_p),
        ("B", ctypes.c_int32), ("C", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
        ("d_h", ctypes.c_int32), ("window", ctypes.c_int32), ("scale", ctypes.c_float),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("row_counts", ctypes.c_void_p), ("append", ctypes.c_int32),
    ]


class SwaDeviceErrors(ctypes.Structure):
    """Mirror of ``swa_device_errors`` in include/swa.h."""

    _fields_ = [("prefill", ctypes.c_uint32), ("split", ctypes.c_uint32), ("cache", ctypes.c_uint32)]


class SwaDebugFaults(ctypes.Structure):
    """Mirror of ``swa_debug_faults`` in include/swa.h."""

    _fields_ = [("band_stop_fill", ctypes.c_int32), ("split_stop_stage", ctypes.c_int32)]


# bits of the device error words
DEVERR_WAIT_TIMEOUT = 1
DEVERR_DRAIN_TIMEOUT = 2
DEVERR_GLOBAL_LIST = 4
DEVERR_BAD_POSITION = 1
DEVERR_CACHE_MISMATCH = 2
DEVERR_BOUNDS = 8

GLOBAL_FULL = 0  # global tokens: full rows and columns
GLOBAL_SINK = 1  # attention sinks: key columns only, never right of a row's band

STATUS = {0: "SWA_OK", 1: "SWA_ERR_INVALID_ARG", 2: "SWA_ERR_UNSUPPORTED", 3: "SWA_ERR_CUDA",
          4: "SWA_ERR_TIMEOUT", 5: "SWA_ERR_WORKSPACE"}


class SwaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} returned {STATUS.get(status, status)}: {swa_status_string(status)}"
        if status == 3:
            msg += f" ({load_library().swa_last_error_string().decode()})"
        super().__init__(msg)


_lib = None


def library_path() -> str:
    return _build_mod.LIB


def build(force: bool = False, debug: bool = False) -> str:
    """Compile libswa.so for sm_103a (in-tree) and return its path; debug=True builds
    libswa_debug.so, whose kernels check every computed index (SWA_DEVERR_BOUNDS)."""
    return _build_mod.build(force=force, debug=debug)


def load_library(path: str | None = None):
    """Load libswa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libswa.so not found at {p}; call sliding_window_attention_swa_gb300.build() first")
    lib = ctypes.CDLL(p)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.swa_fwd_workspace_size.argtypes = [ctypes.POINTER(SwaFwdParams)]
    lib.swa_fwd_workspace_size.restype = sz
    lib.swa_fwd.argtypes = [ctypes.POINTER(SwaFwdParams), vp, sz, vp]
    lib.swa_fwd.restype = ctypes.c_int
    lib.swa_decode_workspace_size.argtypes = [ctypes.POINTER(SwaDecodeParams)]
    lib.swa_decode_workspace_size.restype = sz
    lib.swa_decode.argtypes = [ctypes.POINTER(SwaDecodeParams), vp, sz, vp]
    lib.swa_decode.restype = ctypes.c_int
    lib.swa_decode_noalloc.argtypes = [ctypes.POINTER(SwaDecodeParams), vp]
    lib.swa_decode_noalloc.restype = ctypes.c_int
    lib.swa_cache_append.argtypes = [ctypes.POINTER(SwaCacheParams), vp, vp, ctypes.c_int32, vp, vp]
    lib.swa_cache_append.restype = ctypes.c_int
    lib.swa_decode_append.argtypes = [ctypes.POINTER(SwaDecodeParams), vp, vp, vp, sz, vp]
    lib.swa_decode_append.restype = ctypes.c_int
    lib.swa_prefill_chunk_workspace_size.argtypes = [ctypes.POINTER(SwaChunkParams), ctypes.POINTER(SwaCacheParams)]
    lib.swa_prefill_chunk_workspace_size.restype = sz
    lib.swa_prefill_chunk.argtypes = [ctypes.POINTER(SwaChunkParams), ctypes.POINTER(SwaCacheParams), vp, sz, vp]
    lib.swa_prefill_chunk.restype = ctypes.c_int
    lib.swa_check_device_error.argtypes = [vp]
    lib.swa_check_device_error.restype = ctypes.c_int
    lib.swa_read_device_errors.argtypes = [vp, ctypes.POINTER(SwaDeviceErrors)]
    lib.swa_read_device_errors.restype = ctypes.c_int
    lib.swa_debug_set_faults.argtypes = [ctypes.POINTER(SwaDebugFaults)]
    lib.swa_debug_set_faults.restype = ctypes.c_int
    lib.swa_last_error_string.argtypes = []
    lib.swa_last_error_string.restype = ctypes.c_char_p
    lib.swa_status_string.argtypes = [ctypes.c_int]
    lib.swa_status_string.restype = ctypes.c_char_p
    lib.swa_abi_version.argtypes = []
    lib.swa_abi_version.restype = ctypes.c_int32
    if path is None:
        _lib = lib
    return lib


def use_library(lib):
    """Make `lib` (as returned by load_library(path)) the library the functions of this
    module call -- for example the debug build -- and return the previous one (None if
    none was loaded yet)."""
    global _lib
    prev, _lib = _lib, lib
    return prev


def swa_status_string(status: int) -> str:
    return load_library().swa_status_string(int(status)).decode()


def swa_abi_version() -> int:
    return int(load_library().swa_abi_version())


def _stream_handle(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_bf16(name, t, ndim):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != ndim or t.stride(-1) != 1:
        raise ValueError(f"{name}: expected a CUDA bf16 tensor of rank {ndim} with a contiguous last dim")


def fwd_params(q, k, v, window_left: int, window_right: int, scale: float, global_idx, o, lse, row_counts,
               global_mode: int = GLOBAL_FULL, qkv_g=None, dilation=None):
    """Fill a SwaFwdParams from tensors (q/k/v/o [B,T,H,d] bf16; lse/row_counts [B,H_q,T]).

    qkv_g: optional (q_g, k_g, v_g) separate global projections; dilation: optional
    per-query-head list of band dilations (host ints)."""
    B, T, Hq, D = q.shape
    p = SwaFwdParams()
    p.q, p.k, p.v, p.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    p.q_strides = _c_i64x3(*q.stride()[:3])
    p.k_strides = _c_i64x3(*k.stride()[:3])
    p.v_strides = _c_i64x3(*v.stride()[:3])
    p.o_strides = _c_i64x3(*o.stride()[:3])
    p.B, p.T, p.H_q, p.H_kv, p.d_h = B, T, Hq, k.shape[2], D
    p.window_left, p.window_right = int(window_left), int(window_right)
    p.scale = float(scale)
    p.global_idx = None if global_idx is None else global_idx.data_ptr()
    p.n_global = 0 if global_idx is None else int(global_idx.numel())
    p.lse = lse.data_ptr()
    p.row_counts = None if row_counts is None else row_counts.data_ptr()
    p.global_mode = int(global_mode)
    if qkv_g is not None:
        qg, kg, vg = qkv_g
        p.q_g, p.k_g, p.v_g = qg.data_ptr(), kg.data_ptr(), vg.data_ptr()
        p.qg_strides = _c_i64x3(*qg.stride()[:3])
        p.kg_strides = _c_i64x3(*kg.stride()[:3])
        p.vg_strides = _c_i64x3(*vg.stride()[:3])
    if dilation is not None:
        arr = (ctypes.c_int32 * Hq)(*[int(x) for x in dilation])
        p._dilation_keepalive = arr  # the C call reads it through the pointer
        p.dilation = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
    return p


def swa_fwd_workspace_size(params: SwaFwdParams) -> int:
    return int(load_library().swa_fwd_workspace_size(ctypes.byref(params)))


def swa_fwd(q, k, v, window_left: int, window_right: int, scale: float | None = None, global_idx=None, *,
            o=None, lse=None, row_counts=None, want_counts: bool = False, workspace=None, stream=None,
            global_mode: int = GLOBAL_FULL, q_g=None, k_g=None, v_g=None, dilation=None):
    """Banded attention over q [B,T,H_q,d], k/v [B,T,H_kv,d] (bf16, CUDA).

    Keys s with t - window_left <= s <= t + window_right (negative: unbounded side),
    plus global positions (int32 CUDA tensor, strictly increasing) used as
    global_mode says (GLOBAL_FULL rows and columns, GLOBAL_SINK pinned columns).
    q_g, k_g, v_g: separate global projections (shapes of q, k, v).  dilation:
    per-query-head band dilations (ints >= 1; window sides then count steps).
    Returns (o [B,T,H_q,d] bf16, lse [B,H_q,T] fp32, row_counts [B,H_q,T] int32 or None).
    """
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(name, t, 4)
    B, T, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    if global_idx is not None:
        if global_idx.dtype != torch.int32 or not global_idx.is_cuda:
            raise ValueError("global_idx: expected a CUDA int32 tensor")
        global_idx = global_idx.contiguous()
        if global_idx.numel() == 0:
            global_idx = None
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    if row_counts is None and want_counts:
        row_counts = torch.empty((B, Hq, T), dtype=torch.int32, device=q.device)
    qkv_g = None
    if q_g is not None or k_g is not None or v_g is not None:
        if q_g is None or k_g is None or v_g is None:
            raise ValueError("q_g, k_g and v_g go together")
        for name, t, ref in (("q_g", q_g, q), ("k_g", k_g, k), ("v_g", v_g, v)):
            _check_bf16(name, t, 4)
            if t.shape != ref.shape:
                raise ValueError(f"{name}: expected shape {tuple(ref.shape)}")
        qkv_g = (q_g, k_g, v_g)
    if dilation is not None and len(dilation) != Hq:
        raise ValueError(f"dilation: expected {Hq} entries")
    p = fwd_params(q, k, v, window_left, window_right, scale, global_idx, o, lse, row_counts, global_mode, qkv_g,
                   dilation)
    need = int(lib.swa_fwd_workspace_size(ctypes.byref(p)))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _ptr(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.swa_fwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream_handle(stream))
    if st != 0:
        raise SwaError("swa_fwd", st)
    return o, lse, row_counts


def decode_params(q, k_cache, v_cache, slot_pos, q_pos, scale: float, o, lse, row_counts, window: int = 0,
                  n_sink: int = 0):
    B, Hq, D = q.shape
    p = SwaDecodeParams()
    p.q, p.k_cache, p.v_cache = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr()
    p.slot_pos, p.q_pos = slot_pos.data_ptr(), q_pos.data_ptr()
    p.B, p.H_q, p.H_kv, p.d_h, p.W = B, Hq, k_cache.shape[1], D, k_cache.shape[2]
    p.scale = float(scale)
    p.o, p.lse = o.data_ptr(), lse.data_ptr()
    p.row_counts = None if row_counts is None else row_counts.data_ptr()
    p.window, p.n_sink = int(window), int(n_sink)
    return p


def swa_decode_workspace_size(params: SwaDecodeParams) -> int:
    return int(load_library().swa_decode_workspace_size(ctypes.byref(params)))


def swa_decode(q, k_cache, v_cache, slot_pos, q_pos, scale: float | None = None, *, o=None, lse=None,
               row_counts=None, want_counts: bool = False, workspace=None, stream=None, window: int = 0,
               n_sink: int = 0):
    """Ring-buffer decode: q [B,H_q,d], caches [B,H_kv,W,d] (bf16), slot_pos [B,W], q_pos [B] (int32).

    window: the window in positions (0: the number of slots W); n_sink: the first
    positions that are always attended.  Returns (o [B,H_q,d] bf16, lse [B,H_q] fp32,
    row_counts [B,H_q] int32 or None).
    """
    import torch

    lib = load_library()
    _check_bf16("q", q, 3)
    _check_bf16("k_cache", k_cache, 4)
    _check_bf16("v_cache", v_cache, 4)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("slot_pos", slot_pos), ("q_pos", q_pos)):
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
    if slot_pos.dtype != torch.int32 or q_pos.dtype != torch.int32:
        raise ValueError("slot_pos and q_pos must be int32")
    B, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    if row_counts is None and want_counts:
        row_counts = torch.empty((B, Hq), dtype=torch.int32, device=q.device)
    p = decode_params(q, k_cache, v_cache, slot_pos, q_pos, scale, o, lse, row_counts, window, n_sink)
    need = int(lib.swa_decode_workspace_size(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.swa_decode(ctypes.byref(p), _ptr(workspace), ws_bytes, _stream_handle(stream))
    if st != 0:
        raise SwaError("swa_decode", st)
    return o, lse, row_counts


def cache_params(k_cache, v_cache, slot_pos, n_sink: int = 0) -> SwaCacheParams:
    """caches bf16 [B,H_kv,n_slots,d] and slot_pos int32 [B,n_slots] (contiguous, CUDA)."""
    c = SwaCacheParams()
    c.k_cache, c.v_cache, c.slot_pos = k_cache.data_ptr(), v_cache.data_ptr(), slot_pos.data_ptr()
    c.B, c.H_kv, c.n_slots, c.d_h = k_cache.shape
    c.n_sink = int(n_sink)
    return c


def _check_cache(k_cache, v_cache, slot_pos):
    import torch

    _check_bf16("k_cache", k_cache, 4)
    _check_bf16("v_cache", v_cache, 4)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("slot_pos", slot_pos)):
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
    if slot_pos.dtype != torch.int32 or v_cache.shape != k_cache.shape or tuple(slot_pos.shape) != tuple(k_cache.shape[::2]):
        raise ValueError("slot_pos: expected int32 [B, n_slots] matching the caches")


def swa_cache_append(k_cache, v_cache, slot_pos, k_new, v_new, p0, *, n_sink: int = 0, stream=None) -> None:
    """Append k_new/v_new [B,n,H_kv,d] (positions p0[b] + i, p0 int32 CUDA [B]) to the
    ring cache in place (slot rule of include/swa.h with n_sink pinned sinks)."""
    import torch

    _check_cache(k_cache, v_cache, slot_pos)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _check_bf16(name, t, 4)
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
    if p0.dtype != torch.int32 or not p0.is_contiguous():
        raise ValueError("p0: expected a contiguous int32 tensor")
    c = cache_params(k_cache, v_cache, slot_pos, n_sink)
    st = load_library().swa_cache_append(ctypes.byref(c), _ptr(k_new), _ptr(v_new), int(k_new.shape[1]), _ptr(p0),
                                         _stream_handle(stream))
    if st != 0:
        raise SwaError("swa_cache_append", st)


def swa_decode_append(q, k_cache, v_cache, slot_pos, q_pos, k_new, v_new, scale: float | None = None, *, o=None,
                      lse=None, want_counts: bool = False, workspace=None, stream=None, window: int = 0,
                      n_sink: int = 0):
    """swa_decode with the current token's k_new/v_new [B,H_kv,d] appended to the cache
    (in place) in the same pass.  Returns (o, lse, row_counts or None)."""
    import torch

    lib = load_library()
    _check_bf16("q", q, 3)
    _check_cache(k_cache, v_cache, slot_pos)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _check_bf16(name, t, 3)
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
    B, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    row_counts = torch.empty((B, Hq), dtype=torch.int32, device=q.device) if want_counts else None
    p = decode_params(q, k_cache, v_cache, slot_pos, q_pos, scale, o, lse, row_counts, window, n_sink)
    need = int(lib.swa_decode_workspace_size(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib.swa_decode_append(ctypes.byref(p), _ptr(k_new), _ptr(v_new), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != 0:
        raise SwaError("swa_decode_append", st)
    return o, lse, row_counts


def chunk_params(q, k_new, v_new, p0, window: int, scale: float, o, lse, row_counts, append: bool) -> SwaChunkParams:
    B, C, Hq, D = q.shape
    p = SwaChunkParams()
    p.q, p.k_new, p.v_new, p.p0 = q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), p0.data_ptr()
    p.B, p.C, p.H_q, p.H_kv, p.d_h = B, C, Hq, k_new.shape[2], D
    p.window, p.scale = int(window), float(scale)
    p.o, p.lse = o.data_ptr(), lse.data_ptr()
    p.row_counts = None if row_counts is None else row_counts.data_ptr()
    p.append = 1 if append else 0
    return p


def swa_prefill_chunk(q, k_new, v_new, k_cache, v_cache, slot_pos, p0, window: int, scale: float | None = None, *,
                      append: bool = False, o=None, lse=None, want_counts: bool = False, workspace=None,
                      stream=None, n_sink: int = 0):
    """Chunked prefill: q [B,C,H_q,d] and the chunk's k_new/v_new [B,C,H_kv,d] at positions
    p0[b] + i attend to the ring cache's history and to the chunk (causal window), and to
    the cache's n_sink pinned sinks.  append: afterwards the chunk joins the cache.  Returns (o [B,C,H_q,d], lse [B,H_q,C],
    row_counts or None)."""
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new)):
        _check_bf16(name, t, 4)
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
    _check_cache(k_cache, v_cache, slot_pos)
    if p0.dtype != torch.int32 or not p0.is_contiguous():
        raise ValueError("p0: expected a contiguous int32 tensor")
    B, C, Hq, D = q.shape
    if scale is None:
        scale = D ** -0.5
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, C), dtype=torch.float32, device=q.device) if lse is None else lse
    row_counts = torch.empty((B, Hq, C), dtype=torch.int32, device=q.device) if want_counts else None
    p = chunk_params(q, k_new, v_new, p0, window, scale, o, lse, row_counts, append)
    c = cache_params(k_cache, v_cache, slot_pos, n_sink)
    need = int(lib.swa_prefill_chunk_workspace_size(ctypes.byref(p), ctypes.byref(c)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib.swa_prefill_chunk(ctypes.byref(p), ctypes.byref(c), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != 0:
        raise SwaError("swa_prefill_chunk", st)
    return o, lse, row_counts


def swa_check_device_error(stream=None) -> None:
    """Synchronise the stream and raise if a kernel gave up on a bounded wait or found
    device data breaking its contract."""
    st = load_library().swa_check_device_error(_stream_handle(stream))
    if st != 0:
        raise SwaError("swa_check_device_error", st)


def swa_read_device_errors(stream=None) -> tuple[int, dict]:
    """Synchronise the stream, read and clear the device error words: (status, words)
    with words = {"prefill": bits, "split": bits, "cache": bits}."""
    e = SwaDeviceErrors()
    st = load_library().swa_read_device_errors(_stream_handle(stream), ctypes.byref(e))
    return int(st), {"prefill": int(e.prefill), "split": int(e.split), "cache": int(e.cache)}


def swa_debug_set_faults(band_stop_fill: int = -1, split_stop_stage: int = -1) -> None:
    """Failure-detection test hook (process-wide): the prefill kernel's producer stops
    before ring fill band_stop_fill, the split pass's before stage split_stop_stage
    (-1: off).  Called with no arguments it restores normal operation."""
    f = SwaDebugFaults(int(band_stop_fill), int(split_stop_stage))
    st = load_library().swa_debug_set_faults(ctypes.byref(f))
    if st != 0:
        raise SwaError("swa_debug_set_faults", st)
