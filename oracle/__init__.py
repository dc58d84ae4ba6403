"""CPU oracle for sliding-window attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA path (it never imports
the product package) and the product never imports it.

Two independent restatements of the definition live here:

* ``fwd`` / ``decode``: the fp64 C oracle (``swa_oracle.c``) -- an explicit mask
  row per query, then a masked softmax over the allowed keys;
* ``dense_bruteforce``: a numpy transcription of the pages' dense sketch (full
  [T, T] score grid, -inf outside the mask, row softmax, times V), for tiny T.

Inputs are uint16 arrays of bf16 bit patterns; outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libswa_oracle.so")
_lib = None

_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_P = ctypes.c_void_p


def build(force: bool = False, extra_flags=(), out_path: str | None = None) -> str:
    """Compile swa_oracle.c with gcc (-O2, OpenMP, no fast-math)."""
    out = out_path or _LIB_PATH
    src = os.path.join(_HERE, "swa_oracle.c")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


def _bind(lib):
    lib.swa_oracle_mask_row.argtypes = [_I64, _I64, _I32, _I32, _P, _I64, _P]
    lib.swa_oracle_mask_row.restype = None
    lib.swa_oracle_fwd.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I32, _I32, ctypes.c_double,
                                   _P, _I64, _P, _I64, _P, _P, _P]
    lib.swa_oracle_fwd.restype = ctypes.c_int
    lib.swa_oracle_decode.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
                                      _P, _P, _P]
    lib.swa_oracle_decode.restype = ctypes.c_int
    lib.swa_oracle_num_threads.argtypes = []
    lib.swa_oracle_num_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; a path loads a variant build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _globals(G):
    if G is None or len(G) == 0:
        return None, 0
    g = np.ascontiguousarray(np.asarray(G, dtype=np.int32))
    return g, g.shape[0]


def mask_row(T: int, t: int, wl: int, wr: int, G=None, lib=None) -> np.ndarray:
    """Explicit mask row of query t (bool [T])."""
    lib = lib or load()
    g, ng = _globals(G)
    out = np.zeros(max(T, 1), dtype=np.uint8)
    lib.swa_oracle_mask_row(T, t, wl, wr, _ptr(g), ng, _ptr(out))
    return out[:T].astype(bool)


def fwd(q, k, v, wl: int, wr: int, scale: float, G=None, rows=None, lib=None):
    """Prefill / encoder oracle.

    q [B,T,Hq,D], k/v [B,T,Hkv,D] bf16 bits.  rows: optional int array [n, 3] of
    (b, h, t).  Returns (o, lse, counts): o [B,Hq,T,D] / lse [B,Hq,T] /
    counts [B,Hq,T] when rows is None, else o [n,D] / lse [n] / counts [n].
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, D) and v.shape == k.shape
    g, ng = _globals(G)
    if rows is None:
        n = B * Hq * T
        r = None
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = r.shape[0]
    o = np.zeros((max(n, 1), D), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    cnt = np.zeros(max(n, 1), dtype=np.int64)
    rc = lib.swa_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, T, Hq, Hkv, D, wl, wr, float(scale), _ptr(g), ng,
                            _ptr(r), n, _ptr(o), _ptr(lse), _ptr(cnt))
    if rc != 0:
        raise ValueError("swa_oracle_fwd rejected its arguments")
    o, lse, cnt = o[:n], lse[:n], cnt[:n]
    if rows is None:
        return o.reshape(B, Hq, T, D), lse.reshape(B, Hq, T), cnt.reshape(B, Hq, T)
    return o, lse, cnt


def decode(q, k_cache, v_cache, slot_pos, q_pos, scale: float, lib=None):
    """Ring-buffer decode oracle: returns o [B,Hq,D], lse [B,Hq], counts [B,Hq]."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint16)
    sp = np.ascontiguousarray(slot_pos, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int32)
    B, Hq, D = q.shape
    _, Hkv, W, _ = kc.shape
    o = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    cnt = np.zeros((B, Hq), dtype=np.int64)
    rc = lib.swa_oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(sp), _ptr(qp), B, Hq, Hkv, D, W, float(scale),
                               _ptr(o), _ptr(lse), _ptr(cnt))
    if rc != 0:
        raise ValueError("swa_oracle_decode rejected its arguments")
    return o, lse, cnt


def num_threads(lib=None) -> int:
    return int((lib or load()).swa_oracle_num_threads())


# --------------------------------------------------------------------------------------
# Dense brute force (numpy), tiny T only.
# --------------------------------------------------------------------------------------


def _widen(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def dense_mask(T: int, wl: int, wr: int, G=None) -> np.ndarray:
    """Bool [T, T] connectivity: the banded mask built densely on the index grid.

    Rows are queries t, columns keys s.  Band: s >= t - wl (unless wl < 0) and
    s <= t + wr (unless wr < 0); a global position opens its whole row and column.
    """
    t_idx = np.arange(T).reshape(T, 1)
    s_idx = np.arange(T).reshape(1, T)
    left = np.ones((T, T), dtype=bool) if wl < 0 else (s_idx >= t_idx - wl)
    right = np.ones((T, T), dtype=bool) if wr < 0 else (s_idx <= t_idx + wr)
    mask = left & right
    if G is not None and len(G):
        g = np.zeros(T, dtype=bool)
        g[np.asarray(G, dtype=np.int64)] = True
        mask = mask | g[:, None] | g[None, :]
    return mask


def dense_bruteforce(q, k, v, wl: int, wr: int, scale: float, G=None):
    """Full-grid masked attention in fp64: scores = scale*QK^T, -inf off the mask,
    row softmax, times V.  Returns o [B,Hq,T,D], lse [B,Hq,T], counts [B,Hq,T]."""
    qd, kd, vd = _widen(q), _widen(k), _widen(v)
    B, T, Hq, D = qd.shape
    Hkv = kd.shape[2]
    grp = Hq // Hkv
    mask = dense_mask(T, wl, wr, G)
    o = np.zeros((B, Hq, T, D))
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            Q = qd[b, :, h, :]
            K = kd[b, :, h // grp, :]
            V = vd[b, :, h // grp, :]
            scores = (Q @ K.T) * scale
            scores = np.where(mask, scores, -np.inf)
            m = scores.max(axis=1, keepdims=True)
            e = np.exp(scores - m)
            l = e.sum(axis=1, keepdims=True)
            o[b, h] = (e / l) @ V
            lse[b, h] = (m + np.log(l))[:, 0]
    counts = np.broadcast_to(mask.sum(axis=1), (B, Hq, T)).astype(np.int64)
    return o, lse, counts
