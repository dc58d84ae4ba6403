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
    lib.swa_oracle_mask_row_ex.argtypes = [_I64, _I64, _I32, _I32, _I32, _P, _I64, _I32, _P]
    lib.swa_oracle_mask_row_ex.restype = None
    lib.swa_oracle_fwd_ex.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I32, _I32, _P,
                                      ctypes.c_double, _P, _I64, _I32, _P, _I64, _P, _P, _P]
    lib.swa_oracle_fwd_ex.restype = ctypes.c_int
    lib.swa_oracle_decode_ex.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                         ctypes.c_double, _P, _P, _P]
    lib.swa_oracle_decode_ex.restype = ctypes.c_int
    lib.swa_oracle_cache_append.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _I64, _P]
    lib.swa_oracle_cache_append.restype = ctypes.c_int
    lib.swa_oracle_cache_append_ex.argtypes = [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P, _I64, _P]
    lib.swa_oracle_cache_append_ex.restype = ctypes.c_int
    lib.swa_oracle_chunk.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
                                     ctypes.c_double, _P, _P, _P]
    lib.swa_oracle_chunk.restype = ctypes.c_int
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


GLOBAL_FULL = 0  # global positions: full rows and columns (Longformer)
GLOBAL_SINK = 1  # pinned key columns only, never right of the band (attention sinks)


def mask_row(T: int, t: int, wl: int, wr: int, G=None, lib=None, dil: int = 1,
             gmode: int = GLOBAL_FULL) -> np.ndarray:
    """Explicit mask row of query t (bool [T]); dil: band dilation, gmode: global mode."""
    lib = lib or load()
    g, ng = _globals(G)
    out = np.zeros(max(T, 1), dtype=np.uint8)
    if dil == 1 and gmode == GLOBAL_FULL:
        lib.swa_oracle_mask_row(T, t, wl, wr, _ptr(g), ng, _ptr(out))
    else:
        lib.swa_oracle_mask_row_ex(T, t, wl, wr, dil, _ptr(g), ng, gmode, _ptr(out))
    return out[:T].astype(bool)


def _bits(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint16)


def fwd(q, k, v, wl: int, wr: int, scale: float, G=None, rows=None, lib=None, dilation=None,
        gmode: int = GLOBAL_FULL, qg=None, kg=None, vg=None):
    """Prefill / encoder oracle.

    q [B,T,Hq,D], k/v [B,T,Hkv,D] bf16 bits.  rows: optional int array [n, 3] of
    (b, h, t).  dilation: per-query-head band dilation [Hq] (None: 1).  gmode:
    GLOBAL_FULL or GLOBAL_SINK for the positions G.  qg/kg/vg: separate global
    projections (GLOBAL_FULL only).  Returns (o, lse, counts): o [B,Hq,T,D] / lse
    [B,Hq,T] / counts [B,Hq,T] when rows is None, else o [n,D] / lse [n] / counts [n].
    """
    lib = lib or load()
    q, k, v = _bits(q), _bits(k), _bits(v)
    qg, kg, vg = _bits(qg), _bits(kg), _bits(vg)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, D) and v.shape == k.shape
    if qg is not None:
        assert qg.shape == q.shape and kg.shape == k.shape and vg.shape == k.shape
    g, ng = _globals(G)
    dil = None if dilation is None else np.ascontiguousarray(np.asarray(dilation, dtype=np.int32))
    if dil is not None:
        assert dil.shape == (Hq,)
    if rows is None:
        n = B * Hq * T
        r = None
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = r.shape[0]
    o = np.zeros((max(n, 1), D), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    cnt = np.zeros(max(n, 1), dtype=np.int64)
    if dil is None and gmode == GLOBAL_FULL and qg is None:
        rc = lib.swa_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, T, Hq, Hkv, D, wl, wr, float(scale), _ptr(g), ng,
                                _ptr(r), n, _ptr(o), _ptr(lse), _ptr(cnt))
    else:
        rc = lib.swa_oracle_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(qg), _ptr(kg), _ptr(vg), B, T, Hq, Hkv, D, wl,
                                   wr, _ptr(dil), float(scale), _ptr(g), ng, gmode, _ptr(r), n, _ptr(o), _ptr(lse),
                                   _ptr(cnt))
    if rc != 0:
        raise ValueError("swa_oracle_fwd rejected its arguments")
    o, lse, cnt = o[:n], lse[:n], cnt[:n]
    if rows is None:
        return o.reshape(B, Hq, T, D), lse.reshape(B, Hq, T), cnt.reshape(B, Hq, T)
    return o, lse, cnt


def decode(q, k_cache, v_cache, slot_pos, q_pos, scale: float, lib=None, window=None, n_sink: int = 0):
    """Ring-buffer decode oracle: returns o [B,Hq,D], lse [B,Hq], counts [B,Hq].

    The caches hold S slots; window (default S) is the window W in positions and
    n_sink the number of pinned first positions."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint16)
    sp = np.ascontiguousarray(slot_pos, dtype=np.int32)
    qp = np.ascontiguousarray(q_pos, dtype=np.int32)
    B, Hq, D = q.shape
    _, Hkv, S, _ = kc.shape
    o = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    cnt = np.zeros((B, Hq), dtype=np.int64)
    if window is None and n_sink == 0:
        rc = lib.swa_oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(sp), _ptr(qp), B, Hq, Hkv, D, S, float(scale),
                                   _ptr(o), _ptr(lse), _ptr(cnt))
    else:
        rc = lib.swa_oracle_decode_ex(_ptr(q), _ptr(kc), _ptr(vc), _ptr(sp), _ptr(qp), B, Hq, Hkv, D, S,
                                      S if window is None else window, n_sink, float(scale), _ptr(o), _ptr(lse),
                                      _ptr(cnt))
    if rc != 0:
        raise ValueError("swa_oracle_decode rejected its arguments")
    return o, lse, cnt


def cache_append(k_cache, v_cache, slot_pos, k_new, v_new, p0, lib=None, n_sink: int = 0):
    """Ring append on copies: returns (k_cache, v_cache, slot_pos) after writing the n
    tokens of k_new/v_new [B,n,Hkv,D] at positions p0[b] + i into slots p mod S (with
    n_sink pinned sinks: slot p below n_sink, n_sink + (p - n_sink) mod (S - n_sink) else)."""
    lib = lib or load()
    kc = np.array(k_cache, dtype=np.uint16, order="C", copy=True)
    vc = np.array(v_cache, dtype=np.uint16, order="C", copy=True)
    sp = np.array(slot_pos, dtype=np.int32, order="C", copy=True)
    kn, vn = _bits(k_new), _bits(v_new)
    p = np.ascontiguousarray(p0, dtype=np.int32)
    B, Hkv, S, D = kc.shape
    n = kn.shape[1]
    assert kn.shape == (B, n, Hkv, D) and vn.shape == kn.shape and p.shape == (B,)
    if n_sink == 0:
        rc = lib.swa_oracle_cache_append(_ptr(kc), _ptr(vc), _ptr(sp), B, Hkv, S, D, _ptr(kn), _ptr(vn), n, _ptr(p))
    else:
        rc = lib.swa_oracle_cache_append_ex(_ptr(kc), _ptr(vc), _ptr(sp), B, Hkv, S, D, n_sink, _ptr(kn), _ptr(vn),
                                            n, _ptr(p))
    if rc != 0:
        raise ValueError("swa_oracle_cache_append rejected its arguments")
    return kc, vc, sp


def chunk(q, k_new, v_new, k_cache, v_cache, slot_pos, p0, window: int, scale: float, n_sink: int = 0, lib=None):
    """Chunked prefill against a ring cache: o [B,Hq,C,D], lse [B,Hq,C], counts [B,Hq,C]."""
    lib = lib or load()
    q, kn, vn = _bits(q), _bits(k_new), _bits(v_new)
    kc, vc = _bits(k_cache), _bits(v_cache)
    sp = np.ascontiguousarray(slot_pos, dtype=np.int32)
    p = np.ascontiguousarray(p0, dtype=np.int32)
    B, C, Hq, D = q.shape
    _, Hkv, S, _ = kc.shape
    o = np.zeros((B, Hq, max(C, 1), D), dtype=np.float64)
    lse = np.zeros((B, Hq, max(C, 1)), dtype=np.float64)
    cnt = np.zeros((B, Hq, max(C, 1)), dtype=np.int64)
    rc = lib.swa_oracle_chunk(_ptr(q), _ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sp), _ptr(p), B, C, Hq, Hkv, D,
                              S, window, n_sink, float(scale), _ptr(o), _ptr(lse), _ptr(cnt))
    if rc != 0:
        raise ValueError("swa_oracle_chunk rejected its arguments")
    return o[:, :, :C], lse[:, :, :C], cnt[:, :, :C]


def num_threads(lib=None) -> int:
    return int((lib or load()).swa_oracle_num_threads())


# --------------------------------------------------------------------------------------
# Dense brute force (numpy), tiny T only.
# --------------------------------------------------------------------------------------


def _widen(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def dense_mask(T: int, wl: int, wr: int, G=None, dil: int = 1, gmode: int = GLOBAL_FULL) -> np.ndarray:
    """Bool [T, T] connectivity: the banded mask built densely on the index grid.

    Rows are queries t, columns keys s.  Band: s = t + k*dil for integer k with
    k >= -wl (unless wl < 0) and k <= wr (unless wr < 0).  GLOBAL_FULL: a global
    position opens its whole row and column.  GLOBAL_SINK: a listed position opens
    its column for the rows whose band reaches it from the right (s <= t + wr*dil).
    """
    t_idx = np.arange(T).reshape(T, 1)
    s_idx = np.arange(T).reshape(1, T)
    diff = s_idx - t_idx
    grid = (diff % dil) == 0
    steps = diff // dil
    left = np.ones((T, T), dtype=bool) if wl < 0 else (steps >= -wl)
    right = np.ones((T, T), dtype=bool) if wr < 0 else (steps <= wr)
    mask = grid & left & right
    if G is not None and len(G):
        g = np.zeros(T, dtype=bool)
        g[np.asarray(G, dtype=np.int64)] = True
        if gmode == GLOBAL_FULL:
            mask = mask | g[:, None] | g[None, :]
        else:
            reach = np.ones((T, T), dtype=bool) if wr < 0 else (diff <= wr * dil)
            mask = mask | (g[None, :] & reach)
    return mask


def dense_bruteforce(q, k, v, wl: int, wr: int, scale: float, G=None, dilation=None, gmode: int = GLOBAL_FULL,
                     qg=None, kg=None, vg=None):
    """Full-grid masked attention in fp64: scores = scale*QK^T, -inf off the mask,
    row softmax, times V.  With separate global projections a global row's scores
    are Q_g K_g^T against V_g, and a local row scores global keys with K_g and
    weights V_g.  Returns o [B,Hq,T,D], lse [B,Hq,T], counts [B,Hq,T]."""
    qd, kd, vd = _widen(q), _widen(k), _widen(v)
    sep = qg is not None
    if sep:
        qgd, kgd, vgd = _widen(qg), _widen(kg), _widen(vg)
    B, T, Hq, D = qd.shape
    Hkv = kd.shape[2]
    grp = Hq // Hkv
    is_g = np.zeros(T, dtype=bool)
    if G is not None and len(G):
        is_g[np.asarray(G, dtype=np.int64)] = True
    o = np.zeros((B, Hq, T, D))
    lse = np.zeros((B, Hq, T))
    counts = np.zeros((B, Hq, T), dtype=np.int64)
    for h in range(Hq):
        dil = 1 if dilation is None else int(dilation[h])
        mask = dense_mask(T, wl, wr, G, dil, gmode)
        counts[:, h] = mask.sum(axis=1)
        for b in range(B):
            Q = qd[b, :, h, :]
            K = kd[b, :, h // grp, :]
            V = vd[b, :, h // grp, :]
            if sep:
                Kg, Vg = kgd[b, :, h // grp, :], vgd[b, :, h // grp, :]
                Kmix = np.where(is_g[:, None], Kg, K)
                Vmix = np.where(is_g[:, None], Vg, V)
                scores = (Q @ Kmix.T) * scale
                scores[is_g] = (qgd[b, is_g, h, :] @ Kg.T) * scale
            else:
                scores = (Q @ K.T) * scale
            scores = np.where(mask, scores, -np.inf)
            m = scores.max(axis=1, keepdims=True)
            e = np.exp(scores - m)
            l = e.sum(axis=1, keepdims=True)
            if sep:
                out = (e / l) @ Vmix
                out[is_g] = (e[is_g] / l[is_g]) @ Vg
            else:
                out = (e / l) @ V
            o[b, h] = out
            lse[b, h] = (m + np.log(l))[:, 0]
    return o, lse, counts
