"""Seeded synthetic inputs for sliding-window attention workloads.

This module is shared by the CUDA path's callers (tests, bench, smoke) and by
the CPU oracle's callers.  It holds no attention arithmetic: only a
counter-based random stream, the normal transform, rounding to bf16, the
rotary position transform that the Gemma-3 local-layer workload pre-applies
to q/k, and the ring-buffer cache layout of the decode workload.

Random stream: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Draw i of stream `seed` is
mix(seed + (i + 1) * 0x9E3779B97F4A7C15).  It is evaluated with numpy uint64
arithmetic, so the same seed gives the same bits on x86 and on Arm.

Normals: Box-Muller on pairs of draws, in float64, rounded once to float32
(scaled in float32 when a scale is asked for), then rounded to bf16 with
round-to-nearest-even.  All tensors are returned as uint16 arrays holding
bf16 bit patterns.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21  # pairs per chunk; bounds per-thread temporaries to ~100 MB


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Draws start .. start+n-1 of the SplitMix64 stream `seed` (uint64)."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_chunk(seed: int, p0: int, p1: int) -> np.ndarray:
    """Normals 2*p0 .. 2*p1-1 of stream `seed` (Box-Muller on draw pairs), float32."""
    z = splitmix64(seed, 2 * p0, 2 * (p1 - p0))
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    rad = np.sqrt(-2.0 * np.log(u1))
    ang = (2.0 * math.pi) * u2
    pair = np.empty((p1 - p0, 2), dtype=np.float64)
    pair[:, 0] = rad * np.cos(ang)
    pair[:, 1] = rad * np.sin(ang)
    return pair.reshape(-1).astype(np.float32)


def normal_f32(seed: int, n: int) -> np.ndarray:
    """n iid N(0,1) values as float32 from stream `seed` (Box-Muller pairs).

    The stream is counter-based, so chunks are generated independently on a
    thread pool; the result does not depend on the number of threads.
    """
    out = np.empty(n, dtype=np.float32)
    npairs = (n + 1) // 2
    bounds = [(p0, min(npairs, p0 + _CHUNK)) for p0 in range(0, npairs, _CHUNK)]

    def work(b):
        p0, p1 = b
        flat = _normal_chunk(seed, p0, p1)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = flat[: hi - lo]

    if len(bounds) <= 1:
        for b in bounds:
            work(b)
    else:
        workers = min(len(bounds), os.cpu_count() or 1, 32)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, bounds))
    return out


def normal_bf16(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """iid N(0,1) * scale rounded to bf16, as uint16 bits of the given shape."""
    n = int(np.prod(shape))
    x = normal_f32(seed, n)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x).reshape(shape)


def uniform_int(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (inclusive) from stream `seed` (multiply-shift)."""
    z = splitmix64(seed, 0, n)
    span = np.uint64(hi - lo + 1)
    # (z >> 32) * span >> 32 maps the top 32 bits onto [0, span) with negligible bias.
    with np.errstate(over="ignore"):
        v = ((z >> np.uint64(32)) * span) >> np.uint64(32)
    return (v.astype(np.int64) + lo)


def rope_rotate_half_f32(x: np.ndarray, base: float) -> np.ndarray:
    """Rotary position transform over x[..., T, H, d] (token axis -3), rotate-half pairing.

    Pair (i, i + d/2) is rotated by angle t * base**(-2i/d) for token t.  The pages
    give only the base (1e4 on local layers); the pairing and frequency schedule are
    the common rotate-half convention.  Computed in float64, returned as float32.
    """
    T, H, d = x.shape[-3], x.shape[-2], x.shape[-1]
    half = d // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.arange(T, dtype=np.float64)[:, None] * inv[None, :]  # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x64 = x.astype(np.float64)
    a = x64[..., :half]
    b = x64[..., half:]
    out = np.empty_like(x64)
    out[..., :half] = a * c - b * s
    out[..., half:] = b * c + a * s
    return out.astype(np.float32)


# --------------------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------------------


@dataclass(frozen=True)
class PrefillConfig:
    """A prefill / encoder workload: Q [B,T,Hq,d], K/V [B,T,Hkv,d] bf16."""

    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    window_left: int  # keys s >= t - window_left (-1: unbounded)
    window_right: int  # keys s <= t + window_right (-1: unbounded)
    globals_: tuple = ()
    qkv_scale: float = 1.0
    rope_base: float = 0.0  # 0: no rotary transform
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclass(frozen=True)
class DecodeConfig:
    """A ring-buffer decode workload: one query token per sequence."""

    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    W: int
    max_len: int
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def causal(W: int) -> tuple:
    """Causal window of W keys including the query: t - W < s <= t."""
    return (W - 1, 0)


def bidirectional(r: int) -> tuple:
    """Symmetric window |t - s| <= r."""
    return (r, r)


# The five workloads (sizes, windows, distributions) that the measurements and
# parity cases use.  Seeds are per workload; each tensor draws its own stream.
TINY_BIDIR = PrefillConfig("tiny-bidirectional-r2", 1, 16, 1, 1, 64, *bidirectional(2), seed=16)
TINY_CAUSAL = PrefillConfig("tiny-causal-W4", 1, 16, 1, 1, 64, *causal(4), seed=17)
MISTRAL = PrefillConfig("mistral7b-causal-prefill", 1, 16384, 32, 8, 128, *causal(4096), qkv_scale=0.5, seed=32)
GEMMA_LOCAL = PrefillConfig("gemma3-local-causal-prefill", 2, 32768, 16, 8, 256, *causal(1024), rope_base=1e4, seed=48)
LONGFORMER = PrefillConfig("longformer-bidirectional-encoder", 8, 4096, 12, 12, 64, *bidirectional(256),
                           globals_=(0, 2048), seed=64)
DECODE = DecodeConfig("ring-buffer-decode", 64, 32, 8, 128, 4096, 131072, seed=80)


def prefill_inputs(cfg: PrefillConfig):
    """(q, k, v) uint16 bf16 bits, shapes [B,T,Hq,d], [B,T,Hkv,d], [B,T,Hkv,d]."""
    qs = (cfg.B, cfg.T, cfg.Hq, cfg.d)
    ks = (cfg.B, cfg.T, cfg.Hkv, cfg.d)
    out = []
    for tid, shape in enumerate((qs, ks, ks)):
        seed = cfg.seed * 16 + tid
        if cfg.rope_base and tid < 2:
            x = normal_f32(seed, int(np.prod(shape))).reshape(shape)
            x = rope_rotate_half_f32(x, cfg.rope_base)
            out.append(f32_to_bf16_bits(x).reshape(shape))
        else:
            out.append(normal_bf16(seed, shape, cfg.qkv_scale))
    return tuple(out)


def decode_lengths(cfg: DecodeConfig) -> np.ndarray:
    """Per-sequence context length L_b, uniform on [1, max_len]."""
    return uniform_int(cfg.seed * 16 + 5, cfg.B, 1, cfg.max_len)


def ring_slot_positions(L: np.ndarray, W: int) -> np.ndarray:
    """True token position held by each ring-buffer slot, int32 [B, W].

    Token p lives in slot p mod W and overwrites older tokens there.  With
    t = L - 1 the current (already appended) token:
      * L >= W: slot j holds the unique p in (t - W, t] with p = j (mod W);
      * L <  W: slots j < L hold p = j; slots j >= L are stale and hold -1
        (never written) for odd j and L + j (a position after t) for even j,
        so that both validity guards of a decode kernel are exercised.
    """
    B = L.shape[0]
    j = np.arange(W, dtype=np.int64)[None, :]
    t = (L - 1).astype(np.int64)[:, None]
    full = t - ((t - j) % W)  # largest p <= t with p = j (mod W)
    short = np.where(j < L[:, None], j, np.where(j % 2 == 1, -1, L[:, None] + j))
    pos = np.where(L[:, None] >= W, full, short)
    assert pos.shape == (B, W)
    return pos.astype(np.int32)


def sink_ring_slot_positions(L: np.ndarray, W: int, n_sink: int) -> np.ndarray:
    """Slot positions of a cache with n_sink pinned slots and a W-slot ring, int32 [B, n_sink + W].

    Slots 0 .. n_sink-1 hold positions 0 .. n_sink-1 (those below L); position
    p >= n_sink lives in slot n_sink + (p - n_sink) mod W, and the ring holds the
    last W positions of the sequence (t = L - 1) that are not sinks.  Slots never
    written hold -1.
    """
    B = L.shape[0]
    pos = np.full((B, n_sink + W), -1, dtype=np.int64)
    j = np.arange(n_sink)[None, :]
    pos[:, :n_sink] = np.where(j < L[:, None], j, -1)
    r = np.arange(W)[None, :]
    t = (L - 1).astype(np.int64)[:, None]
    # largest p <= t with p >= n_sink and (p - n_sink) = r (mod W)
    p = t - ((t - n_sink - r) % W)
    ok = (p >= n_sink) & (p > t - W)
    pos[:, n_sink:] = np.where(ok, p, -1)
    return pos.astype(np.int32)


def decode_inputs(cfg: DecodeConfig):
    """(q [B,Hq,d], k_cache [B,Hkv,W,d], v_cache [B,Hkv,W,d], slot_pos [B,W], q_pos [B])."""
    L = decode_lengths(cfg)
    q = normal_bf16(cfg.seed * 16 + 0, (cfg.B, cfg.Hq, cfg.d))
    kc = normal_bf16(cfg.seed * 16 + 1, (cfg.B, cfg.Hkv, cfg.W, cfg.d))
    vc = normal_bf16(cfg.seed * 16 + 2, (cfg.B, cfg.Hkv, cfg.W, cfg.d))
    return q, kc, vc, ring_slot_positions(L, cfg.W), (L - 1).astype(np.int32)
