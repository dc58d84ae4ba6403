"""Benchmark: sliding-window attention on one GB300 (or N replicas).

Headline: band-TFLOP/s of swa_fwd on the Mistral-7B-shape causal prefill
(B=1, T=16384, H_q=32, H_kv=8, d=128, W=4096, bf16; FLOPs = 4*d per attended
query-key pair).  The same line carries the ring-buffer decode workload
(64 sequences, W=4096, H_q=32, H_kv=8, d=128; GB/s of algorithmic bytes), the
Gemma-3 local-layer and Longformer encoder workloads, the end-to-end number
through host buffers, the roofline of the dominant kernel, the clocks seen
during the timed region, and the CPU oracle timed on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 the script runs under torch.distributed (one process per GPU); every
rank processes its own copy of the workload (independent units, no data-path
collective) and the whole-job value is N x work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sliding_window_attention_swa_gb300 import inputs as I  # noqa: E402

L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
METRIC = "SWA prefill band-TFLOP/s (Mistral-shape causal prefill); decode GB/s in secondary"


def headline_config(world: int) -> dict:
    """The headline workload's config, identical in both arms."""
    c = I.MISTRAL
    return {"workload": c.name, "B": c.B, "T": c.T, "H_q": c.Hq, "H_kv": c.Hkv, "d_h": c.d,
            "window": c.window_left + 1, "causal": True,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed before every timed step (256 MB write, then 256 MB read: cold, clean L2)", "flops_per_step": prefill_flops(c)}
KERNELS = {"band": "band_fwd_kernel", "split": "stream_attn_kernel", "merge": "merge_kernel"}


# ----------------------------------------------------------------------------- work counts
def prefill_pairs(cfg) -> int:
    """Attended query-key pairs (all batches and query heads), closed form per row."""
    T, wl, wr = cfg.T, cfg.window_left, cfg.window_right
    t = np.arange(T, dtype=np.int64)
    lo = np.zeros(T, dtype=np.int64) if wl < 0 else np.maximum(0, t - wl)
    hi = np.full(T, T - 1, dtype=np.int64) if wr < 0 else np.minimum(T - 1, t + wr)
    cnt = hi - lo + 1
    if cfg.globals_:
        G = np.asarray(cfg.globals_)
        cnt = cnt + ((G[None, :] < lo[:, None]) | (G[None, :] > hi[:, None])).sum(axis=1)
        cnt[G] = T
    return int(cnt.sum()) * cfg.B * cfg.Hq


def prefill_flops(cfg) -> float:
    return 4.0 * cfg.d * prefill_pairs(cfg)


def variant_pairs(cfg, variant) -> int:
    """Attended pairs of a prefill variant, closed form per row: sinks add the sink
    positions left of each row's band; a dilated head of dilation d keeps, of the
    band, the keys of its residue class, min(wl, t//d) + min(wr, (T-1-t)//d) + 1."""
    T, wl, wr = cfg.T, cfg.window_left, cfg.window_right
    t = np.arange(T, dtype=np.int64)
    if variant.get("dilation") is not None:
        total = 0
        for d in variant["dilation"]:
            left = t // d if wl < 0 else np.minimum(wl, t // d)
            right = (T - 1 - t) // d if wr < 0 else np.minimum(wr, (T - 1 - t) // d)
            total += int((left + right + 1).sum())
        return total * cfg.B
    if variant.get("sinks"):
        lo = np.zeros(T, dtype=np.int64) if wl < 0 else np.maximum(0, t - wl)
        hi = np.full(T, T - 1, dtype=np.int64) if wr < 0 else np.minimum(T - 1, t + wr)
        S = np.asarray(variant["sinks"])
        cnt = hi - lo + 1 + (S[None, :] < lo[:, None]).sum(axis=1)
        return int(cnt.sum()) * cfg.B * cfg.Hq
    return prefill_pairs(cfg)


def band_launches(cfg, dilation) -> int:
    """Band-kernel launches of one dilated swa_fwd call: d per run of whole GQA groups
    sharing dilation d, d per head of a group that mixes dilations."""
    if dilation is None or all(x == 1 for x in dilation):
        return 1
    G = cfg.Hq // cfg.Hkv
    groups = [tuple(dilation[g * G:(g + 1) * G]) for g in range(cfg.Hkv)]
    n, prev = 0, None
    for grp in groups:
        if len(set(grp)) > 1:
            n += sum(grp)
            prev = None
        elif grp[0] != prev:
            n += grp[0]
            prev = grp[0]
    return n


def prefill_bytes(cfg) -> int:
    """Algorithmic bytes: Q, K, V read once, O and lse written once."""
    q = cfg.B * cfg.T * cfg.Hq * cfg.d * 2
    kv = 2 * cfg.B * cfg.T * cfg.Hkv * cfg.d * 2
    return q + kv + q + cfg.B * cfg.Hq * cfg.T * 4


def decode_bytes(cfg, L: np.ndarray) -> int:
    """Algorithmic bytes: the valid slots' K and V, all slot positions, q, o, lse."""
    kv = int(np.minimum(L, cfg.W).sum()) * cfg.Hkv * cfg.d * 2 * 2
    return kv + cfg.B * cfg.W * 4 + 2 * cfg.B * cfg.Hq * cfg.d * 2 + cfg.B * cfg.Hq * 4 + cfg.B * 4


def decode_flops(cfg, L: np.ndarray) -> float:
    return 4.0 * cfg.d * int(np.minimum(L, cfg.W).sum()) * cfg.Hq


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], 0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- device timing
def to_dev(bits, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


class L2Flush:
    """Leaves L2 cold before a timed call: a 256 MB write evicts whatever the previous
    call left there, then a 256 MB read evicts the written (dirty) lines in turn, so
    their write-back to HBM happens here and not inside the next call's events."""

    def __init__(self, device):
        import torch

        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=device)
        self.out = torch.empty((), dtype=torch.int64, device=device)

    def zero_(self):
        import torch

        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.out)


def timed_steps(fn, steps: int, warmup: int, flush, stream, sampler=None):
    """W untimed warm-up calls, then K calls each bracketed by CUDA events on `stream`
    with an L2 flush (L2Flush: a 256 MB write, then a 256 MB read) before each call,
    outside its events.  The optional clock sampler runs only around the K timed calls."""
    import torch

    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with (sampler or _Null()):
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    return np.array([a.elapsed_time(b) for a, b in ev])  # ms


def measure_prefill(cfg, steps, warmup, device, flush, sampler=None, variant=None):
    """variant: None, or {"sinks": [...]} (pinned sink columns), {"sep": True} (separate
    global projections q_g, k_g, v_g for cfg's globals), {"dilation": [...]}."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    variant = variant or {}
    q, k, v = I.prefill_inputs(cfg)
    qd, kd, vd = to_dev(q, device), to_dev(k, device), to_dev(v, device)
    extra = {}
    if variant.get("sep"):
        for i, (name, a) in enumerate((("q_g", q), ("k_g", k), ("v_g", v))):
            extra[name] = to_dev(I.normal_bf16(cfg.seed * 16 + 8 + i, a.shape), device)
    del q, k, v
    gl = variant.get("sinks") or list(cfg.globals_)
    g = torch.tensor(gl, dtype=torch.int32, device=device) if gl else None
    gmode = swa.GLOBAL_SINK if variant.get("sinks") else swa.GLOBAL_FULL
    dil = variant.get("dilation")
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq, cfg.T), dtype=torch.float32, device=device)
    qkv_g = (extra["q_g"], extra["k_g"], extra["v_g"]) if extra else None
    p = swa.fwd_params(qd, kd, vd, cfg.window_left, cfg.window_right, cfg.scale, g, o, lse, None, gmode, qkv_g, dil)
    need = swa.swa_fwd_workspace_size(p)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def run():
        swa.swa_fwd(qd, kd, vd, cfg.window_left, cfg.window_right, cfg.scale, g, o=o, lse=lse, workspace=ws,
                    stream=stream, global_mode=gmode, dilation=dil, **extra)

    ms = timed_steps(run, steps, warmup, flush, stream, sampler)
    swa.swa_check_device_error()
    launches = band_launches(cfg, dil) + (2 if (gl and gmode == swa.GLOBAL_FULL) else 0)
    nbytes = prefill_bytes(cfg) + (2 * sum(t.numel() for t in extra.values()) if extra else 0)
    return {"ms": ms, "flops": 4.0 * cfg.d * variant_pairs(cfg, variant), "bytes": nbytes,
            "launches_per_step": launches, "tensors": (qd, kd, vd, g, o, lse, ws)}


def measure_decode(cfg, steps, warmup, device, flush, n_sink: int = 0):
    """n_sink > 0: a cache of n_sink pinned slots plus a W-slot ring (same lengths)."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    q, kc, vc, pos, qpos = I.decode_inputs(cfg)
    L = qpos.astype(np.int64) + 1
    if n_sink:
        pos = I.sink_ring_slot_positions(L, cfg.W, n_sink)
        pad = I.normal_bf16(cfg.seed * 16 + 7, (cfg.B, cfg.Hkv, n_sink, cfg.d))
        kc = np.concatenate([pad, kc], axis=2)
        vc = np.concatenate([pad, vc], axis=2)
    qd, kd, vd = to_dev(q, device), to_dev(kc, device), to_dev(vc, device)
    del kc, vc
    posd = torch.from_numpy(pos).to(device)
    qposd = torch.from_numpy(qpos).to(device)
    o = torch.empty_like(qd)
    lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device=device)
    p = swa.decode_params(qd, kd, vd, posd, qposd, cfg.scale, o, lse, None, cfg.W, n_sink)
    ws = torch.empty(swa.swa_decode_workspace_size(p), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def run():
        swa.swa_decode(qd, kd, vd, posd, qposd, cfg.scale, o=o, lse=lse, workspace=ws, stream=stream,
                       window=cfg.W, n_sink=n_sink)

    ms = timed_steps(run, steps, warmup, flush, stream)
    swa.swa_check_device_error()
    nbytes, flops = decode_bytes(cfg, L), decode_flops(cfg, L)
    if n_sink:
        # the sinks outside the window: their K/V and positions
        extra = int(np.maximum(0, np.minimum(n_sink, L - cfg.W)).sum())
        nbytes += extra * cfg.Hkv * cfg.d * 2 * 2 + cfg.B * n_sink * 4
        flops += 4.0 * cfg.d * extra * cfg.Hq
    return {"ms": ms, "flops": flops, "bytes": nbytes, "launches_per_step": 2}


def measure_cache_paths(steps, warmup, device, flush):
    """The ring-buffer cache paths on the decode and Mistral shapes:
    * chunked prefill: the last 4096 tokens of the Mistral-shape sequence as one chunk
      against a 4096-slot ring holding the 4096 tokens before it (gather + band kernel);
    * append: 512 new tokens for each of the 64 decode sequences (after their lengths);
    * decode with the current token appended in the same pass (decode workload)."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    out = {}
    stream = torch.cuda.current_stream()
    # chunked prefill
    cfg = I.MISTRAL
    W, C = cfg.window_left + 1, 4096
    p0 = cfg.T - C
    q, k, v = I.prefill_inputs(cfg)
    qc = to_dev(q[:, p0:], device)
    kn, vn = to_dev(k[:, p0:], device), to_dev(v[:, p0:], device)
    kh, vh = to_dev(k[:, p0 - W:p0], device), to_dev(v[:, p0 - W:p0], device)
    del q, k, v
    kc = torch.empty((1, cfg.Hkv, W, cfg.d), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    pos = torch.full((1, W), -1, dtype=torch.int32, device=device)
    swa.swa_cache_append(kc, vc, pos, kh, vh, torch.tensor([p0 - W], dtype=torch.int32, device=device))
    p0d = torch.tensor([p0], dtype=torch.int32, device=device)
    o = torch.empty_like(qc)
    lse = torch.empty((1, cfg.Hq, C), dtype=torch.float32, device=device)
    pc = swa.chunk_params(qc, kn, vn, p0d, W, cfg.scale, o, lse, None, False)
    cc = swa.cache_params(kc, vc, pos)
    ws = torch.empty(int(swa.load_library().swa_prefill_chunk_workspace_size(pc, cc)), dtype=torch.uint8,
                     device=device)

    def chunk():
        swa.swa_prefill_chunk(qc, kn, vn, kc, vc, pos, p0d, W, cfg.scale, o=o, lse=lse, workspace=ws, stream=stream)

    ms = timed_steps(chunk, steps, warmup, flush, stream)
    swa.swa_check_device_error()
    flops = 4.0 * cfg.d * C * W * cfg.Hq
    out["chunked_prefill"] = {"ms": ms, "flops": flops, "launches_per_step": 2,
                              "workload": f"{cfg.name}: chunk of {C} tokens at position {p0}, {W}-slot ring"}
    del qc, kn, vn, kh, vh, kc, vc, pos, o, lse, ws
    # append and decode with append, on the decode workload's cache
    dcfg = I.DECODE
    qd_, kc_, vc_, pos_, qpos_ = I.decode_inputs(dcfg)
    L = qpos_.astype(np.int64) + 1
    qd, kcd, vcd = to_dev(qd_, device), to_dev(kc_, device), to_dev(vc_, device)
    del kc_, vc_
    posd = torch.from_numpy(pos_).to(device)
    n_app = 512
    kn = to_dev(I.normal_bf16(dcfg.seed * 16 + 11, (dcfg.B, n_app, dcfg.Hkv, dcfg.d)), device)
    vn = to_dev(I.normal_bf16(dcfg.seed * 16 + 12, (dcfg.B, n_app, dcfg.Hkv, dcfg.d)), device)
    p0a = torch.from_numpy(L.astype(np.int32)).to(device)

    def append():
        swa.swa_cache_append(kcd, vcd, posd, kn, vn, p0a, stream=stream)

    ms = timed_steps(append, steps, warmup, flush, stream)
    swa.swa_check_device_error()
    nbytes = 2 * (2 * dcfg.B * n_app * dcfg.Hkv * dcfg.d * 2) + dcfg.B * n_app * 4 + dcfg.B * 4
    out["cache_append"] = {"ms": ms, "bytes": nbytes, "launches_per_step": 1,
                           "workload": f"{dcfg.name}: {n_app} tokens appended to each of {dcfg.B} sequences"}
    del kn, vn
    # decode with append: token at position L (the appended block moved the caches on;
    # restore the decode workload's cache contents' positions first)
    posd.copy_(torch.from_numpy(pos_).to(device))
    qpos = torch.from_numpy(qpos_).to(device)
    k1 = to_dev(I.normal_bf16(dcfg.seed * 16 + 13, (dcfg.B, dcfg.Hkv, dcfg.d)), device)
    v1 = to_dev(I.normal_bf16(dcfg.seed * 16 + 14, (dcfg.B, dcfg.Hkv, dcfg.d)), device)
    od = torch.empty_like(qd)
    lsed = torch.empty((dcfg.B, dcfg.Hq), dtype=torch.float32, device=device)
    pdp = swa.decode_params(qd, kcd, vcd, posd, qpos, dcfg.scale, od, lsed, None)
    wsd = torch.empty(swa.swa_decode_workspace_size(pdp), dtype=torch.uint8, device=device)

    def dec_append():
        swa.swa_decode_append(qd, kcd, vcd, posd, qpos, k1, v1, dcfg.scale, o=od, lse=lsed, workspace=wsd,
                              stream=stream)

    ms = timed_steps(dec_append, steps, warmup, flush, stream)
    swa.swa_check_device_error()
    out["decode_append"] = {"ms": ms, "bytes": decode_bytes(dcfg, L) + 2 * (2 * dcfg.B * dcfg.Hkv * dcfg.d * 2),
                            "launches_per_step": 2,
                            "workload": f"{dcfg.name}: the current token appended, then attended"}
    return out


def measure_e2e_prefill(cfg, steps, warmup, device, dev_tensors):
    """Same metric through the public call with host buffers, as a serving loop runs it:
    every step copies its q/k/v from pinned host memory to the device, calls swa_fwd and
    copies o and lse back to pinned host memory, all inside the timed region.  Steps are
    double-buffered on three streams, so step i+1's upload and step i-1's download
    overlap step i's kernel (each buffer set is reused only after its previous step's
    kernel and download are done)."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    qd0, kd0, vd0, g, o0, lse0, ws0 = dev_tensors
    hq = torch.empty(qd0.shape, dtype=qd0.dtype, pin_memory=True).copy_(qd0)
    hk = torch.empty(kd0.shape, dtype=kd0.dtype, pin_memory=True).copy_(kd0)
    hv = torch.empty(vd0.shape, dtype=vd0.dtype, pin_memory=True).copy_(vd0)
    sets = [(qd0, kd0, vd0, o0, lse0, ws0)]
    sets.append((torch.empty_like(qd0), torch.empty_like(kd0), torch.empty_like(vd0), torch.empty_like(o0),
                 torch.empty_like(lse0), torch.empty_like(ws0)))
    host_out = [(torch.empty(o0.shape, dtype=o0.dtype, pin_memory=True),
                 torch.empty(lse0.shape, dtype=lse0.dtype, pin_memory=True)) for _ in range(2)]
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ran = [torch.cuda.Event() for _ in range(2)]    # kernel of the set's last step done
    loaded = [torch.cuda.Event() for _ in range(2)]  # inputs of the set's current step on the device
    saved = [torch.cuda.Event() for _ in range(2)]   # outputs of the set's last step on the host

    def step(i):
        x = i % 2
        qd, kd, vd, o, lse, ws = sets[x]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ran[x])
            qd.copy_(hq, non_blocking=True)
            kd.copy_(hk, non_blocking=True)
            vd.copy_(hv, non_blocking=True)
            loaded[x].record(s_in)
        s_run.wait_event(loaded[x])
        if i >= 2:
            s_run.wait_event(saved[x])
        swa.swa_fwd(qd, kd, vd, cfg.window_left, cfg.window_right, cfg.scale, g, o=o, lse=lse, workspace=ws,
                    stream=s_run)
        ran[x].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ran[x])
            host_out[x][0].copy_(o, non_blocking=True)
            host_out[x][1].copy_(lse, non_blocking=True)
            saved[x].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_event(ran[(steps - 1) % 2])
    b.record(s_out)  # after the last step's download (the last work of the pipeline)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    ms = a.elapsed_time(b) / steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    return ms, h2d, d2h


# ----------------------------------------------------------------------------- CPU oracle
class OracleSampler:
    """Times the fp64 oracle on bounded samples of query rows (uniform over the
    batch, heads and sequence) of a prefill workload."""

    def __init__(self, cfg, seed: int = 1):
        import oracle

        self.oracle = oracle
        self.cfg = cfg
        self.G = list(cfg.globals_) or None
        self.q, self.k, self.v = I.prefill_inputs(cfg)
        self.rng = np.random.default_rng(seed)
        cal = self.rows(256)
        t0 = time.perf_counter()
        self.run(cal)
        self.sec_per_row = max((time.perf_counter() - t0) / 256, 1e-7)

    def rows(self, n):
        c = self.cfg
        return np.stack([self.rng.integers(0, c.B, n), self.rng.integers(0, c.Hq, n),
                         self.rng.integers(0, c.T, n)], axis=1).astype(np.int64)

    def pairs(self, rows):
        c, t = self.cfg, rows[:, 2]
        lo = np.zeros_like(t) if c.window_left < 0 else np.maximum(0, t - c.window_left)
        hi = np.full_like(t, c.T - 1) if c.window_right < 0 else np.minimum(c.T - 1, t + c.window_right)
        return int((hi - lo + 1).sum())

    def run(self, rows):
        c = self.cfg
        self.oracle.fwd(self.q, self.k, self.v, c.window_left, c.window_right, c.scale, self.G, rows=rows)

    def step(self, budget_s: float):
        """One timed sample of about budget_s seconds: (TFLOP/s, rows, seconds)."""
        n = int(max(64, budget_s / self.sec_per_row))
        rows = self.rows(n)
        t0 = time.perf_counter()
        self.run(rows)
        dt = time.perf_counter() - t0
        return 4.0 * self.cfg.d * self.pairs(rows) / dt / 1e12, n, dt

    def threads(self) -> int:
        return self.oracle.num_threads()


def kernel_code_digest(path: str) -> str:
    """sha256 of a CUDA source with its comments and whitespace removed: a comment-only
    edit leaves it unchanged, any change to the code changes it."""
    import hashlib
    import re

    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()


def band_traffic_per_launch():
    """DRAM bytes (read + write) of one band-kernel launch on the Mistral workload, from
    the committed ncu summary -- only if it was captured from the current kernel code."""
    path = os.path.join(ROOT, "profiles", "band_fwd_mistral_traffic.txt")
    src = os.path.join(ROOT, "sliding_window_attention_swa_gb300", "csrc", "swa_band.cu")
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if line.strip() and not line.startswith("#"):
                    k, v = line.split(None, 1)
                    fields[k] = v.strip()
        if fields.get("kernel_code_sha256") != kernel_code_digest(src):
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- main
def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def reduce_over_ranks(x: float, op: str, world: int, device) -> float:
    """Max or sum of a per-rank scalar over all ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def job_rate(local_work: float, local_seconds: float, world: int, device) -> float:
    """Whole-job throughput: the work all ranks processed / the slowest rank's time."""
    total = reduce_over_ranks(local_work, "sum", world, device)
    slowest = reduce_over_ranks(local_seconds, "max", world, device)
    return total / slowest


def dist_setup(n_gpus):
    import torch

    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist

    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = I.MISTRAL
    sampler = OracleSampler(cfg)
    budget = min(10.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    vals = []
    for i in range(args.warmup + args.steps):
        v, n, dt = sampler.step(budget)
        if i >= args.warmup:
            vals.append((v, n, dt, sampler.threads()))
    value = float(np.mean([x[0] for x in vals]))
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": float(np.mean([x[2] for x in vals]) * 1e3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": vals[0][3], "kind": "oracle",
                         "sample": f"about {int(np.mean([x[1] for x in vals]))} random query rows of the "
                                   f"workload per step ({budget:.2f} s of fp64 work)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="comma list of workloads: mistral,decode,gemma,longformer,variants,cache")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    args.warmup = max(args.warmup, 3)

    import torch
    import sliding_window_attention_swa_gb300 as swa

    rank, world, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    swa.load_library()
    hbm_peak, bf16_peak, peak_kind = load_peaks()
    only = set(args.only.split(",")) if args.only else {"mistral", "decode", "gemma", "longformer", "variants",
                                                         "cache"}
    flush = L2Flush(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return reduce_over_ranks(x, "max", world, device)

    out = {}
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) if world == 1 else local
    clocks = None
    # headline: Mistral-shape prefill
    barrier()
    cs = ClockSampler(gpu_index)
    res = measure_prefill(I.MISTRAL, args.steps, args.warmup, device, flush, cs)
    barrier()
    clocks = cs.summary()
    ms = max_over_ranks(float(res["ms"].mean()))
    flops = res["flops"]
    tflops = job_rate(flops, float(res["ms"].mean()) * 1e-3, world, device) / 1e12
    kernel_tflops = flops / (float(res["ms"].mean()) * 1e-3) / 1e12
    e2e_ms, h2d, d2h = measure_e2e_prefill(I.MISTRAL, max(10, args.steps // 10), args.warmup, device, res["tensors"])
    e2e_ms = max_over_ranks(e2e_ms)
    del res["tensors"]

    secondary = {}
    gpu_launches = res["launches_per_step"] * args.steps
    if "decode" in only:
        d = measure_decode(I.DECODE, args.steps, args.warmup, device, flush)
        dms = max_over_ranks(float(d["ms"].mean()))
        gbs = world * d["bytes"] / (dms * 1e-3) / 1e9
        secondary["decode"] = {
            "workload": I.DECODE.name, "value": gbs, "unit": "GB/s", "ms_per_step": dms,
            "algorithmic_bytes": d["bytes"], "roofline": {"bound": "hbm", "achieved": d["bytes"] / (float(d["ms"].mean()) * 1e-3) / 1e9,
                                                          "peak": hbm_peak, "unit": "GB/s",
                                                          "frac": d["bytes"] / (float(d["ms"].mean()) * 1e-3) / 1e9 / hbm_peak,
                                                          "peak_kind": peak_kind}}
        gpu_launches += d["launches_per_step"] * args.steps
    for key, cfg in (("gemma", I.GEMMA_LOCAL), ("longformer", I.LONGFORMER)):
        if key not in only:
            continue
        r = measure_prefill(cfg, max(20, args.steps // 4), args.warmup, device, flush)
        del r["tensors"]
        rms = max_over_ranks(float(r["ms"].mean()))
        secondary[key] = {
            "workload": cfg.name, "value": world * r["flops"] / (rms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": rms, "frac_of_bf16_peak": r["flops"] / (rms * 1e-3) / 1e12 / bf16_peak,
            "hbm_gbs": r["bytes"] / (rms * 1e-3) / 1e9, "frac_of_hbm_peak": r["bytes"] / (rms * 1e-3) / 1e9 / hbm_peak}
        gpu_launches += r["launches_per_step"] * max(20, args.steps // 4)

    if "variants" in only:
        # the pages' variants on the same workloads: four attention sinks on the Mistral
        # shape, separate global projections and a dilation mix on the Longformer shape,
        # and decode with four sink slots beside the ring
        import dataclasses

        lf_local = dataclasses.replace(I.LONGFORMER, globals_=(), name=I.LONGFORMER.name + "-no-globals")
        vsteps = max(20, args.steps // 8)
        for key, cfg, variant in (
                ("mistral_sinks4", I.MISTRAL, {"sinks": [0, 1, 2, 3]}),
                ("longformer_separate_global_projections", I.LONGFORMER, {"sep": True}),
                ("longformer_dilation_heads8to11_d2", lf_local, {"dilation": [1] * 8 + [2] * 4})):
            r = measure_prefill(cfg, vsteps, args.warmup, device, flush, variant=variant)
            del r["tensors"]
            rms = max_over_ranks(float(r["ms"].mean()))
            secondary[key] = {
                "workload": cfg.name, "variant": {k: (v if k != "sinks" else len(v)) for k, v in variant.items()},
                "value": world * r["flops"] / (rms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": rms,
                "frac_of_bf16_peak": r["flops"] / (rms * 1e-3) / 1e12 / bf16_peak,
                "hbm_gbs": r["bytes"] / (rms * 1e-3) / 1e9}
            gpu_launches += r["launches_per_step"] * vsteps
        d = measure_decode(I.DECODE, vsteps, args.warmup, device, flush, n_sink=4)
        dms = max_over_ranks(float(d["ms"].mean()))
        secondary["decode_sinks4"] = {
            "workload": I.DECODE.name, "variant": {"n_sink": 4}, "value": world * d["bytes"] / (dms * 1e-3) / 1e9,
            "unit": "GB/s", "ms_per_step": dms, "frac_of_hbm_peak": d["bytes"] / (dms * 1e-3) / 1e9 / hbm_peak}
        gpu_launches += d["launches_per_step"] * vsteps

    if "cache" in only:
        csteps = max(20, args.steps // 8)
        cp = measure_cache_paths(csteps, args.warmup, device, flush)
        for key, r in cp.items():
            rms = max_over_ranks(float(r["ms"].mean()))
            e = {"workload": r["workload"], "ms_per_step": rms}
            if "flops" in r:
                e.update({"value": world * r["flops"] / (rms * 1e-3) / 1e12, "unit": "TFLOP/s",
                          "frac_of_bf16_peak": r["flops"] / (rms * 1e-3) / 1e12 / bf16_peak})
            else:
                e.update({"value": world * r["bytes"] / (rms * 1e-3) / 1e9, "unit": "GB/s",
                          "frac_of_hbm_peak": r["bytes"] / (rms * 1e-3) / 1e9 / hbm_peak})
            secondary[key] = e
            gpu_launches += r["launches_per_step"] * csteps

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        osamp = OracleSampler(I.MISTRAL)
        v, n, dt = osamp.step(12.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": osamp.threads(), "kind": "oracle",
               "sample": f"{n} random query rows of the Mistral-shape workload ({dt:.1f} s, fp64)"}

    traffic = band_traffic_per_launch()

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": headline_config(world),
            "roofline": {"bound": "tensor", "achieved": kernel_tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": kernel_tflops / bf16_peak, "traffic": traffic,
                         "peak_kind": f"{peak_kind} bf16 burst (cuBLAS)", "kernel": KERNELS["band"]},
            "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": gpu_launches,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "secondary": secondary,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
