"""swa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a serving loop that must not allocate once running, or a plugin
interface that passes only inputs and outputs) get the split partials from a
fixed scratch array inside the library instead of a workspace they allocate.
This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  Each call of the new entry
point is checked against swa_decode (the allocating entry point) with the
parity tolerances the other tests use, on two calls in a row whose shapes
differ, so stale scratch contents from the first call cannot pass unnoticed.
"""
import ctypes

import numpy as np
import pytest

from parity import assert_parity, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _noalloc_lib():
    import sliding_window_attention_swa_gb300 as swa

    lib = swa.load_library()
    lib.swa_decode_noalloc.argtypes = [ctypes.POINTER(swa.SwaDecodeParams), ctypes.c_void_p]
    lib.swa_decode_noalloc.restype = ctypes.c_int
    return lib


def _inputs(cfg):
    q, kc, vc, pos, qpos = I.decode_inputs(cfg)
    return to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos)


def _noalloc_call(lib, q, kc, vc, pos, qpos, scale):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hq, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=q.device)
    cnt = torch.full((B, Hq), -7, dtype=torch.int32, device=q.device)
    p = swa.decode_params(q, kc, vc, pos, qpos, scale, o, lse, cnt)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = lib.swa_decode_noalloc(ctypes.byref(p), stream)
    assert status == 0, swa.swa_status_string(status)
    torch.cuda.synchronize()
    return o, lse, cnt


def test_decode_noalloc_matches_decode():
    import torch
    import sliding_window_attention_swa_gb300 as swa

    lib = _noalloc_lib()
    cases = [I.DECODE, I.DecodeConfig("noalloc-second-call", 6, 16, 4, 64, 700, 5000, seed=91)]
    for cfg in cases:  # two calls in a row, different shapes
        q, kc, vc, pos, qpos = _inputs(cfg)
        o_ref, lse_ref, cnt_ref = swa.swa_decode(q, kc, vc, pos, qpos, cfg.scale, want_counts=True)
        torch.cuda.synchronize()
        o, lse, cnt = _noalloc_call(lib, q, kc, vc, pos, qpos, cfg.scale)
        assert_parity(to_host_f64(o), lse.cpu().numpy().astype(np.float64), cnt.cpu().numpy(),
                      to_host_f64(o_ref), lse_ref.cpu().numpy().astype(np.float64), cnt_ref.cpu().numpy(),
                      f"noalloc vs decode: {cfg.name}")


def test_decode_noalloc_rejects_oversized_problem():
    import torch
    import sliding_window_attention_swa_gb300 as swa

    lib = _noalloc_lib()
    # 40 sequences x 128 query heads x 4 splits (1024 slots each) x 256 dims of fp32
    # partials: > 16 MiB.  The buffers are full size, so the call would stay in bounds
    # even if it ran.
    B, Hq, Hkv, d, W = 40, 128, 8, 256, 4096
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(B, Hkv, W, d, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(B, W, dtype=torch.int32, device="cuda")
    qpos = torch.zeros(B, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    p = swa.decode_params(q, kc, kc, pos, qpos, 0.1, o, lse, None)
    assert swa.swa_decode_workspace_size(p) > (16 << 20)
    status = lib.swa_decode_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 5  # SWA_ERR_WORKSPACE


def _decode_at(B, Hq=16, Hkv=1, d=64, W=64):
    """Device tensors of a decode problem whose workspace grows by one row block per sequence."""
    import torch

    g = torch.Generator(device="cuda")
    g.manual_seed(B)
    q = torch.randn(B, Hq, d, generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn(B, Hkv, W, d, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(B, Hkv, W, d, generator=g, device="cuda").to(torch.bfloat16)
    L = np.arange(B) * 37 % (3 * W) + 1  # a mix of part-filled and wrapped rings
    pos = i32_dev(I.ring_slot_positions(L, W))
    qpos = i32_dev((L - 1).astype(np.int32))
    return q, kc, vc, pos, qpos, d ** -0.5


def test_decode_noalloc_at_the_scratch_limit():
    """The largest problem whose split partials fit the scratch array exactly (within one
    sequence's share of it) runs and matches swa_decode, twice in a row; one sequence more
    is rejected with SWA_ERR_WORKSPACE before anything is launched."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    lib = _noalloc_lib()
    limit = 16 << 20

    def need(B):
        q = torch.empty(B, 16, 64, dtype=torch.bfloat16, device="cuda")
        kc = torch.empty(B, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
        pos = torch.empty(B, 64, dtype=torch.int32, device="cuda")
        qpos = torch.empty(B, dtype=torch.int32, device="cuda")
        lse = torch.empty(B, 16, dtype=torch.float32, device="cuda")
        return swa.swa_decode_workspace_size(swa.decode_params(q, kc, kc, pos, qpos, 0.1, q, lse, None))

    lo, hi = 1, 1 << 16  # need(lo) <= limit < need(hi)
    assert need(lo) <= limit < need(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= limit else (lo, mid)
    assert limit - need(lo) < need(lo + 1) - need(lo)  # within one sequence's share
    for _ in range(2):
        q, kc, vc, pos, qpos, scale = _decode_at(lo)
        o_ref, lse_ref, cnt_ref = swa.swa_decode(q, kc, vc, pos, qpos, scale, want_counts=True)
        torch.cuda.synchronize()
        o, lse, cnt = _noalloc_call(lib, q, kc, vc, pos, qpos, scale)
        assert_parity(to_host_f64(o), lse.cpu().numpy().astype(np.float64), cnt.cpu().numpy(),
                      to_host_f64(o_ref), lse_ref.cpu().numpy().astype(np.float64), cnt_ref.cpu().numpy(),
                      f"noalloc at the limit, B={lo}")
    q, kc, vc, pos, qpos, scale = _decode_at(hi)
    o = torch.empty_like(q)
    lse = torch.empty(hi, 16, dtype=torch.float32, device="cuda")
    p = swa.decode_params(q, kc, vc, pos, qpos, scale, o, lse, None)
    status = lib.swa_decode_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 5  # SWA_ERR_WORKSPACE
