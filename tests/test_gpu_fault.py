"""Failure detection without a GPU fault, and the device-side check of the global list.

Planted faults (swa_debug_set_faults): a producer stops issuing copies at a chosen
fill or stage, so the waits of its kernel's other roles run out.  Nothing faults or
hangs: each wait is bounded (about 2.1 s), the CTA that gives up drains the copies and
tensor-core work it did issue, frees its tensor memory and returns.  The host then
reads SWA_ERR_TIMEOUT with only the wait-expiry bit set (no drain expired), and a
normal call in the same process still matches the oracle, so the context is usable.

The prefill kernel's producer pairs its fills (V_j and K_{j+1} on one barrier); the
cases cover two query tiles at d = 128 with an odd ring and at d = 64 with an even
ring, each with and without global positions (whose column tile the producer gathers
with plain stores), and one query tile at d = 256.  The producer of the decode /
global-row split pass is covered as well.

Global list: a list that is not strictly increasing within [0, T) is reported as
SWA_ERR_INVALID_ARG, and the call writes nothing outside its own output buffers.
"""
import time

import numpy as np
import pytest

import oracle
from parity import assert_parity, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu

SWA_ERR_INVALID_ARG = 1
SWA_ERR_TIMEOUT = 4


def _inputs(seed, B, T, Hq, Hkv, d):
    return (I.normal_bf16(seed, (B, T, Hq, d)), I.normal_bf16(seed + 1, (B, T, Hkv, d)),
            I.normal_bf16(seed + 2, (B, T, Hkv, d)))


def _fwd_checked(q, k, v, wl, wr, scale, G, what):
    """A normal swa_fwd call, compared with the oracle."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    o, lse, cnt = swa.swa_fwd(to_dev(q), to_dev(k), to_dev(v), wl, wr, scale, None if G is None else i32_dev(G),
                              want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, scale, G)
    assert_parity(to_host_f64(o).transpose(0, 2, 1, 3), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref,
                  cnt_ref, what)


BAND = [
    # name, (B, T, Hq, Hkv, d, wl, wr), globals, stop fill
    ("paired-d128-odd-ring", (1, 2000, 8, 2, 128, 999, 0), None, 8),
    ("paired-d128-globals", (1, 2000, 8, 2, 128, 999, 0), [0, 1000], 8),
    ("paired-d64-even-ring", (1, 4000, 4, 4, 64, 2000, 0), None, 26),
    ("paired-d64-globals-short-band", (1, 2000, 4, 4, 64, 256, 256), [0, 1000], 10),
    ("paired-d256-one-tile", (1, 1500, 2, 1, 256, 1000, 0), None, 12),
    ("paired-d128-first-fill", (1, 700, 4, 2, 128, 300, 0), None, 0),
]


@pytest.mark.parametrize("case", BAND, ids=[c[0] for c in BAND])
def test_band_producer_stop_times_out_and_recovers(case):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    name, (B, T, Hq, Hkv, d, wl, wr), G, stop = case
    q, k, v = _inputs(5000 + stop + d, B, T, Hq, Hkv, d)
    scale = d ** -0.5
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    gd = None if G is None else i32_dev(G)
    swa.swa_debug_set_faults(band_stop_fill=stop)
    try:
        t0 = time.time()
        swa.swa_fwd(qd, kd, vd, wl, wr, scale, gd)
        st, words = swa.swa_read_device_errors()
        waited = time.time() - t0
    finally:
        swa.swa_debug_set_faults()
    assert st == SWA_ERR_TIMEOUT, (name, st, words)
    assert words == {"prefill": swa.DEVERR_WAIT_TIMEOUT, "split": 0, "cache": 0}, (name, words)
    assert waited < 30.0  # one bounded wait (~2.1 s) and the drain, not a hang
    # the words were cleared and the context works: the same call, normally
    st, words = swa.swa_read_device_errors()
    assert st == 0 and words == {"prefill": 0, "split": 0, "cache": 0}
    _fwd_checked(q, k, v, wl, wr, scale, G, name + " after the planted stop")
    torch.cuda.synchronize()


def test_stop_past_every_fill_changes_nothing():
    """A stop beyond every CTA's last fill: SWA_OK and the oracle's result (the
    planted-stop compare does not disturb a normal run)."""
    import sliding_window_attention_swa_gb300 as swa

    B, T, Hq, Hkv, d = 1, 1000, 8, 2, 128
    q, k, v = _inputs(5101, B, T, Hq, Hkv, d)
    swa.swa_debug_set_faults(band_stop_fill=1 << 30, split_stop_stage=1 << 30)
    try:
        _fwd_checked(q, k, v, 400, 0, d ** -0.5, [3, 500], "stop past the end")
    finally:
        swa.swa_debug_set_faults()


def _decode_case():
    B, Hq, Hkv, d, W = 4, 8, 2, 128, 4096
    q = I.normal_bf16(5201, (B, Hq, d))
    kc = I.normal_bf16(5202, (B, Hkv, W, d))
    vc = I.normal_bf16(5203, (B, Hkv, W, d))
    L = np.array([9000, 4096, 5000, 20000])
    pos = I.ring_slot_positions(L, W)
    qpos = (L - 1).astype(np.int32)
    return q, kc, vc, pos, qpos, d


def test_decode_producer_stop_times_out_and_recovers():
    import torch
    import sliding_window_attention_swa_gb300 as swa

    q, kc, vc, pos, qpos, d = _decode_case()
    args = (to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos), d ** -0.5)
    swa.swa_debug_set_faults(split_stop_stage=5)
    try:
        t0 = time.time()
        swa.swa_decode(*args)
        st, words = swa.swa_read_device_errors()
        waited = time.time() - t0
    finally:
        swa.swa_debug_set_faults()
    assert st == SWA_ERR_TIMEOUT, (st, words)
    assert words == {"prefill": 0, "split": swa.DEVERR_WAIT_TIMEOUT, "cache": 0}, words
    assert waited < 30.0
    o, lse, cnt = swa.swa_decode(*args, want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, d ** -0.5)
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref,
                  "decode after the planted stop")


def test_global_row_pass_stop_times_out_and_recovers():
    """The split pass of the global rows (a programmatic dependent of the band kernel)."""
    import sliding_window_attention_swa_gb300 as swa

    B, T, Hq, Hkv, d = 1, 3000, 8, 2, 128
    q, k, v = _inputs(5301, B, T, Hq, Hkv, d)
    G = [0, 1500]
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    swa.swa_debug_set_faults(split_stop_stage=2)
    try:
        swa.swa_fwd(qd, kd, vd, 200, 200, d ** -0.5, i32_dev(G))
        st, words = swa.swa_read_device_errors()
    finally:
        swa.swa_debug_set_faults()
    assert st == SWA_ERR_TIMEOUT, (st, words)
    assert words == {"prefill": 0, "split": swa.DEVERR_WAIT_TIMEOUT, "cache": 0}, words
    _fwd_checked(q, k, v, 200, 200, d ** -0.5, G, "global rows after the planted stop")


# ----------------------------------------------------------------------------- global list
BAD_LISTS = [
    ("unsorted", [700, 3, 500]),
    ("duplicate", [3, 500, 500]),
    ("negative", [-1, 3, 500]),
    ("past-the-end", [3, 500, 1000]),
    ("long-unsorted", list(range(0, 900, 6)) + [5]),   # more than one tile of positions
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("mode", ["full", "sink"])
@pytest.mark.parametrize("case", BAD_LISTS, ids=[c[0] for c in BAD_LISTS])
def test_bad_global_list_is_reported(case, mode, d):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    name, G = case
    B, T, Hq, Hkv = 1, 1000, 4, 2
    q, k, v = _inputs(5401, B, T, Hq, Hkv, d)
    gmode = swa.GLOBAL_SINK if mode == "sink" else swa.GLOBAL_FULL
    # outputs inside guarded buffers: nothing may be written outside the views
    guard = 4096
    obuf = torch.zeros(2 * guard + B * T * Hq * d, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.zeros(2 * guard + B * Hq * T, dtype=torch.float32, device="cuda")
    cbuf = torch.zeros(2 * guard + B * Hq * T, dtype=torch.int32, device="cuda")
    o = obuf[guard:guard + B * T * Hq * d].view(B, T, Hq, d)
    lse = lbuf[guard:guard + B * Hq * T].view(B, Hq, T)
    cnt = cbuf[guard:guard + B * Hq * T].view(B, Hq, T)
    swa.swa_fwd(to_dev(q), to_dev(k), to_dev(v), 100, 0, d ** -0.5, i32_dev(G), o=o, lse=lse, row_counts=cnt,
                global_mode=gmode)
    st, words = swa.swa_read_device_errors()
    assert st == SWA_ERR_INVALID_ARG, (name, st, words)
    assert words["prefill"] == swa.DEVERR_GLOBAL_LIST and words["cache"] == 0, words
    for buf in (obuf, lbuf, cbuf):
        assert (buf[:guard] == 0).all() and (buf[-guard:] == 0).all(), name
    # a valid list afterwards: no error carried over
    _fwd_checked(q, k, v, 100, 0, d ** -0.5, sorted(set(g for g in G if 0 <= g < T)), name + " then a valid list")
