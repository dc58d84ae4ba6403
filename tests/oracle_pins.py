"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Each ``check_*`` takes a loaded oracle library (``oracle.load()`` or a variant
build) and raises AssertionError when the oracle disagrees with its pin.  The
pins are independent of the oracle's own code: worked examples printed on the
pages (tests/golden), closed-form counts, special cases that reduce to a
library routine (torch's scaled_dot_product_attention in fp64), exact
identities (a one-key window returns its value row), softmax invariants, and a
dense numpy brute force.  ``ALL_CHECKS`` is the list the mutation test runs.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle  # noqa: E402
from sliding_window_attention_swa_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------- golden
def _read_rows(name):
    meta, rows, total, bound = {}, {}, None, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                i, rest = line.split(":")
                keys, cnt = rest.split("|")
                rows[int(i)] = ([int(x) for x in keys.split()], int(cnt))
            else:
                key, *vals = line.split()
                if key == "total":
                    total = int(vals[0])
                elif key == "bound":
                    bound = int(vals[0])
                else:
                    meta[key] = [int(x) for x in vals]
    return meta, rows, total, bound


def _read_kv(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def check_n16_r2_rows(lib):
    meta, rows, total, _ = _read_rows("longformer_n16_r2_rows.txt")
    n, r = meta["n"][0], meta["r"][0]
    got_total = 0
    for t in range(n):
        m = oracle.mask_row(n, t, r, r, lib=lib)
        got_total += int(m.sum())
        if t in rows:
            keys, cnt = rows[t]
            assert list(np.nonzero(m)[0]) == keys, (t, np.nonzero(m)[0], keys)
            assert int(m.sum()) == cnt
    assert got_total == total == 74


def check_n16_globals(lib):
    meta, rows, total, bound = _read_rows("longformer_n16_r2_globals_0_8_rows.txt")
    n, r, G = meta["n"][0], meta["r"][0], meta["G"]
    got_total = 0
    for t in range(n):
        m = oracle.mask_row(n, t, r, r, G, lib=lib)
        keys, cnt = rows[t]
        assert list(np.nonzero(m)[0]) == keys, (t, np.nonzero(m)[0], keys)
        assert int(m.sum()) == cnt
        got_total += cnt
    assert got_total == total == 120 and got_total <= bound


def check_causal_windows(lib):
    for tag, Ts, Ws, ts, ks in _read_kv("causal_windows.txt"):
        T, W, t = int(Ts[2:]), int(Ws[2:]), int(ts[2:])
        lo, hi = (int(x) for x in ks[5:].split(".."))
        m = oracle.mask_row(T, t, W - 1, 0, lib=lib)
        idx = np.nonzero(m)[0]
        assert idx[0] == lo and idx[-1] == hi and len(idx) == hi - lo + 1, (tag, idx[0], idx[-1])


def _total(lib, T, wl, wr, G=None):
    return sum(int(oracle.mask_row(T, t, wl, wr, G, lib=lib).sum()) for t in range(T))


def check_n16_totals(lib):
    want = {k: int(v) for k, v in _read_kv("n16_pattern_totals.txt")}
    assert _total(lib, 16, -1, -1) == want["full_bidirectional"]
    assert _total(lib, 16, 15, 15) == want["full_bidirectional"]
    assert _total(lib, 16, -1, 0) == want["full_causal"]
    assert _total(lib, 16, 15, 0) == want["full_causal"]
    assert _total(lib, 16, 2, 2) == want["window_r2"]


def check_closed_form_counts(lib):
    # (2r+1)n - r(r+1) for the clipped symmetric band (Longformer page section 1.3), n >= 2r.
    for n, r in [(16, 2), (37, 5), (64, 31), (100, 1), (9, 4)]:
        assert _total(lib, n, r, r) == (2 * r + 1) * n - r * (r + 1), (n, r)
    # sum_t min(t+1, W) = W*T - W(W-1)/2 for the causal window, W <= T.
    for T, W in [(16, 4), (50, 7), (33, 33), (40, 1)]:
        assert _total(lib, T, W - 1, 0) == W * T - W * (W - 1) // 2, (T, W)
    # Asymmetric window (wl, wr): interior rows see wl + wr + 1 keys.
    m = oracle.mask_row(100, 50, 7, 3, lib=lib)
    assert list(np.nonzero(m)[0]) == list(range(43, 54))


def _rand_case(seed, B, T, Hq, Hkv, D):
    q = I.normal_bf16(seed * 4 + 0, (B, T, Hq, D))
    k = I.normal_bf16(seed * 4 + 1, (B, T, Hkv, D))
    v = I.normal_bf16(seed * 4 + 2, (B, T, Hkv, D))
    return q, k, v


def _widen(h):
    return I.bf16_bits_to_f32(h).astype(np.float64)


def _sdpa(q, k, v, scale, causal):
    """torch fp64 reference with K/V heads expanded for the contiguous GQA map."""
    qd, kd, vd = (torch.from_numpy(_widen(x)).permute(0, 2, 1, 3) for x in (q, k, v))
    g = qd.shape[1] // kd.shape[1]
    kd = kd.repeat_interleave(g, dim=1)
    vd = vd.repeat_interleave(g, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=causal, scale=scale)
    s = (qd @ kd.transpose(-1, -2)) * scale
    if causal:
        T = s.shape[-1]
        s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


def check_full_windows_match_library(lib):
    # W >= T is standard causal attention (lizeman page, section 2, first display);
    # unbounded / all-global windows are full bidirectional attention.
    q, k, v = _rand_case(3, 2, 40, 4, 2, 32)
    scale = 0.17
    o_ref, lse_ref = _sdpa(q, k, v, scale, causal=True)
    for wl in (39, 100, -1):
        o, lse, cnt = oracle.fwd(q, k, v, wl, 0, scale, lib=lib)
        np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-12, rtol=1e-10)
        assert (cnt == np.arange(1, 41)[None, None, :]).all()
    o_ref, lse_ref = _sdpa(q, k, v, scale, causal=False)
    for wl, wr, G in ((-1, -1, None), (39, 39, None), (1, 0, list(range(40)))):
        o, lse, cnt = oracle.fwd(q, k, v, wl, wr, scale, G, lib=lib)
        np.testing.assert_allclose(o, o_ref, atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-12, rtol=1e-10)
        assert (cnt == 40).all()


def check_one_key_window(lib):
    # W = 1: the window is {t}, the softmax weight is exactly 1, so o_t = v_t and
    # lse_t = scale * q_t . k_t.
    q, k, v = _rand_case(5, 1, 24, 4, 2, 64)
    scale = 0.125
    o, lse, cnt = oracle.fwd(q, k, v, 0, 0, scale, lib=lib)
    vd, qd, kd = _widen(v), _widen(q), _widen(k)
    for h in range(4):
        np.testing.assert_array_equal(o[0, h], vd[0, :, h // 2, :])
        ref = scale * np.einsum("td,td->t", qd[0, :, h, :], kd[0, :, h // 2, :])
        np.testing.assert_allclose(lse[0, h], ref, atol=1e-12, rtol=1e-12)
    assert (cnt == 1).all()


def check_softmax_invariants(lib):
    # Weights sum to 1 (value rows all one give o = 1) and o lies in the
    # per-dimension hull of the attended value rows.
    q, k, v = _rand_case(7, 1, 48, 2, 1, 16)
    ones = np.full_like(v, 0x3F80)  # bf16 1.0
    o, _, _ = oracle.fwd(q, k, ones, 5, 2, 0.3, [0, 20], lib=lib)
    np.testing.assert_allclose(o, 1.0, atol=1e-13)
    o, _, _ = oracle.fwd(q, k, v, 5, 2, 0.3, [0, 20], lib=lib)
    vd = _widen(v)[0, :, 0, :]
    mask = oracle.dense_mask(48, 5, 2, [0, 20])
    for t in range(48):
        sel = vd[mask[t]]
        assert (o[0, :, t, :] >= sel.min(axis=0) - 1e-12).all()
        assert (o[0, :, t, :] <= sel.max(axis=0) + 1e-12).all()


def check_bruteforce(lib):
    cases = [
        (1, 16, 1, 1, 64, 2, 2, None),
        (1, 16, 1, 1, 64, 3, 0, None),
        (2, 33, 4, 2, 16, 6, 0, None),
        (1, 40, 3, 1, 32, 4, 9, [3, 17, 39]),
        (2, 29, 2, 2, 8, 0, 5, [0]),
        (1, 45, 4, 4, 16, 2, 2, [0, 8, 9, 44]),
        (1, 20, 2, 1, 32, -1, 3, None),
        (1, 20, 2, 1, 32, 4, -1, [10]),
    ]
    for i, (B, T, Hq, Hkv, D, wl, wr, G) in enumerate(cases):
        q, k, v = _rand_case(11 + i, B, T, Hq, Hkv, D)
        scale = 1.0 / np.sqrt(D)
        o, lse, cnt = oracle.fwd(q, k, v, wl, wr, scale, G, lib=lib)
        ob, lseb, cntb = oracle.dense_bruteforce(q, k, v, wl, wr, scale, G)
        np.testing.assert_allclose(o, ob, atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lseb, atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt, cntb)
    # Row selection returns the same values as the full evaluation.
    q, k, v = _rand_case(30, 2, 33, 4, 2, 16)
    o, lse, cnt = oracle.fwd(q, k, v, 6, 1, 0.25, [5], lib=lib)
    rows = np.array([[1, 3, 32], [0, 0, 0], [1, 1, 5], [0, 2, 17]])
    o2, lse2, cnt2 = oracle.fwd(q, k, v, 6, 1, 0.25, [5], rows=rows, lib=lib)
    for i, (b, h, t) in enumerate(rows):
        np.testing.assert_array_equal(o2[i], o[b, h, t])
        assert lse2[i] == lse[b, h, t] and cnt2[i] == cnt[b, h, t]


def check_gqa_contiguous_groups(lib):
    # Query head h reads key/value head h // (Hq/Hkv): expanding K/V by
    # repeat-interleave and running one key/value head per query head is the same.
    q, k, v = _rand_case(41, 1, 24, 6, 2, 16)
    o, lse, _ = oracle.fwd(q, k, v, 4, 0, 0.2, lib=lib)
    kx = np.repeat(k, 3, axis=2)
    vx = np.repeat(v, 3, axis=2)
    o2, lse2, _ = oracle.fwd(q, kx, vx, 4, 0, 0.2, lib=lib)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def check_decode_matches_prefill(lib):
    # The ring buffer holds token p in slot p mod W (lizeman page, KV cache paragraph);
    # a decode step at t = L-1 must equal row t of causal-window prefill.
    rng = np.random.default_rng(0)
    for L, W in [(1, 8), (5, 8), (8, 8), (9, 8), (37, 8), (100, 16), (16, 32)]:
        B, Hq, Hkv, D = 2, 4, 2, 16
        q, k, v = _rand_case(50 + L, B, L, Hq, Hkv, D)
        o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, W - 1, 0, 0.25, lib=lib)
        kc = I.normal_bf16(999, (B, Hkv, W, D))  # stale slots hold unrelated data
        vc = I.normal_bf16(998, (B, Hkv, W, D))
        pos = I.ring_slot_positions(np.array([L] * B), W)
        for b in range(B):
            for j in range(W):
                p = pos[b, j]
                if 0 <= p < L:
                    kc[b, :, j, :] = k[b, p]
                    vc[b, :, j, :] = v[b, p]
        qd = q[:, L - 1]  # [B, Hq, D]
        o, lse, cnt = oracle.decode(qd, kc, vc, pos, np.array([L - 1] * B), 0.25, lib=lib)
        np.testing.assert_allclose(o, o_ref[:, :, L - 1], atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lse_ref[:, :, L - 1], atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt, np.minimum(L, W))
        # Permuting the slots (with their positions) changes nothing.
        perm = rng.permutation(W)
        o2, lse2, cnt2 = oracle.decode(qd, kc[:, :, perm], vc[:, :, perm], pos[:, perm],
                                       np.array([L - 1] * B), 0.25, lib=lib)
        np.testing.assert_allclose(o2, o, atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt2, cnt)


def check_decode_guards(lib):
    # Stale slots (negative, future, or older than the window) are excluded.
    B, Hq, Hkv, D, W = 1, 2, 1, 8, 6
    q = I.normal_bf16(61, (B, Hq, D))
    kc = I.normal_bf16(62, (B, Hkv, W, D))
    vc = I.normal_bf16(63, (B, Hkv, W, D))
    t = 20
    pos = np.array([[20, -1, 15, 14, 21, 16]], dtype=np.int32)  # valid: 20, 15, 16
    o, lse, cnt = oracle.decode(q, kc, vc, pos, np.array([t]), 0.5, lib=lib)
    assert (cnt == 3).all()
    drop = [1, 3, 4]  # excluded slots: their K/V contents must not matter
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, :, drop] = I.normal_bf16(64, (B, Hkv, 3, D), 4.0)
    vc2[:, :, drop] = I.normal_bf16(65, (B, Hkv, 3, D), 4.0)
    o2, lse2, _ = oracle.decode(q, kc2, vc2, pos, np.array([t]), 0.5, lib=lib)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    # ... while a kept slot's contents do.
    kc2[:, :, 2] = kc[:, :, 3]
    o3, _, _ = oracle.decode(q, kc2, vc, pos, np.array([t]), 0.5, lib=lib)
    assert np.abs(o3 - o).max() > 1e-6


def check_workload_counts(lib):
    # Attended pairs per head of the three prefill workloads, from closed forms
    # computed here without the oracle: causal W*T - W(W-1)/2; clipped symmetric
    # band (2r+1)n - r(r+1); with globals, each global row sees all T keys and each
    # local row adds the global columns outside its band.
    assert _total(lib, 4096, 256, 256) == 513 * 4096 - 256 * 257 == 2_035_456
    T, r, G = 4096, 256, [0, 2048]
    t = np.arange(T)
    band = np.minimum(T - 1, t + r) - np.maximum(0, t - r) + 1
    local = ~np.isin(t, G)
    extra = sum(((np.abs(t - g) > r) & local).sum() for g in G)
    want = int(band[local].sum() + extra + len(G) * T)
    assert want == 2_050_298
    assert _total(lib, T, r, r, G) == want
    # Causal workloads, spot rows plus the closed-form total (the mask is
    # translation-invariant away from the start, so the first W rows and one
    # interior row determine it).
    for T, W, want in [(16384, 4096, 58_722_304), (32768, 1024, 33_030_656)]:
        assert W * T - W * (W - 1) // 2 == want
        head = sum(int(oracle.mask_row(T, t, W - 1, 0, lib=lib).sum()) for t in range(0, W, 97))
        assert head == sum(min(t + 1, W) for t in range(0, W, 97))
        assert int(oracle.mask_row(T, T - 1, W - 1, 0, lib=lib).sum()) == W


# ----------------------------------------------------------------------------- dilation
def check_dilated_n16_rows(lib):
    meta, rows, total, _ = _read_rows("longformer_n16_r2_d2_dilated_rows.txt")
    n, r, d = meta["n"][0], meta["r"][0], meta["d"][0]
    got_total = 0
    for t in range(n):
        m = oracle.mask_row(n, t, r, r, lib=lib, dil=d)
        keys, cnt = rows[t]
        assert list(np.nonzero(m)[0]) == keys, (t, np.nonzero(m)[0], keys)
        assert int(m.sum()) == cnt
        got_total += cnt
    assert got_total == total == 68


def check_dilated_closed_forms(lib):
    # Causal dilated window {t - i*d : 0 <= i < W} (lizeman page, "Dilation"):
    # min(W, floor(t/d) + 1) keys.  Symmetric dilated band: the undilated count of
    # the row's residue class, i.e. min(r, floor(t/d)) + min(r, floor((n-1-t)/d)) + 1.
    for T, W, d in [(50, 4, 3), (40, 7, 2), (33, 1, 5), (64, 8, 8)]:
        for t in range(T):
            m = oracle.mask_row(T, t, W - 1, 0, lib=lib, dil=d)
            assert int(m.sum()) == min(W, t // d + 1), (T, W, d, t)
            assert all((t - s) % d == 0 and 0 <= t - s < W * d for s in np.nonzero(m)[0])
    for n, r, d in [(16, 2, 2), (45, 3, 4), (30, 6, 3)]:
        for t in range(n):
            want = min(r, t // d) + min(r, (n - 1 - t) // d) + 1
            assert int(oracle.mask_row(n, t, r, r, lib=lib, dil=d).sum()) == want


def check_dilated_residue_identity(lib):
    # Dilation d splits the sequence into d residue classes; on each class the
    # dilated band is the ordinary band of the subsequence (same wl, wr in steps).
    q, k, v = _rand_case(70, 2, 37, 4, 2, 16)
    dil = [1, 2, 3, 2]
    o, lse, cnt = oracle.fwd(q, k, v, 3, 2, 0.2, lib=lib, dilation=dil)
    for h, d in enumerate(dil):
        for r in range(d):
            o2, lse2, cnt2 = oracle.fwd(q[:, r::d], k[:, r::d], v[:, r::d], 3, 2, 0.2, lib=lib)
            np.testing.assert_array_equal(o[:, h, r::d], o2[:, h])
            np.testing.assert_array_equal(lse[:, h, r::d], lse2[:, h])
            np.testing.assert_array_equal(cnt[:, h, r::d], cnt2[:, h])


def check_dilated_bruteforce(lib):
    cases = [
        (1, 16, 2, 1, 16, 2, 2, [2, 1]),
        (1, 30, 4, 2, 8, 3, 0, [1, 2, 3, 4]),
        (2, 25, 2, 2, 16, -1, 1, [3, 2]),
    ]
    for i, (B, T, Hq, Hkv, D, wl, wr, dil) in enumerate(cases):
        q, k, v = _rand_case(80 + i, B, T, Hq, Hkv, D)
        o, lse, cnt = oracle.fwd(q, k, v, wl, wr, 0.3, lib=lib, dilation=dil)
        ob, lseb, cntb = oracle.dense_bruteforce(q, k, v, wl, wr, 0.3, dilation=dil)
        np.testing.assert_allclose(o, ob, atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lseb, atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt, cntb)


# ----------------------------------------------------------------------------- sinks
def check_sink_counts(lib):
    # Causal window W plus sinks {0..ns-1}: the band's min(t+1, W) keys plus the
    # sinks left of it, max(0, min(ns, t-W+1)).  Bidirectional radius r: sinks are
    # kept only left of the band (a sink right of it is beyond t + r).
    S = oracle.GLOBAL_SINK
    for T, W, ns in [(40, 4, 3), (64, 16, 4), (20, 25, 2), (30, 1, 1)]:
        for t in range(T):
            m = oracle.mask_row(T, t, W - 1, 0, list(range(ns)), lib=lib, gmode=S)
            assert int(m.sum()) == min(t + 1, W) + max(0, min(ns, t - W + 1)), (T, W, ns, t)
            assert not m[t + 1:].any()
    for n, r, ns in [(30, 3, 4), (16, 2, 2)]:
        for t in range(n):
            m = oracle.mask_row(n, t, r, r, list(range(ns)), lib=lib, gmode=S)
            band = min(n - 1, t + r) - max(0, t - r) + 1
            assert int(m.sum()) == band + max(0, min(ns, t - r)), (n, r, ns, t)


def check_sink_bruteforce(lib):
    S = oracle.GLOBAL_SINK
    cases = [
        (1, 40, 2, 1, 16, 5, 0, [0, 1, 2, 3]),
        (2, 33, 4, 2, 16, 3, 2, [0, 5, 17]),
        (1, 24, 2, 2, 8, -1, 0, [0]),
    ]
    for i, (B, T, Hq, Hkv, D, wl, wr, G) in enumerate(cases):
        q, k, v = _rand_case(90 + i, B, T, Hq, Hkv, D)
        o, lse, cnt = oracle.fwd(q, k, v, wl, wr, 0.25, G, lib=lib, gmode=S)
        ob, lseb, cntb = oracle.dense_bruteforce(q, k, v, wl, wr, 0.25, G, gmode=S)
        np.testing.assert_allclose(o, ob, atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lseb, atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt, cntb)
    # Sinks already inside every row's band change nothing (window >= T).
    q, k, v = _rand_case(95, 1, 20, 2, 1, 16)
    o, lse, cnt = oracle.fwd(q, k, v, 19, 0, 0.25, [0, 1], lib=lib, gmode=S)
    o2, lse2, cnt2 = oracle.fwd(q, k, v, 19, 0, 0.25, lib=lib)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(cnt, cnt2)


def _sink_cache(k, v, L, W, ns, S_slots, seed):
    """Cache of ns sink slots then a W-slot ring for positions >= ns (p at ns + (p-ns) % W),
    holding tokens 0..L-1 of k/v [B,L,Hkv,D]; built here without the oracle."""
    B, _, Hkv, D = k.shape
    kc = I.normal_bf16(seed, (B, Hkv, S_slots, D))
    vc = I.normal_bf16(seed + 1, (B, Hkv, S_slots, D))
    pos = np.full((B, S_slots), -1, dtype=np.int32)
    for p in range(L):
        if p < ns:
            j = p
        elif p > L - 1 - W:
            j = ns + (p - ns) % W
        else:
            continue
        pos[:, j] = p
        kc[:, :, j] = k[:, p]
        vc[:, :, j] = v[:, p]
    return kc, vc, pos


def check_decode_sinks(lib):
    # Decode with the first ns positions pinned equals row t of the sink prefill.
    for L, W, ns in [(30, 8, 2), (9, 8, 3), (3, 8, 2), (50, 4, 4)]:
        B, Hq, Hkv, D = 2, 4, 2, 16
        q, k, v = _rand_case(100 + L, B, L, Hq, Hkv, D)
        o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, W - 1, 0, 0.25, list(range(ns)), lib=lib,
                                             gmode=oracle.GLOBAL_SINK)
        kc, vc, pos = _sink_cache(k, v, L, W, ns, ns + W, 700 + L)
        o, lse, cnt = oracle.decode(q[:, L - 1], kc, vc, pos, np.array([L - 1] * B), 0.25, lib=lib, window=W,
                                    n_sink=ns)
        np.testing.assert_allclose(o, o_ref[:, :, L - 1], atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lse_ref[:, :, L - 1], atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt, min(L, W) + max(0, min(ns, L - W)))


# ----------------------------------------------------------------------------- global projections
def check_global_projection_identity(lib):
    # With Q_g = Q, K_g = K, V_g = V the two-projection design is the one-projection
    # attention (Longformer page 5.3: the global projections start as copies).
    q, k, v = _rand_case(110, 2, 30, 4, 2, 16)
    G = [0, 7, 29]
    o, lse, cnt = oracle.fwd(q, k, v, 3, 3, 0.25, G, lib=lib)
    o2, lse2, cnt2 = oracle.fwd(q, k, v, 3, 3, 0.25, G, lib=lib, qg=q, kg=k, vg=v)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    np.testing.assert_array_equal(cnt, cnt2)


def check_global_projection_roles(lib):
    q, k, v = _rand_case(111, 1, 30, 4, 2, 16)
    qg, kg, vg = _rand_case(112, 1, 30, 4, 2, 16)
    G = [0, 12]
    o, lse, _ = oracle.fwd(q, k, v, 2, 2, 0.25, G, lib=lib, qg=qg, kg=kg, vg=vg)
    ob, lseb, _ = oracle.dense_bruteforce(q, k, v, 2, 2, 0.25, G, qg=qg, kg=kg, vg=vg)
    np.testing.assert_allclose(o, ob, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(lse, lseb, atol=1e-12, rtol=1e-10)
    # Global rows read only Q_g, K_g, V_g: replacing Q, K, V leaves them unchanged.
    q2, k2, v2 = _rand_case(113, 1, 30, 4, 2, 16)
    o2, lse2, _ = oracle.fwd(q2, k2, v2, 2, 2, 0.25, G, lib=lib, qg=qg, kg=kg, vg=vg)
    np.testing.assert_array_equal(o2[:, :, G], o[:, :, G])
    np.testing.assert_array_equal(lse2[:, :, G], lse[:, :, G])
    # Local rows read Q_g nowhere and K_g, V_g only at global positions.
    loc = [t for t in range(30) if t not in G]
    qg3, kg3, vg3 = _rand_case(114, 1, 30, 4, 2, 16)
    kg3[:, G], vg3[:, G] = kg[:, G], vg[:, G]
    o3, lse3, _ = oracle.fwd(q, k, v, 2, 2, 0.25, G, lib=lib, qg=qg3, kg=kg3, vg=vg3)
    np.testing.assert_array_equal(o3[:, :, loc], o[:, :, loc])
    # ... and they do read K_g, V_g at a global position, even inside their band.
    kg4 = kg.copy()
    kg4[:, 12] = k[:, 12]
    o4, _, _ = oracle.fwd(q, k, v, 2, 2, 0.25, G, lib=lib, qg=qg, kg=kg4, vg=vg)
    assert np.abs(o4[:, :, 11] - o[:, :, 11]).max() > 1e-6


# ----------------------------------------------------------------------------- ring append, chunks
def _ring_closed_form(L, W):
    """Slot positions after tokens 0..L-1 went into slot p mod W: the largest
    p <= L-1 with p = j (mod W), or -1 for a slot never written."""
    j = np.arange(W)
    last = L - 1 - ((L - 1 - j) % W)
    return np.where(j < L, last, -1) if L < W else last


def check_append_ring(lib):
    B, Hkv, D, W = 2, 2, 8, 8
    for L, pieces in [(5, [5]), (8, [3, 5]), (21, [1, 6, 7, 7]), (30, [30]), (17, [16, 1])]:
        k = I.normal_bf16(120 + L, (B, L, Hkv, D))
        v = I.normal_bf16(121 + L, (B, L, Hkv, D))
        kc = I.normal_bf16(122, (B, Hkv, W, D))
        vc = I.normal_bf16(123, (B, Hkv, W, D))
        pos = np.full((B, W), -1, dtype=np.int32)
        p0 = 0
        for n in pieces:
            kc, vc, pos = oracle.cache_append(kc, vc, pos, k[:, p0:p0 + n], v[:, p0:p0 + n], [p0] * B, lib=lib)
            p0 += n
        want = _ring_closed_form(L, W)
        for b in range(B):
            np.testing.assert_array_equal(pos[b], want)
            for j in range(W):
                if want[j] >= 0:
                    np.testing.assert_array_equal(kc[b, :, j], k[b, want[j]])
                    np.testing.assert_array_equal(vc[b, :, j], v[b, want[j]])


def check_append_with_sinks(lib):
    # Appending tokens 0..L-1 in pieces to a cache with pinned sinks reproduces the
    # layout built directly (sink slots, then the ring of the last positions), and
    # each written slot holds its token's rows.
    B, Hkv, D, W, ns = 2, 2, 8, 8, 3
    for L, pieces in [(2, [2]), (5, [1, 4]), (11, [11]), (30, [7, 7, 16]), (40, [40])]:
        k = I.normal_bf16(150 + L, (B, L, Hkv, D))
        v = I.normal_bf16(151 + L, (B, L, Hkv, D))
        kc = I.normal_bf16(152, (B, Hkv, ns + W, D))
        vc = I.normal_bf16(153, (B, Hkv, ns + W, D))
        pos = np.full((B, ns + W), -1, dtype=np.int32)
        p0 = 0
        for n in pieces:
            kc, vc, pos = oracle.cache_append(kc, vc, pos, k[:, p0:p0 + n], v[:, p0:p0 + n], [p0] * B, lib=lib,
                                              n_sink=ns)
            p0 += n
        kref, vref, pref = _sink_cache(k, v, L, W, ns, ns + W, 152)
        np.testing.assert_array_equal(pos, pref)
        np.testing.assert_array_equal(pos, I.sink_ring_slot_positions(np.array([L] * B), W, ns))
        for b in range(B):
            for j in range(ns + W):
                if pos[b, j] >= 0:
                    np.testing.assert_array_equal(kc[b, :, j], k[b, pos[b, j]])
                    np.testing.assert_array_equal(vc[b, :, j], v[b, pos[b, j]])


def check_chunk_matches_prefill(lib):
    # Chunked prefill (history in the ring, chunk as new tokens) equals rows
    # p0 .. p0+C-1 of the causal-window prefill over the whole sequence.
    B, Hq, Hkv, D = 2, 4, 2, 16
    for p0, C, W in [(0, 5, 4), (3, 4, 8), (10, 6, 4), (20, 20, 8), (7, 1, 8), (16, 9, 16)]:
        L = p0 + C
        q, k, v = _rand_case(130 + L, B, L, Hq, Hkv, D)
        o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, W - 1, 0, 0.25, lib=lib)
        kc = I.normal_bf16(131, (B, Hkv, W, D))
        vc = I.normal_bf16(132, (B, Hkv, W, D))
        pos = np.full((B, W), -1, dtype=np.int32)
        if p0:
            kc, vc, pos = oracle.cache_append(kc, vc, pos, k[:, :p0], v[:, :p0], [0] * B, lib=lib)
        o, lse, cnt = oracle.chunk(q[:, p0:], k[:, p0:], v[:, p0:], kc, vc, pos, [p0] * B, W, 0.25, lib=lib)
        np.testing.assert_allclose(o, o_ref[:, :, p0:], atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(lse, lse_ref[:, :, p0:], atol=1e-12, rtol=1e-10)
        np.testing.assert_array_equal(cnt, cnt_ref[:, :, p0:])
    # Slots holding positions at or after p0 (left by tokens that were rolled back)
    # are not history: a cache of W+3 slots keeps the whole window even after three
    # such tokens were appended, and the chunk must ignore them.
    p0, C, W = 12, 5, 8
    L = p0 + C
    q, k, v = _rand_case(135, B, L, Hq, Hkv, D)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, W - 1, 0, 0.25, lib=lib)
    kc = I.normal_bf16(136, (B, Hkv, W + 3, D))
    vc = I.normal_bf16(137, (B, Hkv, W + 3, D))
    pos = np.full((B, W + 3), -1, dtype=np.int32)
    kc, vc, pos = oracle.cache_append(kc, vc, pos, k[:, :p0], v[:, :p0], [0] * B, lib=lib)
    junk_k, junk_v = I.normal_bf16(138, (B, 3, Hkv, D), 3.0), I.normal_bf16(139, (B, 3, Hkv, D), 3.0)
    kc, vc, pos = oracle.cache_append(kc, vc, pos, junk_k, junk_v, [p0] * B, lib=lib)
    o, lse, cnt = oracle.chunk(q[:, p0:], k[:, p0:], v[:, p0:], kc, vc, pos, [p0] * B, W, 0.25, lib=lib)
    np.testing.assert_allclose(o, o_ref[:, :, p0:], atol=1e-12, rtol=1e-10)
    np.testing.assert_array_equal(cnt, cnt_ref[:, :, p0:])
    # With pinned sinks, against the sink prefill.
    p0, C, W, ns = 20, 6, 8, 2
    L = p0 + C
    q, k, v = _rand_case(140, B, L, Hq, Hkv, D)
    o_ref, lse_ref, _ = oracle.fwd(q, k, v, W - 1, 0, 0.25, list(range(ns)), lib=lib, gmode=oracle.GLOBAL_SINK)
    kc, vc, pos = _sink_cache(k, v, p0, W, ns, ns + W, 141)
    o, lse, _ = oracle.chunk(q[:, p0:], k[:, p0:], v[:, p0:], kc, vc, pos, [p0] * B, W, 0.25, n_sink=ns, lib=lib)
    np.testing.assert_allclose(o, o_ref[:, :, p0:], atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(lse, lse_ref[:, :, p0:], atol=1e-12, rtol=1e-10)


ALL_CHECKS = [
    check_n16_r2_rows,
    check_n16_globals,
    check_causal_windows,
    check_n16_totals,
    check_closed_form_counts,
    check_full_windows_match_library,
    check_one_key_window,
    check_softmax_invariants,
    check_bruteforce,
    check_gqa_contiguous_groups,
    check_decode_matches_prefill,
    check_decode_guards,
    check_workload_counts,
    check_dilated_n16_rows,
    check_dilated_closed_forms,
    check_dilated_residue_identity,
    check_dilated_bruteforce,
    check_sink_counts,
    check_sink_bruteforce,
    check_decode_sinks,
    check_global_projection_identity,
    check_global_projection_roles,
    check_append_ring,
    check_append_with_sinks,
    check_chunk_matches_prefill,
]
