"""Attention sinks, separate global projections, dilated bands and decode windows
(through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from parity import assert_parity, compare_every_row, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _inputs(seed, B, T, Hq, Hkv, d, scale=1.0):
    q = I.normal_bf16(seed, (B, T, Hq, d), scale)
    k = I.normal_bf16(seed + 1, (B, T, Hkv, d), scale)
    v = I.normal_bf16(seed + 2, (B, T, Hkv, d))
    return q, k, v


def _run(q, k, v, wl, wr, scale, G=None, **kw):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    for name in ("q_g", "k_g", "v_g"):
        if kw.get(name) is not None:
            kw[name] = to_dev(kw[name])
    g = None if G is None else i32_dev(G)
    o, lse, cnt = swa.swa_fwd(to_dev(q), to_dev(k), to_dev(v), wl, wr, scale, g, want_counts=True, **kw)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    return to_host_f64(o).transpose(0, 2, 1, 3), lse.cpu().numpy().astype(np.float64), cnt.cpu().numpy()


def _run_full(q, k, v, wl, wr, scale, G=None, **kw):
    """As _run, for full-size outputs: O stays bf16 [B, T, Hq, d] on the host."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    for name in ("q_g", "k_g", "v_g"):
        if kw.get(name) is not None:
            kw[name] = to_dev(kw[name])
    g = None if G is None else i32_dev(G)
    o, lse, cnt = swa.swa_fwd(to_dev(q), to_dev(k), to_dev(v), wl, wr, scale, g, want_counts=True, **kw)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    return o.cpu(), lse.cpu().numpy().astype(np.float64), cnt.cpu().numpy()


# ----------------------------------------------------------------------------- sinks
SINKS = [
    # B, T, Hq, Hkv, d, wl, wr, sinks
    (1, 300, 8, 2, 128, 63, 0, [0, 1, 2, 3]),
    (2, 257, 4, 4, 64, 31, 0, [0]),
    (1, 200, 4, 2, 256, 40, 0, [0, 1]),
    (1, 500, 12, 12, 64, 32, 32, [0, 1, 2, 3]),
    (1, 100, 4, 1, 128, 150, 0, [0, 1, 2, 3]),          # sinks inside every band
    (1, 700, 4, 2, 128, 100, 0, list(range(150))),      # two global-column tiles
    (1, 400, 2, 1, 64, 20, 3, [5, 77, 300]),            # sinks that are not the first tokens
    (1, 1500, 4, 2, 128, 1000, 0, [0, 1, 2, 3]),        # long band (the long-band kernel)
]


@pytest.mark.parametrize("case", SINKS, ids=[f"T{c[1]}-d{c[4]}-wl{c[5]}-wr{c[6]}-n{len(c[7])}" for c in SINKS])
def test_sinks(case):
    B, T, Hq, Hkv, d, wl, wr, G = case
    q, k, v = _inputs(3 * T + d, B, T, Hq, Hkv, d)
    scale = d ** -0.5
    o, lse, cnt = _run(q, k, v, wl, wr, scale, G, global_mode=oracle.GLOBAL_SINK)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, scale, G, gmode=oracle.GLOBAL_SINK)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case))


def test_sinks_full_size_mistral():
    """Mistral-shape causal prefill with four pinned sinks: every row's count against
    the closed form min(t+1, W) + max(0, min(4, t-W+1)), every row's O and lse against
    the oracle."""
    cfg = I.MISTRAL
    q, k, v = I.prefill_inputs(cfg)
    G = [0, 1, 2, 3]
    W = cfg.window_left + 1
    o, lse, cnt = _run_full(q, k, v, cfg.window_left, 0, cfg.scale, G, global_mode=oracle.GLOBAL_SINK)
    t = np.arange(cfg.T)
    want = np.minimum(t + 1, W) + np.maximum(0, np.minimum(4, t - W + 1))
    assert (cnt == want[None, None, :]).all()
    compare_every_row("mistral+4 sinks", o, lse, cnt,
                      lambda r: oracle.fwd(q, k, v, cfg.window_left, 0, cfg.scale, G, rows=r,
                                           gmode=oracle.GLOBAL_SINK), cfg.B, cfg.Hq, cfg.T)


# ----------------------------------------------------------------------------- narrow global tile
# Up to 32 global positions are scored in one 32-key tile (S with N = 32, P V with K = 32,
# a 32-column softmax); 33 or more take full-width tiles.  Both sides of that boundary,
# with globals inside and outside the bands, as full globals and as sinks.
NARROW = [
    # B, T, Hq, Hkv, d, wl, wr, G, mode
    (1, 700, 4, 2, 128, 40, 40, list(range(0, 700, 22))[:32], "full"),      # 32: narrow
    (1, 700, 4, 2, 128, 40, 40, list(range(0, 700, 21))[:33], "full"),      # 33: full width
    (2, 500, 8, 8, 64, 30, 30, [0, 1, 31, 32, 250, 498, 499], "full"),
    (1, 400, 4, 2, 256, 50, 0, list(range(32)), "sink"),                   # 32 sinks, d = 256
    (1, 400, 4, 2, 256, 50, 0, list(range(33)), "sink"),                   # 33 sinks
    (1, 300, 2, 1, 64, 20, 0, [7], "sink"),
]


@pytest.mark.parametrize("case", NARROW, ids=[f"T{c[1]}-d{c[4]}-g{len(c[7])}-{c[8]}" for c in NARROW])
def test_narrow_global_tile(case):
    B, T, Hq, Hkv, d, wl, wr, G, mode = case
    q, k, v = _inputs(7 * T + d + len(G), B, T, Hq, Hkv, d)
    scale = d ** -0.5
    gmode = oracle.GLOBAL_SINK if mode == "sink" else oracle.GLOBAL_FULL
    o, lse, cnt = _run(q, k, v, wl, wr, scale, G, global_mode=gmode)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, scale, G, gmode=gmode)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case[:7]) + f" g={len(G)} {mode}")


# ----------------------------------------------------------------------------- global projections
SEP = [
    # B, T, Hq, Hkv, d, wl, wr, G
    (1, 500, 12, 12, 64, 32, 32, [0, 250, 499]),
    (2, 300, 8, 2, 128, 40, 40, [3, 4, 5, 127, 128]),   # globals inside bands, at tile edges
    (1, 260, 4, 2, 256, 20, 0, [0, 100]),
    (1, 400, 4, 1, 64, 16, 16, list(range(0, 400, 3))),  # many globals, two global tiles
]


@pytest.mark.parametrize("case", SEP, ids=[f"T{c[1]}-d{c[4]}-wl{c[5]}-wr{c[6]}-g{len(c[7])}" for c in SEP])
def test_separate_global_projections(case):
    B, T, Hq, Hkv, d, wl, wr, G = case
    q, k, v = _inputs(5 * T + d, B, T, Hq, Hkv, d)
    qg, kg, vg = _inputs(5 * T + d + 100, B, T, Hq, Hkv, d)
    scale = d ** -0.5
    o, lse, cnt = _run(q, k, v, wl, wr, scale, G, q_g=qg, k_g=kg, v_g=vg)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, scale, G, qg=qg, kg=kg, vg=vg)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case))


def test_separate_projections_full_size_longformer():
    """Longformer-shape encoder with separate global projections: every row's O, lse
    and count against the oracle."""
    cfg = I.LONGFORMER
    q, k, v = I.prefill_inputs(cfg)
    qg = I.normal_bf16(cfg.seed * 16 + 8, q.shape)
    kg = I.normal_bf16(cfg.seed * 16 + 9, k.shape)
    vg = I.normal_bf16(cfg.seed * 16 + 10, v.shape)
    G = list(cfg.globals_)
    o, lse, cnt = _run_full(q, k, v, cfg.window_left, cfg.window_right, cfg.scale, G, q_g=qg, k_g=kg, v_g=vg)
    compare_every_row("longformer+Qg/Kg/Vg", o, lse, cnt,
                      lambda r: oracle.fwd(q, k, v, cfg.window_left, cfg.window_right, cfg.scale, G, rows=r,
                                           qg=qg, kg=kg, vg=vg), cfg.B, cfg.Hq, cfg.T)


# ----------------------------------------------------------------------------- dilation
DIL = [
    # B, T, Hq, Hkv, d, wl, wr, dilation per query head
    (1, 400, 8, 8, 64, 16, 16, [1, 1, 1, 1, 1, 1, 2, 2]),   # Longformer page 3.6 mix
    (2, 300, 8, 2, 128, 30, 0, [1, 1, 1, 1, 3, 3, 3, 3]),    # whole GQA groups share d
    (1, 333, 4, 2, 128, 20, 20, [1, 2, 4, 4]),               # a group that mixes d
    (1, 257, 2, 1, 256, 12, 3, [2, 2]),
    (1, 100, 4, 2, 64, 7, 0, [8, 8, 8, 8]),
]


@pytest.mark.parametrize("case", DIL, ids=[f"T{c[1]}-d{c[4]}-wl{c[5]}-wr{c[6]}-dil{''.join(map(str, c[7]))}" for c in DIL])
def test_dilation(case):
    B, T, Hq, Hkv, d, wl, wr, dil = case
    q, k, v = _inputs(11 * T + d, B, T, Hq, Hkv, d)
    scale = d ** -0.5
    o, lse, cnt = _run(q, k, v, wl, wr, scale, dilation=dil)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, scale, dilation=dil)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case))


def test_dilation_full_size_longformer():
    """Longformer-shape encoder, heads 8-11 dilated by 2 (no globals): every row's
    count against the residue-class closed form, every row's O and lse against the
    oracle."""
    cfg = I.LONGFORMER
    q, k, v = I.prefill_inputs(cfg)
    dil = [1] * 8 + [2] * 4
    r = cfg.window_left
    o, lse, cnt = _run_full(q, k, v, r, r, cfg.scale, dilation=dil)
    t = np.arange(cfg.T)
    for h in range(cfg.Hq):
        d = dil[h]
        want = np.minimum(r, t // d) + np.minimum(r, (cfg.T - 1 - t) // d) + 1
        assert (cnt[:, h] == want[None, :]).all(), h
    compare_every_row("longformer dilation mix", o, lse, cnt,
                      lambda rows: oracle.fwd(q, k, v, r, r, cfg.scale, rows=rows, dilation=dil),
                      cfg.B, cfg.Hq, cfg.T)


# ----------------------------------------------------------------------------- decode window / sinks
def _sink_cache(k, v, L, W, ns):
    """ns sink slots, then a W-slot ring of the positions >= ns (p at ns + (p-ns) % W)."""
    B, _, Hkv, D = k.shape
    S = ns + W
    kc = I.normal_bf16(4242, (B, Hkv, S, D))
    vc = I.normal_bf16(4243, (B, Hkv, S, D))
    pos = np.full((B, S), -1, dtype=np.int32)
    for b in range(B):
        for p in range(L[b]):
            if p < ns:
                j = p
            elif p > L[b] - 1 - W:
                j = ns + (p - ns) % W
            else:
                continue
            pos[b, j] = p
            kc[b, :, j] = k[b, p]
            vc[b, :, j] = v[b, p]
    return kc, vc, pos


@pytest.mark.parametrize("W,ns,d", [(64, 4, 128), (600, 2, 64), (100, 1, 256), (512, 0, 128)])
def test_decode_sinks_and_window(W, ns, d):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hq, Hkv = 6, 8, 2
    L = np.array([1, 3, W, W + ns + 5, 3 * W + 7, 2000])[:B]
    Tm = int(L.max())
    k = I.normal_bf16(31 + d, (B, Tm, Hkv, d))
    v = I.normal_bf16(32 + d, (B, Tm, Hkv, d))
    q = I.normal_bf16(33 + d, (B, Hq, d))
    kc, vc, pos = _sink_cache(k, v, L, W, ns)
    qpos = (L - 1).astype(np.int32)
    o, lse, cnt = swa.swa_decode(to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos), d ** -0.5,
                                 want_counts=True, window=W, n_sink=ns)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, d ** -0.5, window=W, n_sink=ns)
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref, f"W{W} ns{ns}")
    want = np.minimum(L, W) + np.maximum(0, np.minimum(ns, L - W))
    assert (cnt.cpu().numpy() == want[:, None]).all()


def test_decode_rows_without_valid_slots():
    """A sequence whose every slot is stale or in the future: the empty row gives
    O = 0, lse = -inf and count 0 (the empty-set reading of the mask); other
    sequences of the same call are unaffected."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hq, Hkv, d, W = 3, 8, 2, 128, 256
    q = I.normal_bf16(71, (B, Hq, d))
    kc = I.normal_bf16(72, (B, Hkv, W, d))
    vc = I.normal_bf16(73, (B, Hkv, W, d))
    pos = I.ring_slot_positions(np.array([300, 5, 1000]), W)
    pos[1, :] = -1          # never written
    pos[2, :] = 5000        # every slot after the query position
    qpos = np.array([299, 4, 999], dtype=np.int32)
    o, lse, cnt = swa.swa_decode(to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos), d ** -0.5,
                                 want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, d ** -0.5)
    assert (cnt_ref[1:] == 0).all()
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref, "empty rows")
    assert (to_host_f64(o)[1:] == 0).all()


def test_gqa_group_16_head_dim_256():
    B, T, Hq, Hkv, d = 1, 200, 16, 1, 256
    q, k, v = _inputs(81, B, T, Hq, Hkv, d)
    o, lse, cnt = _run(q, k, v, 50, 0, d ** -0.5)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, 50, 0, d ** -0.5)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, "G=16 d=256")


def test_decode_sinks_full_size():
    """The benchmark's decode with four pinned sink slots beside the 4096-slot ring (the
    decode workload's lengths): every row against the oracle, counts against the closed
    form min(L, W) + max(0, min(4, L - W))."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    cfg = I.DECODE
    q, kc, vc, _, qpos = I.decode_inputs(cfg)
    L = qpos.astype(np.int64) + 1
    ns = 4
    pos = I.sink_ring_slot_positions(L, cfg.W, ns)
    pad = I.normal_bf16(cfg.seed * 16 + 7, (cfg.B, cfg.Hkv, ns, cfg.d))
    kc = np.concatenate([pad, kc], axis=2)
    vc = np.concatenate([pad, vc], axis=2)
    o, lse, cnt = swa.swa_decode(to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos), cfg.scale,
                                 want_counts=True, window=cfg.W, n_sink=ns)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, cfg.scale, window=cfg.W, n_sink=ns)
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref,
                  "decode with 4 sinks, full size")
    want = np.minimum(L, cfg.W) + np.maximum(0, np.minimum(ns, L - cfg.W))
    assert (cnt.cpu().numpy() == want[:, None]).all()
