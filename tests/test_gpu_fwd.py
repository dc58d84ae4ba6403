"""swa_fwd (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from parity import assert_parity, compare_every_row, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(q, k, v, wl, wr, scale, G=None, strided=False):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    if strided:
        # q, k, v as head-slices of one packed [B, T, Hq + 2 Hkv, d] tensor
        Hq, Hkv = q.shape[2], k.shape[2]
        packed = to_dev(np.concatenate([q, k, v], axis=2))
        qd, kd, vd = packed[:, :, :Hq], packed[:, :, Hq:Hq + Hkv], packed[:, :, Hq + Hkv:]
    else:
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    g = None if G is None else i32_dev(G)
    o, lse, cnt = swa.swa_fwd(qd, kd, vd, wl, wr, scale, g, want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    # to oracle layout: o [B, Hq, T, d]
    return to_host_f64(o).transpose(0, 2, 1, 3), lse.cpu().numpy().astype(np.float64), cnt.cpu().numpy()


def test_tiny_workloads():
    """The T=16, d=64 running examples: r = 2 bidirectional and the causal W = 4 window."""
    for cfg, total in ((I.TINY_BIDIR, 74), (I.TINY_CAUSAL, 58)):
        q, k, v = I.prefill_inputs(cfg)
        o, lse, cnt = _run(q, k, v, cfg.window_left, cfg.window_right, cfg.scale)
        o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, cfg.window_left, cfg.window_right, cfg.scale)
        assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, cfg.name)
        assert int(cnt.sum()) == total


SMALL = [
    # B, T, Hq, Hkv, d, wl, wr, G
    (1, 1, 1, 1, 64, 3, 0, None),
    (2, 100, 4, 1, 64, 15, 0, None),
    (1, 300, 8, 2, 128, 63, 0, None),
    (1, 300, 8, 2, 128, 63, 5, None),
    (2, 257, 2, 2, 256, 100, 100, None),
    (1, 500, 12, 12, 64, 32, 32, [0, 250, 499]),
    (1, 400, 6, 2, 128, -1, 0, None),
    (1, 100, 4, 1, 128, 4095, 0, None),
    (1, 200, 3, 1, 64, 10, 0, None),
    (1, 333, 16, 1, 64, 40, 0, None),
    (1, 260, 4, 4, 128, 0, 0, None),
    (1, 300, 4, 2, 64, -1, -1, None),
    (1, 130, 2, 1, 128, 5, 5, list(range(130))),
    (1, 1000, 4, 2, 128, 200, 0, [3, 999]),
    (2, 700, 8, 8, 64, 256, 256, [0, 350]),
    (1, 600, 4, 2, 256, 31, 0, [17]),
    (1, 389, 8, 4, 256, 129, 70, None),
    # bands of more than eight key tiles per unit with global positions (the long-band
    # kernel; the short ones above take the short-band kernel)
    (1, 1500, 4, 2, 128, 1000, 0, [0, 3, 1499]),
    (1, 1200, 8, 8, 64, 600, 600, [0, 600, 1199]),
    # more units than persistent CTAs, each of one to five key tiles: the K/V ring runs
    # across unit boundaries (a unit's last V_j shares a barrier with the next unit's K_0)
    (8, 1024, 8, 2, 128, 63, 0, None),     # 256 units of 1-2 tiles
    (8, 1024, 8, 2, 128, 0, 0, None),      # 256 units of exactly one tile; o_t = v_t
    (2, 2048, 8, 8, 256, 99, 0, None),     # one query tile per unit: 256 units of 4-5 tiles
    (2, 2048, 8, 8, 256, 0, 0, None),      # 256 units of two 64-key tiles; o_t = v_t
    (6, 1024, 8, 4, 64, 40, 40, None),     # 192 short-band units
    # global rows at head dim 64 with grouped heads: one global-row query block of
    # 16 rows, ragged T, causal windows, an unbounded side, several sequences
    (1, 777, 8, 2, 64, 100, 100, [0, 5, 400, 776]),       # G = 4 x 4 globals = 16 rows, ragged T
    (2, 1000, 8, 2, 64, 63, 0, [10, 500, 999]),          # causal window: global rows see the future
    (1, 600, 4, 4, 64, -1, 50, [3]),                     # unbounded left side
    (3, 2048, 2, 2, 64, 256, 256, [0, 1024, 2047]),
    (1, 3000, 4, 1, 64, 700, 0, [1, 2999]),              # long band (per-fill releases), G = 4
    (1, 300, 8, 2, 64, 20, 20, [0, 100, 150, 200, 299]),  # 20 rows: two query blocks
]


@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}-T{c[1]}-Hq{c[2]}-Hkv{c[3]}-d{c[4]}-wl{c[5]}-wr{c[6]}-g{0 if c[7] is None else len(c[7])}" for c in SMALL])
def test_small_shapes(case):
    B, T, Hq, Hkv, d, wl, wr, G = case
    seed = 7 * T + d + Hq
    q = I.normal_bf16(seed, (B, T, Hq, d))
    k = I.normal_bf16(seed + 1, (B, T, Hkv, d))
    v = I.normal_bf16(seed + 2, (B, T, Hkv, d))
    scale = d ** -0.5
    o, lse, cnt = _run(q, k, v, wl, wr, scale, G)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, scale, G)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case))
    if wl == 0 and wr == 0 and not G:
        # one-key window: o_t is v_t itself (bf16 in, bf16 out)
        vv = I.bf16_bits_to_f32(v).astype(np.float64)
        for h in range(Hq):
            np.testing.assert_array_equal(o[:, h], vv[:, :, h // (Hq // Hkv), :])


def test_strided_inputs():
    B, T, Hq, Hkv, d = 2, 333, 8, 2, 128
    q = I.normal_bf16(901, (B, T, Hq, d))
    k = I.normal_bf16(902, (B, T, Hkv, d))
    v = I.normal_bf16(903, (B, T, Hkv, d))
    o, lse, cnt = _run(q, k, v, 47, 0, 0.09, [5, 200], strided=True)
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, 47, 0, 0.09, [5, 200])
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, "strided")


def test_output_with_16_byte_alignment():
    """O written through a view whose base and row strides are 16- but not 32-byte
    aligned (the kernel then stores 16 bytes at a time)."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, T, Hq, Hkv, d = 1, 300, 4, 2, 128
    q = I.normal_bf16(911, (B, T, Hq, d))
    k = I.normal_bf16(912, (B, T, Hkv, d))
    v = I.normal_bf16(913, (B, T, Hkv, d))
    buf = torch.zeros((B, T, Hq, d + 8), dtype=torch.bfloat16, device="cuda")
    o = buf[..., 8:]  # 16 bytes past a 256-byte aligned base; row stride 272 bytes
    _, lse, cnt = swa.swa_fwd(to_dev(q), to_dev(k), to_dev(v), 40, 0, d ** -0.5, o=o, want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, 40, 0, d ** -0.5)
    assert_parity(to_host_f64(o).transpose(0, 2, 1, 3), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref,
                  cnt_ref, "16-byte aligned O")
    assert (buf[..., :8] == 0).all()  # nothing written outside the view


def _closed_form_counts(T, wl, wr, G):
    t = np.arange(T)
    lo = np.zeros(T, dtype=np.int64) if wl < 0 else np.maximum(0, t - wl)
    hi = np.full(T, T - 1, dtype=np.int64) if wr < 0 else np.minimum(T - 1, t + wr)
    cnt = hi - lo + 1
    if G:
        Ga = np.asarray(G)
        outside = ((Ga[None, :] < lo[:, None]) | (Ga[None, :] > hi[:, None])).sum(axis=1)
        cnt = cnt + outside
        cnt[Ga] = T
    return cnt


def _sample_rows(cfg, rng, n_random=96):
    W = cfg.window_left + 1
    ts = {0, 1, 2, 31, 32, 127, 128, 129, W - 2, W - 1, W, W + 1, cfg.T // 2, cfg.T - 2, cfg.T - 1}
    for g in cfg.globals_:
        ts |= {g, g - 1, g + 1}
    ts |= set(int(x) for x in rng.integers(0, cfg.T, n_random))
    ts = sorted(x for x in ts if 0 <= x < cfg.T)
    rows = []
    for t in ts:
        b = int(rng.integers(0, cfg.B))
        h = int(rng.integers(0, cfg.Hq))
        rows.append((b, h, t))
    for h in range(cfg.Hq):  # every head at the last token
        rows.append((cfg.B - 1, h, cfg.T - 1))
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("cfg", [I.MISTRAL, I.GEMMA_LOCAL, I.LONGFORMER], ids=lambda c: c.name)
def test_full_size_workloads(cfg):
    """Full-size prefill / encoder workloads: every row's count against the closed form,
    then sampled edge rows (a fast first check), then every row's O and lse against the
    oracle, a few heads at a time."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    q, k, v = I.prefill_inputs(cfg)
    G = list(cfg.globals_) or None
    wl, wr = cfg.window_left, cfg.window_right
    od, lsed, cntd = swa.swa_fwd(to_dev(q), to_dev(k), to_dev(v), wl, wr, cfg.scale,
                                 None if G is None else i32_dev(G), want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o = od.cpu()  # [B, T, Hq, d] bf16
    del od
    lse, cnt = lsed.cpu().numpy().astype(np.float64), cntd.cpu().numpy()
    want = _closed_form_counts(cfg.T, wl, wr, G)
    assert (cnt == want[None, None, :]).all(), "attended-key counts differ from the closed form"
    rows = _sample_rows(cfg, np.random.default_rng(cfg.seed))
    o_ref, lse_ref, cnt_ref = oracle.fwd(q, k, v, wl, wr, cfg.scale, G, rows=rows)
    b, h, t = rows[:, 0], rows[:, 1], rows[:, 2]
    og = o[torch.from_numpy(b), torch.from_numpy(t), torch.from_numpy(h)].to(torch.float64).numpy()
    assert_parity(og, lse[b, h, t], cnt[b, h, t], o_ref, lse_ref, cnt_ref, cfg.name + " (sampled rows)")
    compare_every_row(cfg.name, o, lse, cnt, lambda r: oracle.fwd(q, k, v, wl, wr, cfg.scale, G, rows=r),
                      cfg.B, cfg.Hq, cfg.T)


RAMP = [
    # B, T, Hq, Hkv, d, wl, wr
    (1, 700, 4, 2, 128, 699, 0),   # two query tiles per unit
    (1, 700, 4, 2, 64, 300, 300),
    (1, 500, 4, 2, 256, 499, 0),   # one query tile, S double-buffered
]


@pytest.mark.parametrize("case", RAMP, ids=[f"T{c[1]}-d{c[4]}-wl{c[5]}-wr{c[6]}" for c in RAMP])
def test_growing_scores_rescale_o(case):
    """Keys whose scores grow along the sequence, by far more than 2^8 per key tile, so
    every row's running max keeps rising and O is rescaled in TMEM on every tile (the
    lazy rescale path); checked against the oracle like any other case."""
    B, T, Hq, Hkv, d, wl, wr = case
    seed = 11 * T + d
    q = I.bf16_bits_to_f32(I.normal_bf16(seed, (B, T, Hq, d))) * 0.5 + 0.5
    k = I.bf16_bits_to_f32(I.normal_bf16(seed + 1, (B, T, Hkv, d))) * 0.5
    ramp = (np.arange(T, dtype=np.float32) / 8.0)[None, :, None, None]
    k = k + ramp * 0.25   # scale * q.k grows by ~sqrt(d) * 4 per 128 keys
    v = I.normal_bf16(seed + 2, (B, T, Hkv, d))
    qb, kb = I.f32_to_bf16_bits(q.astype(np.float32)), I.f32_to_bf16_bits(k.astype(np.float32))
    scale = d ** -0.5
    o, lse, cnt = _run(qb, kb, v, wl, wr, scale, None)
    o_ref, lse_ref, cnt_ref = oracle.fwd(qb, kb, v, wl, wr, scale, None)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case))
