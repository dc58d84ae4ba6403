"""Ring-buffer append, decode with append, and chunked prefill (through the C ABI)
against the fp64 oracle; cache contents compared bit for bit."""
import numpy as np
import pytest

import oracle
from parity import assert_parity, compare_every_row, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _bits(t) -> np.ndarray:
    import torch

    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _empty_cache(seed, B, Hkv, S, D):
    kc = I.normal_bf16(seed, (B, Hkv, S, D))
    vc = I.normal_bf16(seed + 1, (B, Hkv, S, D))
    return kc, vc, np.full((B, S), -1, dtype=np.int32)


APPEND = [
    # B, Hkv, D, n_slots, n_sink, pieces (tokens per call)
    (2, 2, 64, 16, 0, [5, 1, 11, 30]),
    (3, 8, 128, 64, 4, [1, 2, 70, 1]),
    (1, 1, 256, 9, 2, [4, 4, 4, 20]),
    (2, 4, 128, 4096, 0, [4097]),          # more tokens than slots in one call
]


@pytest.mark.parametrize("case", APPEND, ids=[f"S{c[3]}-sink{c[4]}-d{c[2]}" for c in APPEND])
def test_append(case):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hkv, D, S, ns, pieces = case
    kc, vc, pos = _empty_cache(500 + S, B, Hkv, S, D)
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    start = np.array([0, 7, 130][:B], dtype=np.int32)  # sequences at different positions
    p0 = start.copy()
    for i, n in enumerate(pieces):
        kn = I.normal_bf16(600 + i, (B, n, Hkv, D))
        vn = I.normal_bf16(700 + i, (B, n, Hkv, D))
        swa.swa_cache_append(kd, vd, pd, to_dev(kn), to_dev(vn), i32_dev(p0), n_sink=ns)
        kc, vc, pos = oracle.cache_append(kc, vc, pos, kn, vn, p0, n_sink=ns)
        p0 = p0 + n
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    np.testing.assert_array_equal(pd.cpu().numpy(), pos)
    np.testing.assert_array_equal(_bits(kd), kc)
    np.testing.assert_array_equal(_bits(vd), vc)


@pytest.mark.parametrize("W,ns,d", [(512, 0, 128), (64, 4, 128), (300, 2, 64), (100, 0, 256)])
def test_decode_append(W, ns, d):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hq, Hkv = 5, 8, 2
    S = ns + W
    L = np.array([1, 2, W, W + ns + 3, 5 * W + 11])
    kc, vc, pos = _empty_cache(800 + d, B, Hkv, S, d)
    Tm = int(L.max())
    k = I.normal_bf16(810 + d, (B, Tm, Hkv, d))
    v = I.normal_bf16(811 + d, (B, Tm, Hkv, d))
    for b in range(B):  # history: tokens 0 .. L-2 of each sequence
        if L[b] > 1:
            kb, vb, pb = oracle.cache_append(kc[b:b + 1], vc[b:b + 1], pos[b:b + 1], k[b:b + 1, :L[b] - 1],
                                             v[b:b + 1, :L[b] - 1], [0], n_sink=ns)
            kc[b], vc[b], pos[b] = kb[0], vb[0], pb[0]
    q = I.normal_bf16(812 + d, (B, Hq, d))
    kn = np.stack([k[b, L[b] - 1] for b in range(B)])  # [B, Hkv, d]
    vn = np.stack([v[b, L[b] - 1] for b in range(B)])
    qpos = (L - 1).astype(np.int32)
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    o, lse, cnt = swa.swa_decode_append(to_dev(q), kd, vd, pd, i32_dev(qpos), to_dev(kn), to_dev(vn), d ** -0.5,
                                        want_counts=True, window=W, n_sink=ns)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    # oracle: append the token, then decode
    kc2, vc2, pos2 = kc.copy(), vc.copy(), pos.copy()
    for b in range(B):
        kb, vb, pb = oracle.cache_append(kc2[b:b + 1], vc2[b:b + 1], pos2[b:b + 1], kn[b:b + 1, None],
                                         vn[b:b + 1, None], [qpos[b]], n_sink=ns)
        kc2[b], vc2[b], pos2[b] = kb[0], vb[0], pb[0]
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc2, vc2, pos2, qpos, d ** -0.5, window=W, n_sink=ns)
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref, f"W{W} ns{ns}")
    np.testing.assert_array_equal(pd.cpu().numpy(), pos2)
    np.testing.assert_array_equal(_bits(kd), kc2)
    np.testing.assert_array_equal(_bits(vd), vc2)


CHUNK = [
    # B, C, Hq, Hkv, d, W, n_slots, p0 per sequence
    (2, 100, 4, 2, 128, 64, 64, [0, 37]),
    (3, 300, 8, 2, 128, 256, 256, [0, 100, 1000]),
    (2, 129, 8, 8, 64, 128, 200, [5, 700]),        # ring longer than the window
    (2, 64, 4, 1, 256, 128, 40, [10, 300]),        # ring shorter than the window
    (1, 600, 4, 2, 128, 100, 100, [3000]),         # chunk longer than the window
    (2, 1, 8, 2, 128, 64, 64, [0, 500]),           # one-token chunks, one without history
]


@pytest.mark.parametrize("case", CHUNK, ids=[f"C{c[1]}-d{c[4]}-W{c[5]}-S{c[6]}" for c in CHUNK])
def test_prefill_chunk(case):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, C, Hq, Hkv, d, W, S, p0 = case
    p0 = np.array(p0, dtype=np.int32)
    kc, vc, pos = _empty_cache(900 + C, B, Hkv, S, d)
    Tm = int(p0.max())
    kh = I.normal_bf16(910 + C, (B, max(Tm, 1), Hkv, d))
    vh = I.normal_bf16(911 + C, (B, max(Tm, 1), Hkv, d))
    for b in range(B):  # history 0 .. p0-1
        if p0[b]:
            kb, vb, pb = oracle.cache_append(kc[b:b + 1], vc[b:b + 1], pos[b:b + 1], kh[b:b + 1, :p0[b]],
                                             vh[b:b + 1, :p0[b]], [0])
            kc[b], vc[b], pos[b] = kb[0], vb[0], pb[0]
    q = I.normal_bf16(912 + C, (B, C, Hq, d))
    kn = I.normal_bf16(913 + C, (B, C, Hkv, d))
    vn = I.normal_bf16(914 + C, (B, C, Hkv, d))
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    o, lse, cnt = swa.swa_prefill_chunk(to_dev(q), to_dev(kn), to_dev(vn), kd, vd, pd, i32_dev(p0), W, d ** -0.5,
                                        append=True, want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.chunk(q, kn, vn, kc, vc, pos, p0, W, d ** -0.5)
    assert_parity(to_host_f64(o).transpose(0, 2, 1, 3), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref,
                  cnt_ref, str(case))
    kc2, vc2, pos2 = oracle.cache_append(kc, vc, pos, kn, vn, p0)
    np.testing.assert_array_equal(pd.cpu().numpy(), pos2)
    np.testing.assert_array_equal(_bits(kd), kc2)
    np.testing.assert_array_equal(_bits(vd), vc2)


CHUNK_SINKS = [
    # B, C, Hq, Hkv, d, W, n_sink, ring slots, p0 per sequence
    (2, 100, 4, 2, 128, 64, 4, 74, [0, 300]),      # p0 = 0: the sinks are inside the chunk
    (1, 200, 8, 2, 64, 100, 2, 99, [3]),
    (2, 64, 4, 1, 256, 32, 1, 40, [1000, 7]),
    (1, 300, 4, 2, 128, 64, 128, 64, [500]),       # the largest sink count
]


@pytest.mark.parametrize("case", CHUNK_SINKS, ids=[f"C{c[1]}-d{c[4]}-W{c[5]}-ns{c[6]}" for c in CHUNK_SINKS])
def test_prefill_chunk_with_sinks(case):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, C, Hq, Hkv, d, W, ns, R, p0 = case
    p0 = np.array(p0, dtype=np.int32)
    S = ns + R
    kc, vc, pos = _empty_cache(960 + C, B, Hkv, S, d)
    Tm = int(p0.max())
    kh = I.normal_bf16(961 + C, (B, max(Tm, 1), Hkv, d))
    vh = I.normal_bf16(962 + C, (B, max(Tm, 1), Hkv, d))
    for b in range(B):
        if p0[b]:
            kb, vb, pb = oracle.cache_append(kc[b:b + 1], vc[b:b + 1], pos[b:b + 1], kh[b:b + 1, :p0[b]],
                                             vh[b:b + 1, :p0[b]], [0], n_sink=ns)
            kc[b], vc[b], pos[b] = kb[0], vb[0], pb[0]
    q = I.normal_bf16(963 + C, (B, C, Hq, d))
    kn = I.normal_bf16(964 + C, (B, C, Hkv, d))
    vn = I.normal_bf16(965 + C, (B, C, Hkv, d))
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    o, lse, cnt = swa.swa_prefill_chunk(to_dev(q), to_dev(kn), to_dev(vn), kd, vd, pd, i32_dev(p0), W, d ** -0.5,
                                        append=True, want_counts=True, n_sink=ns)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.chunk(q, kn, vn, kc, vc, pos, p0, W, d ** -0.5, n_sink=ns)
    assert_parity(to_host_f64(o).transpose(0, 2, 1, 3), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref,
                  cnt_ref, str(case))
    kc2, vc2, pos2 = oracle.cache_append(kc, vc, pos, kn, vn, p0, n_sink=ns)
    np.testing.assert_array_equal(pd.cpu().numpy(), pos2)
    np.testing.assert_array_equal(_bits(kd), kc2)
    np.testing.assert_array_equal(_bits(vd), vc2)


def test_prefill_chunk_reports_missing_history():
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, C, Hq, Hkv, d, W = 1, 32, 4, 2, 64, 64
    kc, vc, pos = _empty_cache(950, B, Hkv, W, d)  # nothing appended: the history is missing
    q = I.normal_bf16(951, (B, C, Hq, d))
    kn = I.normal_bf16(952, (B, C, Hkv, d))
    swa.swa_prefill_chunk(to_dev(q), to_dev(kn), to_dev(kn), to_dev(kc), to_dev(vc), i32_dev(pos),
                          i32_dev([100]), W)
    torch.cuda.synchronize()
    with pytest.raises(swa.SwaError) as e:
        swa.swa_check_device_error()
    assert e.value.status == 1


def test_prefill_chunk_full_size_mistral():
    """The last 4096 tokens of the Mistral-shape sequence as one chunk against a
    4096-slot ring holding tokens 8192 .. 12287 (appended by the library): every
    row's count is min(t+1, W) and every row matches the full-sequence prefill."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    cfg = I.MISTRAL
    W, C = cfg.window_left + 1, 4096
    p0 = cfg.T - C
    q, k, v = I.prefill_inputs(cfg)
    kd = torch.empty((1, cfg.Hkv, W, cfg.d), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    pd = torch.full((1, W), -1, dtype=torch.int32, device="cuda")
    kdev, vdev = to_dev(k), to_dev(v)
    swa.swa_cache_append(kd, vd, pd, kdev[:, :p0].contiguous(), vdev[:, :p0].contiguous(), i32_dev([0]))
    o, lse, cnt = swa.swa_prefill_chunk(to_dev(q[:, p0:]), kdev[:, p0:].contiguous(), vdev[:, p0:].contiguous(),
                                        kd, vd, pd, i32_dev([p0]), W, cfg.scale, want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    cnt = cnt.cpu().numpy()
    assert (cnt == W).all()
    compare_every_row("mistral chunk (last 4096 tokens)", o.cpu(), lse.cpu().numpy().astype(np.float64), cnt,
                      lambda r: oracle.fwd(q, k, v, W - 1, 0, cfg.scale, rows=r), 1, cfg.Hq, C, t_off=p0)


def _decode_workload_on_device():
    cfg = I.DECODE
    q, kc, vc, pos, qpos = I.decode_inputs(cfg)
    return cfg, q, kc, vc, pos, qpos


def test_append_full_size():
    """The appended block of the benchmark: 512 new tokens for each of the 64 decode
    sequences (after their lengths), into the 4096-slot rings of the decode workload;
    the whole cache and every slot position compared bit for bit with the oracle."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    cfg, _, kc, vc, pos, qpos = _decode_workload_on_device()
    L = qpos.astype(np.int64) + 1
    n_app = 512
    kn = I.normal_bf16(cfg.seed * 16 + 11, (cfg.B, n_app, cfg.Hkv, cfg.d))
    vn = I.normal_bf16(cfg.seed * 16 + 12, (cfg.B, n_app, cfg.Hkv, cfg.d))
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    swa.swa_cache_append(kd, vd, pd, to_dev(kn), to_dev(vn), i32_dev(L.astype(np.int32)))
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    kc2, vc2, pos2 = oracle.cache_append(kc, vc, pos, kn, vn, L.astype(np.int32))
    np.testing.assert_array_equal(pd.cpu().numpy(), pos2)
    np.testing.assert_array_equal(_bits(kd), kc2)
    np.testing.assert_array_equal(_bits(vd), vc2)


def test_decode_append_full_size():
    """Decode with the current token appended in the same pass, on the full decode
    workload (the benchmark's call): every row against the oracle's decode of the cache
    with that token appended, and the appended rows and positions bit for bit."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    cfg, q, kc, vc, pos, qpos = _decode_workload_on_device()
    k1 = I.normal_bf16(cfg.seed * 16 + 13, (cfg.B, cfg.Hkv, cfg.d))
    v1 = I.normal_bf16(cfg.seed * 16 + 14, (cfg.B, cfg.Hkv, cfg.d))
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    o, lse, cnt = swa.swa_decode_append(to_dev(q), kd, vd, pd, i32_dev(qpos), to_dev(k1), to_dev(v1), cfg.scale,
                                        want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    kc2, vc2, pos2 = oracle.cache_append(kc, vc, pos, k1[:, None], v1[:, None], qpos)
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc2, vc2, pos2, qpos, cfg.scale)
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref,
                  "decode with append, full size")
    np.testing.assert_array_equal(pd.cpu().numpy(), pos2)
    np.testing.assert_array_equal(_bits(kd), kc2)
    np.testing.assert_array_equal(_bits(vd), vc2)
