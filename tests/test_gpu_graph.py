"""Calls captured in a CUDA graph, as a serving loop replays its decode step: a replay
gives the same bits as the eager call, and follows new inputs written into the
captured buffers (checked against the fp64 oracle).  The split pass and its merge are
launched back to back with a programmatic dependency, which the capture must keep."""
import numpy as np
import pytest

import oracle
from parity import assert_parity, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _capture(fn):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_graph_replay():
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hq, Hkv, d, W = 8, 32, 8, 128, 2048
    L = np.array([1, 100, 2047, 2048, 2049, 5000, 70000, 3], dtype=np.int64)
    seed = 4200
    q = I.normal_bf16(seed, (B, Hq, d))
    kc = I.normal_bf16(seed + 1, (B, Hkv, W, d))
    vc = I.normal_bf16(seed + 2, (B, Hkv, W, d))
    pos = I.ring_slot_positions(L, W)
    qpos = (L - 1).astype(np.int32)
    scale = d ** -0.5
    qd, kd, vd, pd, qpd = to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos)
    o = torch.empty_like(qd)
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    cnt = torch.empty((B, Hq), dtype=torch.int32, device="cuda")
    p = swa.decode_params(qd, kd, vd, pd, qpd, scale, o, lse, cnt)
    ws = torch.empty(max(1, swa.swa_decode_workspace_size(p)), dtype=torch.uint8, device="cuda")

    def step():
        swa.swa_decode(qd, kd, vd, pd, qpd, scale, o=o, lse=lse, row_counts=cnt, workspace=ws)

    step()
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_e, lse_e, cnt_e = o.clone(), lse.clone(), cnt.clone()
    g = _capture(step)
    o.zero_()
    lse.zero_()
    cnt.zero_()
    g.replay()
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    assert torch.equal(o, o_e) and torch.equal(lse, lse_e) and torch.equal(cnt, cnt_e)

    # new queries and one sequence moved on by a token: the replay follows the buffers
    q2 = I.normal_bf16(seed + 3, (B, Hq, d))
    qpos2 = qpos.copy()
    qpos2[2] += 1
    pos2 = pos.copy()
    pos2[2, qpos2[2] % W] = qpos2[2]
    qd.copy_(to_dev(q2))
    qpd.copy_(i32_dev(qpos2))
    pd.copy_(i32_dev(pos2))
    g.replay()
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.decode(q2, kc, vc, pos2, qpos2, scale)
    assert_parity(to_host_f64(o), lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref, "decode replay")


def test_decode_append_graph_steps():
    """Three serving steps replayed from one graph: each appends its token's K/V to the
    ring and attends to it; the host only rewrites q, k_new, v_new and q_pos."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, Hq, Hkv, d, W, ns = 3, 8, 2, 64, 128, 4
    S = W + ns
    L0 = np.array([1, 130, 400], dtype=np.int64)  # tokens already cached
    seed = 4300
    steps = 3
    Tm = int(L0.max()) + steps
    k = I.normal_bf16(seed, (B, Tm, Hkv, d))
    v = I.normal_bf16(seed + 1, (B, Tm, Hkv, d))
    kc = np.zeros((B, Hkv, S, d), dtype=np.uint16)
    vc = np.zeros((B, Hkv, S, d), dtype=np.uint16)
    pos = np.full((B, S), -1, dtype=np.int32)
    for b in range(B):
        kb, vb, pb = oracle.cache_append(kc[b:b + 1], vc[b:b + 1], pos[b:b + 1], k[b:b + 1, :L0[b]],
                                         v[b:b + 1, :L0[b]], [0], n_sink=ns)
        kc[b], vc[b], pos[b] = kb[0], vb[0], pb[0]
    scale = d ** -0.5
    kd, vd, pd = to_dev(kc), to_dev(vc), i32_dev(pos)
    qd = to_dev(np.zeros((B, Hq, d), dtype=np.uint16))
    knd = to_dev(np.zeros((B, Hkv, d), dtype=np.uint16))
    vnd = to_dev(np.zeros((B, Hkv, d), dtype=np.uint16))
    qpd = i32_dev(L0.astype(np.int32))
    o = torch.empty_like(qd)
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    p = swa.decode_params(qd, kd, vd, pd, qpd, scale, o, lse, None, W, ns)
    ws = torch.empty(max(1, swa.swa_decode_workspace_size(p)), dtype=torch.uint8, device="cuda")

    def step():
        swa.swa_decode_append(qd, kd, vd, pd, qpd, knd, vnd, scale, o=o, lse=lse, workspace=ws, window=W, n_sink=ns)

    g = None
    for i in range(steps):
        t = (L0 + i).astype(np.int32)
        q = I.normal_bf16(seed + 10 + i, (B, Hq, d))
        kn = np.stack([k[b, t[b]] for b in range(B)])
        vn = np.stack([v[b, t[b]] for b in range(B)])
        qd.copy_(to_dev(q))
        knd.copy_(to_dev(kn))
        vnd.copy_(to_dev(vn))
        qpd.copy_(i32_dev(t))
        if g is None:
            # capturing records the launches without running them: nothing is appended here
            g = _capture(step)
        g.replay()
        torch.cuda.synchronize()
        swa.swa_check_device_error()
        for b in range(B):
            kb, vb, pb = oracle.cache_append(kc[b:b + 1], vc[b:b + 1], pos[b:b + 1], kn[b:b + 1, None],
                                             vn[b:b + 1, None], [t[b]], n_sink=ns)
            kc[b], vc[b], pos[b] = kb[0], vb[0], pb[0]
        o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, t, scale, window=W, n_sink=ns)
        assert_parity(to_host_f64(o), lse.cpu().numpy(), None, o_ref, lse_ref, None, f"step {i}")
        np.testing.assert_array_equal(pd.cpu().numpy(), pos)


def test_fwd_with_global_rows_graph_replay():
    """Band kernel, global-row split pass and its merge, captured together."""
    import torch
    import sliding_window_attention_swa_gb300 as swa

    B, T, H, d, r = 2, 1000, 4, 64, 64
    G = np.array([0, 3, 500, 999], dtype=np.int32)
    seed = 4400
    q = I.normal_bf16(seed, (B, T, H, d))
    k = I.normal_bf16(seed + 1, (B, T, H, d))
    v = I.normal_bf16(seed + 2, (B, T, H, d))
    scale = d ** -0.5
    qd, kd, vd, gd = to_dev(q), to_dev(k), to_dev(v), i32_dev(G)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    cnt = torch.empty((B, H, T), dtype=torch.int32, device="cuda")
    p = swa.fwd_params(qd, kd, vd, r, r, scale, gd, o, lse, cnt)
    ws = torch.empty(max(1, swa.swa_fwd_workspace_size(p)), dtype=torch.uint8, device="cuda")

    def run():
        swa.swa_fwd(qd, kd, vd, r, r, scale, gd, o=o, lse=lse, row_counts=cnt, workspace=ws)

    run()
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_e, lse_e, cnt_e = o.clone(), lse.clone(), cnt.clone()
    g = _capture(run)
    o.zero_()
    lse.zero_()
    cnt.zero_()
    g.replay()
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    assert torch.equal(o, o_e) and torch.equal(lse, lse_e) and torch.equal(cnt, cnt_e)

    q2 = I.normal_bf16(seed + 3, (B, T, H, d))
    qd.copy_(to_dev(q2))
    g.replay()
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    o_ref, lse_ref, cnt_ref = oracle.fwd(q2, k, v, r, r, scale, G)
    o_h = to_host_f64(o).transpose(0, 2, 1, 3)
    assert_parity(o_h, lse.cpu().numpy(), cnt.cpu().numpy(), o_ref, lse_ref, cnt_ref, "fwd replay")
