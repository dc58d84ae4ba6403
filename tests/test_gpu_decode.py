"""swa_decode (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from parity import assert_parity, i32_dev, to_dev, to_host_f64
from sliding_window_attention_swa_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(q, kc, vc, pos, qpos, scale):
    import torch
    import sliding_window_attention_swa_gb300 as swa

    o, lse, cnt = swa.swa_decode(to_dev(q), to_dev(kc), to_dev(vc), i32_dev(pos), i32_dev(qpos), scale,
                                 want_counts=True)
    torch.cuda.synchronize()
    swa.swa_check_device_error()
    return to_host_f64(o), lse.cpu().numpy().astype(np.float64), cnt.cpu().numpy()


def test_decode_workload_full():
    """The 64-sequence, W=4096, GQA 32/8, d=128 ring-buffer workload; every row."""
    cfg = I.DECODE
    q, kc, vc, pos, qpos = I.decode_inputs(cfg)
    o, lse, cnt = _run(q, kc, vc, pos, qpos, cfg.scale)
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, cfg.scale)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, "decode workload")
    L = qpos.astype(np.int64) + 1
    assert (cnt == np.minimum(L, cfg.W)[:, None]).all()


CASES = [
    # B, Hq, Hkv, d, W, lengths
    (3, 4, 1, 64, 64, [1, 64, 1000]),
    (2, 8, 2, 128, 37, [5, 37, 38]),
    (2, 16, 1, 128, 1, [1, 9]),
    (4, 2, 2, 256, 600, [1, 599, 600, 5000]),
    (2, 16, 16, 64, 513, [512, 100000]),
    (2, 32, 2, 128, 1024, [700, 1500]),
    (1, 12, 12, 64, 4096, [4097]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}-Hq{c[1]}-Hkv{c[2]}-d{c[3]}-W{c[4]}" for c in CASES])
def test_decode_shapes(case):
    B, Hq, Hkv, d, W, lengths = case
    L = np.array(lengths[:B] + [lengths[-1]] * (B - len(lengths)), dtype=np.int64)
    seed = 1000 + W + d
    q = I.normal_bf16(seed, (B, Hq, d))
    kc = I.normal_bf16(seed + 1, (B, Hkv, W, d))
    vc = I.normal_bf16(seed + 2, (B, Hkv, W, d))
    pos = I.ring_slot_positions(L, W)
    qpos = (L - 1).astype(np.int32)
    scale = d ** -0.5
    o, lse, cnt = _run(q, kc, vc, pos, qpos, scale)
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, scale)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, str(case))


def test_decode_stale_slots_hold_nan():
    """Slots that are not attended may hold any bits (here NaN); results stay exact."""
    B, Hq, Hkv, d, W = 2, 8, 2, 128, 256
    L = np.array([100, 3000])
    q = I.normal_bf16(71, (B, Hq, d))
    kc = I.normal_bf16(72, (B, Hkv, W, d))
    vc = I.normal_bf16(73, (B, Hkv, W, d))
    pos = I.ring_slot_positions(L, W)
    qpos = (L - 1).astype(np.int32)
    stale = (pos < 0) | (pos > qpos[:, None]) | (pos <= qpos[:, None] - W)
    kc2, vc2 = kc.copy(), vc.copy()
    for b in range(B):
        kc2[b][:, stale[b]] = 0x7FC0  # bf16 NaN
        vc2[b][:, stale[b]] = 0x7FC0
    o, lse, cnt = _run(q, kc2, vc2, pos, qpos, 0.1)
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, 0.1)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, "nan in stale slots")


def test_decode_empty_window():
    """No slot in the window: o = 0, lse = -inf, count 0 (the oracle's empty-row convention)."""
    B, Hq, Hkv, d, W = 2, 4, 1, 64, 128
    q = I.normal_bf16(81, (B, Hq, d))
    kc = I.normal_bf16(82, (B, Hkv, W, d))
    vc = I.normal_bf16(83, (B, Hkv, W, d))
    pos = np.full((B, W), -1, dtype=np.int32)
    pos[1, 5] = 40  # sequence 1 has exactly one valid slot
    qpos = np.array([10, 40], dtype=np.int32)
    o, lse, cnt = _run(q, kc, vc, pos, qpos, 0.125)
    o_ref, lse_ref, cnt_ref = oracle.decode(q, kc, vc, pos, qpos, 0.125)
    assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, "empty window")
    assert (o[0] == 0).all() and np.isneginf(lse[0]).all() and (cnt[0] == 0).all()
    assert (cnt[1] == 1).all()
