"""Shared helpers for the GPU parity tests: device transfer and the comparison bar.

Bar (applied element by element against the fp64 oracle run on the same
bf16-rounded inputs): attended-key counts bit-exact; O max-abs error <= 2e-2
and mean-abs error <= 1e-3; lse absolute error <= 1e-3 (both -inf for an
empty row).
"""
from __future__ import annotations

import numpy as np

O_MAX_ABS = 2e-2
O_MEAN_ABS = 1e-3
LSE_ABS = 1e-3


def to_dev(bits: np.ndarray):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def i32_dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).cuda()


def to_host_f64(t) -> np.ndarray:
    import torch

    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, what=""):
    """o/lse/cnt: numpy arrays from the GPU; *_ref: oracle outputs of the same shape."""
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    if cnt is not None:
        bad = np.nonzero(np.asarray(cnt) != np.asarray(cnt_ref))
        assert len(bad[0]) == 0, f"{what}: counts differ at {len(bad[0])} rows, first {[b[0] for b in bad]}: " \
                                 f"{np.asarray(cnt)[tuple(b[0] for b in bad)]} vs {np.asarray(cnt_ref)[tuple(b[0] for b in bad)]}"
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: O max-abs error {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs error {err.mean():.3e}"
    ninf_ref = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == ninf_ref).all(), f"{what}: empty-row lse mismatch"
    fin = ~ninf_ref
    if fin.any():
        le = np.abs(lse[fin] - lse_ref[fin])
        assert le.max() <= LSE_ABS, f"{what}: lse max-abs error {le.max():.3e}"
    return float(err.max()), float(err.mean())
