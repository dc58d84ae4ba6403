"""Shared helpers for the GPU parity tests: device transfer and the comparison bar.

Bar (applied element by element against the fp64 oracle run on the same
bf16-rounded inputs): attended-key counts bit-exact; O max-abs error <= 2e-2
and mean-abs error <= 1e-3; lse absolute error <= 1e-3 (both -inf for an
empty row).

``compare_every_row`` applies the bar to a whole full-size output: the oracle
runs over bounded slices of rows (a few heads at a time, so host memory stays
small), the element checks run per slice, and the mean-abs bar is taken over
every element of the output, not over a sample.
"""
from __future__ import annotations

import numpy as np

O_MAX_ABS = 2e-2
O_MEAN_ABS = 1e-3
LSE_ABS = 1e-3

# (what, rows, O elements, O max-abs, O mean-abs, lse max-abs) of every whole-output
# comparison in this session, for the terminal summary (tests/conftest.py)
RECORDS: list[tuple] = []


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


def _check_elements(o, lse, cnt, o_ref, lse_ref, cnt_ref, what):
    """Per-element part of the bar; returns (O abs errors, lse max-abs error)."""
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    if cnt is not None:
        bad = np.nonzero(np.asarray(cnt) != np.asarray(cnt_ref))
        assert len(bad[0]) == 0, f"{what}: counts differ at {len(bad[0])} rows, first {[b[0] for b in bad]}: " \
                                 f"{np.asarray(cnt)[tuple(b[0] for b in bad)]} vs {np.asarray(cnt_ref)[tuple(b[0] for b in bad)]}"
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    assert err.max(initial=0.0) <= O_MAX_ABS, \
        f"{what}: O max-abs error {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    ninf_ref = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == ninf_ref).all(), f"{what}: empty-row lse mismatch"
    fin = ~ninf_ref
    le = float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert le <= LSE_ABS, f"{what}: lse max-abs error {le:.3e}"
    return err, le


def assert_parity(o, lse, cnt, o_ref, lse_ref, cnt_ref, what=""):
    """o/lse/cnt: numpy arrays from the GPU; *_ref: oracle outputs of the same shape."""
    err, _ = _check_elements(o, lse, cnt, o_ref, lse_ref, cnt_ref, what)
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs error {err.mean():.3e}"
    return float(err.max()), float(err.mean())


def compare_every_row(what, o, lse, cnt, ref, B, Hq, T, t_off=0, rows_per_slice=32768):
    """Every row of a [B, T, Hq, d] output against the oracle, a few heads at a time.

    o: the GPU's O on the host, [B, T, Hq, d] (a torch CPU tensor of any float dtype
    or a numpy array); lse, cnt: numpy [B, Hq, T].  ref(rows) runs the oracle on the
    int64 (b, h, t + t_off) triples `rows` and returns (o [n, d], lse [n], counts [n]).
    Counts must match bit for bit, every O element within O_MAX_ABS, every lse within
    LSE_ABS, and the mean of |O - O_ref| over the whole output within O_MEAN_ABS.
    Returns (O max-abs, O mean-abs, lse max-abs) over the whole output.
    """
    import torch

    if isinstance(o, np.ndarray):
        o = torch.from_numpy(o)
    heads = max(1, min(Hq, rows_per_slice // max(T, 1)))
    tt = np.arange(T, dtype=np.int64)
    n_el, s_abs, mx, lmx = 0, 0.0, 0.0, 0.0
    for b in range(B):
        for h0 in range(0, Hq, heads):
            h1 = min(Hq, h0 + heads)
            hs = np.arange(h0, h1, dtype=np.int64)
            rows = np.stack([np.full(len(hs) * T, b, dtype=np.int64), np.repeat(hs, T),
                             np.tile(tt + t_off, len(hs))], axis=1)
            o_ref, lse_ref, cnt_ref = ref(rows)
            og = o[b, :, h0:h1, :].to(torch.float64).transpose(0, 1).reshape(len(hs) * T, -1).numpy()
            lg = np.asarray(lse[b, h0:h1, :], dtype=np.float64).reshape(-1)
            cg = None if cnt is None else np.asarray(cnt[b, h0:h1, :]).reshape(-1)
            err, le = _check_elements(og, lg, cg, o_ref, lse_ref, cnt_ref, f"{what} (b={b}, heads {h0}..{h1 - 1})")
            n_el += err.size
            s_abs += float(err.sum())
            mx = max(mx, float(err.max(initial=0.0)))
            lmx = max(lmx, le)
    mean = s_abs / max(n_el, 1)
    RECORDS.append((what, B * Hq * T, n_el, mx, mean, lmx))
    assert mean <= O_MEAN_ABS, f"{what}: O mean-abs error over the whole output {mean:.3e}"
    return mx, mean, lmx
