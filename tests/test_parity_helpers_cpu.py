"""The whole-output comparison used by the full-size GPU tests, run on the CPU: the
oracle's own output (in the GPU's [B, T, Hq, d] layout) passes it, and a planted error
in one O element, one lse or one count fails it; a spread of small errors that keeps
every element within the max-abs bar fails the whole-output mean-abs bar."""
import numpy as np
import pytest

import oracle
import parity
from sliding_window_attention_swa_gb300 import inputs as I

B, T, Hq, Hkv, D = 2, 40, 4, 2, 64
WL, WR, SCALE = 5, 3, D ** -0.5


def _case():
    q = I.normal_bf16(6101, (B, T, Hq, D))
    k = I.normal_bf16(6102, (B, T, Hkv, D))
    v = I.normal_bf16(6103, (B, T, Hkv, D))
    o, lse, cnt = oracle.fwd(q, k, v, WL, WR, SCALE, [7])
    ref = lambda r: oracle.fwd(q, k, v, WL, WR, SCALE, [7], rows=r)  # noqa: E731
    return np.ascontiguousarray(o.transpose(0, 2, 1, 3)), lse, cnt, ref


@pytest.mark.parametrize("rows_per_slice", [1, T, 3 * T, 10 ** 6])
def test_oracle_output_passes(rows_per_slice):
    o, lse, cnt, ref = _case()
    mx, mean, lmx = parity.compare_every_row("self", o, lse, cnt, ref, B, Hq, T, rows_per_slice=rows_per_slice)
    assert mx == 0.0 and mean == 0.0 and lmx == 0.0
    assert parity.RECORDS[-1][2] == B * Hq * T * D  # every element was compared


def test_planted_errors_fail():
    o, lse, cnt, ref = _case()
    bad = o.copy()
    bad[1, 17, 3, 5] += 3 * parity.O_MAX_ABS
    with pytest.raises(AssertionError, match="max-abs"):
        parity.compare_every_row("o", bad, lse, cnt, ref, B, Hq, T)
    bad = lse.copy()
    bad[0, 2, 39] += 3 * parity.LSE_ABS
    with pytest.raises(AssertionError, match="lse"):
        parity.compare_every_row("lse", o, bad, cnt, ref, B, Hq, T)
    bad = cnt.copy()
    bad[1, 0, 0] += 1
    with pytest.raises(AssertionError, match="counts"):
        parity.compare_every_row("cnt", o, lse, bad, ref, B, Hq, T)
    # every element off by 2 mean-abs bars: each within the max-abs bar, the mean is not
    with pytest.raises(AssertionError, match="mean-abs"):
        parity.compare_every_row("mean", o + 2 * parity.O_MEAN_ABS, lse, cnt, ref, B, Hq, T, rows_per_slice=T)


def test_row_offset_maps_output_rows_to_positions():
    """t_off: output row i is position i + t_off (a chunk at the end of a sequence)."""
    o, lse, cnt, ref = _case()
    off = 25
    parity.compare_every_row("tail", o[:, off:], lse[:, :, off:], cnt[:, :, off:], ref, B, Hq, T - off, t_off=off)
    with pytest.raises(AssertionError):
        parity.compare_every_row("tail", o[:, off:], lse[:, :, off:], cnt[:, :, off:], ref, B, Hq, T - off,
                                 t_off=off - 1)
