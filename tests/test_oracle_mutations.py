"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutation is applied to a temporary copy of oracle/swa_oracle.c compiled
on the CPU; the oracle itself is never modified.  A mutation that every pin
accepts would mean the pins cannot tell that mistake from the definition.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "swa_oracle.c")

MUTATIONS = {
    "left-edge-off-by-one": ("k >= -wl", "k > -wl"),
    "right-edge-off-by-one": ("k <= wr", "k < wr"),
    "global-row-dropped": ("in_band || row_is_global ||", "in_band ||"),
    "global-column-dropped": ("int column = is_member(G, nG, s);", "int column = 0;"),
    "scale-dropped": ("x[i] = scale * dot;", "x[i] = dot;"),
    "lse-max-term-dropped": ("*lse = m + log(l);", "*lse = log(l);"),
    "max-sign-flipped": ("const double p = exp(x[i] - m);", "const double p = exp(x[i] + m);"),
    "k-and-v-swapped": ("dot += q[c] * widen_bf16(krow[i][c]);", "dot += q[c] * widen_bf16(vrow[i][c]);"),
    "gqa-interleaved-map": ("const int64_t kvh = h / group;", "const int64_t kvh = h % Hkv;"),
    "decode-window-off-by-one": ("p > t - W", "p >= t - W"),
    "decode-future-allowed": ("p >= 0 && p <= t &&", "p >= 0 &&"),
    "decode-never-written-allowed": ("return p >= 0 && ", "return "),
    "normaliser-dropped": ("for (int64_t c = 0; c < D; ++c) o[c] /= l;", ""),
    "dilation-grid-dropped": ("const int on_grid = off % dil == 0;", "const int on_grid = 1;"),
    "dilation-steps-unscaled": ("const int64_t k = off / dil;", "const int64_t k = off;"),
    "sink-reach-dropped": ("if (gmode == 1) column = column && (wr < 0 || off <= (int64_t)wr * dil);", ""),
    "sink-row-opened": ("const int row_is_global = gmode == 0 && is_member(G, nG, t);",
                        "const int row_is_global = is_member(G, nG, t);"),
    "global-proj-local-keys": ("const int from_global = separate && (row_global || is_member(G, nG, s));",
                               "const int from_global = separate && row_global;"),
    "global-proj-query": ("(row_global ? qg : q)", "q"),
    "decode-sink-dropped": (" || p < n_sink", ""),
    "decode-sink-off-by-one": ("p < n_sink", "p <= n_sink"),
    "append-slot-shift": ("n_sink + (p - n_sink) % (S - n_sink);", "n_sink + (p + 1 - n_sink) % (S - n_sink);"),
    "append-sinks-ignored": ("const int64_t j = p < n_sink ? p : n_sink + (p - n_sink) % (S - n_sink);",
                             "const int64_t j = p % S;"),
    "append-order-reversed": ("const int64_t p = (int64_t)p0[b] + i;", "const int64_t p = (int64_t)p0[b] + (n - 1 - i);"),
    "chunk-history-overlap": ("if (p < p0[b] && slot_allowed", "if (slot_allowed"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "swa_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mutated), "-o", str(so), "-lm"])
    lib = oracle.load(str(so))
    caught = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, f"no pin detects mutation {name}"
