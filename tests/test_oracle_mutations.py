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
    "left-edge-off-by-one": ("s >= t - wl", "s > t - wl"),
    "right-edge-off-by-one": ("s <= t + wr", "s < t + wr"),
    "global-row-dropped": ("in_band || row_is_global ||", "in_band ||"),
    "global-column-dropped": ("|| is_member(G, nG, s))", ")"),
    "scale-dropped": ("x[i] = scale * dot;", "x[i] = dot;"),
    "lse-max-term-dropped": ("*lse = m + log(l);", "*lse = log(l);"),
    "max-sign-flipped": ("const double p = exp(x[i] - m);", "const double p = exp(x[i] + m);"),
    "k-and-v-swapped": ("dot += q[c] * widen_bf16(krow[i][c]);", "dot += q[c] * widen_bf16(vrow[i][c]);"),
    "gqa-interleaved-map": ("const int64_t kvh = h / group;", "const int64_t kvh = h % Hkv;"),
    "decode-window-off-by-one": ("p > t - W && p <= t", "p >= t - W && p <= t"),
    "decode-future-allowed": ("p > t - W && p <= t", "p > t - W"),
    "decode-never-written-allowed": ("if (p >= 0 && p > t - W", "if (p > t - W"),
    "normaliser-dropped": ("for (int64_t c = 0; c < D; ++c) o[c] /= l;", ""),
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
