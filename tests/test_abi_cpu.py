"""The C-ABI library on the host: it loads, exports what include/swa.h declares,
and rejects invalid arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import sliding_window_attention_swa_gb300 as swa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swa.h")


@pytest.fixture(scope="module")
def lib():
    swa.build()
    return swa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SWA_API\s+[\w\s\*]+?\b(swa_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"swa_fwd", "swa_decode", "swa_fwd_workspace_size", "swa_decode_workspace_size",
            "swa_check_device_error", "swa_status_string", "swa_abi_version"} <= set(names)
    raw = ctypes.CDLL(swa.library_path())
    for n in names:
        assert hasattr(raw, n), n


def test_version_and_status_strings(lib):
    assert swa.swa_abi_version() == 2
    for s in range(6):
        assert swa.swa_status_string(s)
    assert "unknown" in swa.swa_status_string(99)


def test_struct_layout_matches_header(tmp_path):
    # The C compiler's sizeof / offsetof of every field against the ctypes mirrors.
    structs = {"swa_fwd_params": swa.SwaFwdParams, "swa_decode_params": swa.SwaDecodeParams,
               "swa_cache_params": swa.SwaCacheParams, "swa_chunk_params": swa.SwaChunkParams,
               "swa_device_errors": swa.SwaDeviceErrors, "swa_debug_faults": swa.SwaDebugFaults}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "swa.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    for line in subprocess.check_output([str(exe)]).decode().splitlines():
        cname, field, val = line.split()
        py = structs[cname]
        got = ctypes.sizeof(py) if field == "size" else getattr(py, field).offset
        assert got == int(val), (cname, field, got, val)


def _valid_fwd():
    p = swa.SwaFwdParams()
    fake = 0x10000
    p.q = p.k = p.v = p.o = fake
    p.lse = fake
    for name in ("q_strides", "k_strides", "v_strides", "o_strides"):
        setattr(p, name, (ctypes.c_int64 * 3)(1024 * 64, 64 * 4, 64))
    p.B, p.T, p.H_q, p.H_kv, p.d_h = 1, 1024, 4, 2, 64
    p.window_left, p.window_right = 127, 0
    p.scale = 0.125
    return p


def _valid_decode():
    p = swa.SwaDecodeParams()
    fake = 0x10000
    p.q = p.k_cache = p.v_cache = p.slot_pos = p.q_pos = p.o = p.lse = fake
    p.B, p.H_q, p.H_kv, p.d_h, p.W = 2, 8, 2, 128, 256
    p.scale = 0.1
    return p


@pytest.mark.parametrize("mutate,status", [
    (lambda p: setattr(p, "q", None), 1),
    (lambda p: setattr(p, "lse", None), 1),
    (lambda p: setattr(p, "T", 0), 1),
    (lambda p: setattr(p, "H_kv", 3), 1),
    (lambda p: setattr(p, "n_global", 2), 1),          # no global_idx pointer
    (lambda p: setattr(p, "scale", float("nan")), 1),
    (lambda p: setattr(p, "d_h", 96), 2),
    (lambda p: (setattr(p, "H_q", 34), setattr(p, "H_kv", 2)), 2),  # group 17 > 16
    (lambda p: setattr(p, "scale", -1.0), 2),
    (lambda p: setattr(p, "q", 0x10008), 2),           # misaligned
    (lambda p: setattr(p, "k_strides", (ctypes.c_int64 * 3)(100, 10, 3)), 2),
    (lambda p: setattr(p, "global_mode", 2), 1),
    (lambda p: setattr(p, "q_g", 0x10000), 1),         # q_g without k_g, v_g
    (lambda p: (setattr(p, "q_g", 0x10000), setattr(p, "k_g", 0x10000), setattr(p, "v_g", 0x10000),
                setattr(p, "global_mode", 1)), 1),      # separate projections with sinks
    (lambda p: (setattr(p, "q_g", 0x10000), setattr(p, "k_g", 0x10000), setattr(p, "v_g", 0x10000)), 2),
    (lambda p: setattr(p, "dilation", (ctypes.c_int32 * 4)(1, 0, 1, 1)), 1),
    (lambda p: (setattr(p, "dilation", (ctypes.c_int32 * 4)(1, 2, 1, 1)), setattr(p, "global_idx", 0x20000),
                setattr(p, "n_global", 1)), 2),         # dilation with globals
])
def test_fwd_rejects(lib, mutate, status):
    p = _valid_fwd()
    mutate(p)
    assert lib.swa_fwd(ctypes.byref(p), None, 0, None) == status
    assert lib.swa_fwd_workspace_size(ctypes.byref(p)) == 0


def test_fwd_workspace_needed_for_globals(lib):
    p = _valid_fwd()
    assert lib.swa_fwd_workspace_size(ctypes.byref(p)) == 0
    p.global_idx = 0x20000
    p.n_global = 2
    need = lib.swa_fwd_workspace_size(ctypes.byref(p))
    assert need > 0
    assert lib.swa_fwd(ctypes.byref(p), None, 0, None) == 5
    assert lib.swa_fwd(ctypes.byref(p), ctypes.c_void_p(0x100000), need - 1, None) == 5
    assert lib.swa_fwd(ctypes.byref(p), ctypes.c_void_p(0x100010), need, None) == 5  # not 256-B aligned
    p.global_mode = 1  # sinks: no global rows, no workspace
    assert lib.swa_fwd_workspace_size(ctypes.byref(p)) == 0


@pytest.mark.parametrize("mutate,status", [
    (lambda p: setattr(p, "slot_pos", None), 1),
    (lambda p: setattr(p, "W", 0), 1),
    (lambda p: setattr(p, "H_kv", 3), 1),
    (lambda p: setattr(p, "d_h", 80), 2),
    (lambda p: setattr(p, "v_cache", 0x10004), 2),
    (lambda p: setattr(p, "window", -1), 1),
    (lambda p: setattr(p, "n_sink", -2), 1),
])
def test_decode_rejects(lib, mutate, status):
    p = _valid_decode()
    mutate(p)
    assert lib.swa_decode(ctypes.byref(p), None, 0, None) == status


def test_decode_workspace(lib):
    p = _valid_decode()
    need = lib.swa_decode_workspace_size(ctypes.byref(p))
    assert need > 0
    assert lib.swa_decode(ctypes.byref(p), None, 0, None) == 5


def _valid_cache():
    c = swa.SwaCacheParams()
    c.k_cache = c.v_cache = c.slot_pos = 0x10000
    c.B, c.H_kv, c.d_h, c.n_slots, c.n_sink = 2, 2, 128, 256, 0
    return c


def _valid_chunk():
    p = swa.SwaChunkParams()
    p.q = p.k_new = p.v_new = p.p0 = p.o = p.lse = 0x10000
    p.B, p.C, p.H_q, p.H_kv, p.d_h = 2, 64, 8, 2, 128
    p.window, p.scale = 256, 0.1
    return p


@pytest.mark.parametrize("mutate,status", [
    (lambda c: setattr(c, "slot_pos", None), 1),
    (lambda c: setattr(c, "n_slots", 0), 1),
    (lambda c: setattr(c, "n_sink", 256), 1),      # no ring slot left
    (lambda c: setattr(c, "d_h", 96), 2),
    (lambda c: setattr(c, "k_cache", 0x10008), 2),
])
def test_cache_append_rejects(lib, mutate, status):
    c = _valid_cache()
    mutate(c)
    assert lib.swa_cache_append(ctypes.byref(c), 0x20000, 0x20000, 4, 0x30000, None) == status


def test_cache_append_arguments(lib):
    c = _valid_cache()
    assert lib.swa_cache_append(ctypes.byref(c), None, None, 0, None, None) == 0  # nothing to append
    assert lib.swa_cache_append(ctypes.byref(c), None, 0x20000, 4, 0x30000, None) == 1
    assert lib.swa_cache_append(ctypes.byref(c), 0x20000, 0x20000, -1, 0x30000, None) == 1
    assert lib.swa_cache_append(ctypes.byref(c), 0x20008, 0x20000, 4, 0x30000, None) == 2
    c.B, c.H_kv = 65536, 16
    assert lib.swa_cache_append(ctypes.byref(c), 0x20000, 0x20000, 2048, 0x30000, None) == 2  # 2^31 rows


def test_decode_append_rejects(lib):
    p = _valid_decode()
    assert lib.swa_decode_append(ctypes.byref(p), None, 0x20000, None, 0, None) == 1
    p.n_sink = p.W
    assert lib.swa_decode_append(ctypes.byref(p), 0x20000, 0x20000, None, 0, None) == 1
    p.n_sink = 0
    assert lib.swa_decode_append(ctypes.byref(p), 0x20000, 0x20000, None, 0, None) == 5  # workspace


@pytest.mark.parametrize("mutate,status", [
    (lambda p, c: setattr(p, "p0", None), 1),
    (lambda p, c: setattr(p, "window", 0), 1),
    (lambda p, c: setattr(p, "C", 0), 1),
    (lambda p, c: setattr(p, "B", 3), 1),           # cache of 2 sequences
    (lambda p, c: setattr(p, "d_h", 64), 1),        # cache head dim 128
    (lambda p, c: setattr(c, "n_sink", 4), 2),      # a sink cache whose ring (252) is shorter than window-1 (255)
    (lambda p, c: (setattr(c, "n_sink", 200), setattr(c, "n_slots", 600)), 2),  # more than 128 sinks
    (lambda p, c: setattr(p, "q", 0x10004), 2),
    (lambda p, c: (setattr(p, "B", 4096), setattr(c, "B", 4096), setattr(p, "C", 1 << 18)), 2),  # >= 2^31 rows
])
def test_prefill_chunk_rejects(lib, mutate, status):
    p, c = _valid_chunk(), _valid_cache()
    mutate(p, c)
    assert lib.swa_prefill_chunk(ctypes.byref(p), ctypes.byref(c), None, 0, None) == status
    assert lib.swa_prefill_chunk_workspace_size(ctypes.byref(p), ctypes.byref(c)) == 0


def test_prefill_chunk_workspace(lib):
    p, c = _valid_chunk(), _valid_cache()
    need = lib.swa_prefill_chunk_workspace_size(ctypes.byref(p), ctypes.byref(c))
    # gathered keys and values: B * (W - 1 + C) * H_kv * d_h bf16 each, plus kmin
    assert need >= 2 * 2 * (256 - 1 + 64) * 2 * 128 * 2
    assert lib.swa_prefill_chunk(ctypes.byref(p), ctypes.byref(c), None, 0, None) == 5


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        swa.load_library(str(tmp_path / "nope.so"))


def test_debug_fault_plan_arguments(lib):
    """The failure-detection hook takes -1 (off) or a fill / stage number; anything else
    is rejected on the host."""
    F = swa.SwaDebugFaults
    try:
        for bad in (F(-2, -1), F(-1, -5)):
            assert lib.swa_debug_set_faults(ctypes.byref(bad)) == 1
        for good in (F(-1, -1), F(0, 3), F(12, -1)):
            assert lib.swa_debug_set_faults(ctypes.byref(good)) == 0
        assert lib.swa_debug_set_faults(None) == 0
    finally:
        swa.swa_debug_set_faults()


def test_device_error_bits_match_header():
    """The Python constants mirror the header's SWA_DEVERR_* bits."""
    text = open(HEADER).read()
    bits = dict(re.findall(r"#define SWA_(DEVERR_\w+) (\d+)u", text))
    assert bits and all(getattr(swa, k) == int(v) for k, v in bits.items())
