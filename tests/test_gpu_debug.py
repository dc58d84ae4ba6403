"""The debug build of the library (libswa_debug.so, compiled with -DSWA_DEBUG).

Its kernels check every index they compute from the arguments -- key/value and query
tile coordinates, global-row gathers, output, lse and count stores, split partials,
slot positions, cache rows -- against the extent of the tensor it addresses before the
access.  A failed check sets SWA_DEVERR_BOUNDS in the kernel group's error word and
skips the access, without trapping; swa_check_device_error then reports
SWA_ERR_INVALID_ARG.

Here the small parity cases of every entry point run again, in this process, through
the debug library: the results must match the oracle as before, and no check may fire
(each case ends with swa_check_device_error, and the error words are read once more
after it).  This stands in for a memory checker, which this pool does not offer.
"""
import pytest

import test_gpu_cache as CACHE
import test_gpu_decode as DEC
import test_gpu_fwd as FWD
import test_gpu_variants as VAR

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def debug_library():
    import sliding_window_attention_swa_gb300 as swa

    lib = swa.load_library(swa.build(debug=True))
    prev = swa.use_library(lib)
    try:
        yield lib
    finally:
        swa.use_library(prev)


def _clean():
    import sliding_window_attention_swa_gb300 as swa

    assert swa.load_library()._name.endswith("libswa_debug.so")
    st, words = swa.swa_read_device_errors()
    assert st == 0 and words == {"prefill": 0, "split": 0, "cache": 0}, words


@pytest.mark.parametrize("case", FWD.SMALL, ids=[str(i) for i in range(len(FWD.SMALL))])
def test_prefill_small_shapes(case):
    FWD.test_small_shapes(case)
    _clean()


def test_prefill_layouts():
    FWD.test_tiny_workloads()
    FWD.test_strided_inputs()
    FWD.test_output_with_16_byte_alignment()
    _clean()


@pytest.mark.parametrize("case", VAR.SINKS + VAR.SEP, ids=[f"g{i}" for i in range(len(VAR.SINKS) + len(VAR.SEP))])
def test_prefill_sinks_and_projections(case):
    if case in VAR.SINKS:
        VAR.test_sinks(case)
    else:
        VAR.test_separate_global_projections(case)
    _clean()


@pytest.mark.parametrize("case", VAR.NARROW + VAR.DIL, ids=[f"v{i}" for i in range(len(VAR.NARROW) + len(VAR.DIL))])
def test_prefill_global_tiles_and_dilation(case):
    if case in VAR.NARROW:
        VAR.test_narrow_global_tile(case)
    else:
        VAR.test_dilation(case)
    _clean()


def test_decode():
    for case in DEC.CASES:
        DEC.test_decode_shapes(case)
    DEC.test_decode_stale_slots_hold_nan()
    DEC.test_decode_empty_window()
    for W, ns, d in [(64, 4, 128), (600, 2, 64), (100, 1, 256), (512, 0, 128)]:
        VAR.test_decode_sinks_and_window(W, ns, d)
    VAR.test_decode_rows_without_valid_slots()
    _clean()


def test_cache_paths():
    for case in CACHE.APPEND:
        CACHE.test_append(case)
    for W, ns, d in [(512, 0, 128), (64, 4, 128), (300, 2, 64), (100, 0, 256)]:
        CACHE.test_decode_append(W, ns, d)
    for case in CACHE.CHUNK:
        CACHE.test_prefill_chunk(case)
    for case in CACHE.CHUNK_SINKS:
        CACHE.test_prefill_chunk_with_sinks(case)
    _clean()
