"""The C-ABI library loads on a machine without a GPU and exports every entry
point include/gaac.h declares; host-side validation and the pure-host helpers
answer without touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from lossless_compressed_kv_gaac_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "gaac.h")).read()
    names = re.findall(r"GAAC_API\s+[\w\s\*]+?\b(gaac_\w+)\s*\(", text)
    assert len(names) >= 9
    return names


def test_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_timeline_only_in_the_instrumented_build(lib):
    """gaac_timeline_fetch (include/gaac_timeline.h) exists only in the library built with the timeline; the
    default library carries no instrumentation.  With a NULL destination it reports the record sizes without
    touching a device."""
    from lossless_compressed_kv_gaac_gb300 import build

    assert not hasattr(lib, "gaac_timeline_fetch")
    tl = ctypes.CDLL(build.build(timeline=True))
    tl.gaac_timeline_fetch.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p]
    cb, nc, nb = ctypes.c_size_t(), ctypes.c_int(), ctypes.c_int()
    assert tl.gaac_timeline_fetch(None, 0, ctypes.byref(cb), ctypes.byref(nc), ctypes.byref(nb)) == 0
    assert cb.value == 8 * (4 + 4 * nb.value) and nc.value >= 152


def test_host_helpers(lib):
    lib.gaac_strerror.restype = ctypes.c_char_p
    assert lib.gaac_strerror(0) == b"ok"
    assert lib.gaac_strerror(1) == b"invalid argument"
    assert lib.gaac_format_version() == 3
    lib.gaac_attention_workspace.restype = ctypes.c_size_t
    # (16 m,l floats + 8 heads x 128 acc floats) x 4 bytes per (sequence, kv-head, split),
    # then one 4-byte merge counter per (sequence, kv-head), rounded up to 16 bytes
    assert lib.gaac_attention_workspace(1, 8, 1024, 38) == 1 * 8 * 38 * (16 + 8 * 128) * 4 + 32
    assert lib.gaac_attention_workspace(3, 4, 10, 5) == 3 * 4 * 5 * 1040 * 4 + 48


def test_null_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    EINVAL = 1
    lib.gaac_decode_attention.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P,
                                          ctypes.c_float, ctypes.c_int, P, P, ctypes.c_size_t, P, P]
    assert lib.gaac_decode_attention(None, 1, 32, 8, 16, None, None, None, None, None, 0.1, 0, None, None, 0, None,
                                     None) == EINVAL
    lib.gaac_encode_blocks.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P]
    assert lib.gaac_encode_blocks(None, None, 0, 1024, 0, None, 1, 8, 1, None, None, None, None, None, None, None,
                                  None) == EINVAL
    lib.gaac_calibrate.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, P, P, P]
    assert lib.gaac_calibrate(None, 10, 1024, 8, None, None, None, None) == EINVAL


class _Pools(ctypes.Structure):
    _fields_ = [("slot_pool", ctypes.c_void_p), ("n_slots", ctypes.c_int64), ("raw_pool", ctypes.c_void_p),
                ("n_raw", ctypes.c_int64), ("raw_free", ctypes.c_void_p), ("n_raw_free", ctypes.c_int64),
                ("raw_cursor", ctypes.c_void_p)]


def test_misaligned_bases_rejected_on_host(lib):
    # The block encoder and the append read a K group's bases as words, so both
    # require 16-byte aligned base rows (gaac.h) and refuse others before any
    # launch; the pointers below are never dereferenced.
    P = ctypes.c_void_p
    EINVAL = 1
    good, odd = 0x10000, 0x10004
    pools = _Pools(good, 4, good, 4, None, 4, good)
    lib.gaac_encode_blocks.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P]
    lib.gaac_append.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, P]
    for b3, b4 in ((odd, good), (good, odd)):
        assert lib.gaac_encode_blocks(good, good, 1024, 1024, 64, good, 1, 8, 1, b3, b4, good, good,
                                      ctypes.byref(pools), None, good, None) == EINVAL
        assert lib.gaac_append(good, good, good, 1, 8, 1, b3, b4, good, good, ctypes.byref(pools), None, good,
                               None) == EINVAL
