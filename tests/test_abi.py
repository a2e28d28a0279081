"""Host-side checks of the C ABI: the library loads without a GPU and exports every symbol
that include/fmpq.h declares, and the binding's signature table names exactly those."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "fmpq.h")).read()
    return sorted(set(re.findall(r"^FMPQ_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.MULTILINE)))


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_gemm_fmpq_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_boundary():
    names = _declared()
    for fn in ("fmpq_layout_create", "fmpq_quantize", "w4_pack_weights", "w4ax_gemm", "w4ax_gemm_partials",
               "w4_unpack_weights", "fmpq_device_status"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_signatures_match_header():
    from bit_quantized_gemm_fmpq_gb300 import fmpq
    assert sorted(fmpq.SIGNATURES) == _declared()


def test_host_only_calls(lib):
    lib.fmpq_status_string.restype = ctypes.c_char_p
    assert lib.fmpq_status_string(0) == b"ok"
    assert lib.fmpq_status_string(7) == b"workspace missing or too small"
    assert lib.fmpq_version() == 100
    lib.fmpq_packed_a_bytes.restype = ctypes.c_size_t
    assert lib.fmpq_packed_a_bytes(None, ctypes.c_int64(5)) == 0


def test_invalid_layout_arguments_fail_before_touching_a_device(lib):
    out = ctypes.c_void_p()
    perm = (ctypes.c_int32 * 256)(*range(256))
    mask = (ctypes.c_uint8 * 2)(0, 0)
    assert lib.fmpq_layout_create(100, perm, mask, ctypes.byref(out)) == 2       # K % 128
    bad = (ctypes.c_int32 * 256)(*([0] * 256))
    assert lib.fmpq_layout_create(256, bad, mask, ctypes.byref(out)) == 1        # not a permutation
    badmask = (ctypes.c_uint8 * 2)(0, 3)
    assert lib.fmpq_layout_create(256, perm, badmask, ctypes.byref(out)) == 1    # mask value
    assert lib.fmpq_layout_create(256, None, mask, ctypes.byref(out)) == 1


def test_entry_points_refuse_null_arguments_without_a_device(lib):
    """Every compute entry point checks its pointers before any device call (status 1 =
    FMPQ_ERR_INVALID_ARG), so a caller's mistake is reported synchronously."""
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    z = P(None)
    calls = {
        "fmpq_quantize": (z, z, i64(8), i64(1), z, z, z),
        "fmpq_quantize_asym": (z, z, i64(8), i64(1), z, z, z, z),
        "qoq_quantize": (z, z, i64(8), i64(1), z, z, z, z),
        "w4_pack_weights": (z, z, i64(8), i64(16), z, z, z),
        "qoq_pack_weights": (z, z, i64(8), i64(16), z, z, z, z, z),
        "w4_weight_sums": (z, z, z, i64(16), z, z),
        "w4ax_gemm": (z, z, z, z, z, i64(1), i64(16), z, i64(16), z, ctypes.c_size_t(0), z),
        "w4ax_gemm_asym": (z, z, z, z, z, z, z, i64(1), i64(16), z, i64(16), z, ctypes.c_size_t(0), z),
        "qoq_gemm": (z, z, z, z, z, z, z, z, i64(1), i64(16), z, i64(16), z, ctypes.c_size_t(0), z),
    }
    for name, args in calls.items():
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        assert fn(*args) == 1, name
