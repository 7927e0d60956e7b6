"""The C-ABI library: builds for sm_103a, loads without a GPU, exports every
function the public header declares, and rejects bad arguments on the host
before touching the device.  CPU only: no compute call is made."""

import ctypes
import os

import pytest

from mla_query_projection_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from mla_query_projection_gb300 import build

        build.build()
    return B.load()


def test_exports_every_declared_symbol(lib):
    names = B.exported_symbols()
    assert {"mla_query_create", "mla_query_decode", "mla_query_destroy"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/mla_query.h but not exported"


def test_binding_constants_match_the_header():
    """Every numeric #define of include/mla_query.h has the same value in the
    binding (layouts, paths, error codes, device flags, limits)."""
    import re

    hdr = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla_query.h")
    with open(hdr) as f:
        text = f.read()
    found = re.findall(r"#define\s+(MLA_[A-Z0-9_]+)\s+\(?(-?\d+)u?\)?", text)
    assert len(found) >= 15
    for name, value in found:
        assert getattr(B, name) == int(value), name
    assert B.MLA_KV_NVFP4_DS_MLA == 2


def test_no_unexported_internal_symbols(lib):
    # internal kernels and helpers stay hidden (only the C ABI is public)
    with pytest.raises(AttributeError):
        lib.launch_fused  # noqa: B018


def test_strerror(lib):
    assert B.strerror(B.MLA_OK) == "ok"
    assert "invalid" in B.strerror(B.MLA_EINVAL)
    assert B.strerror(12345) == "unknown error"


def test_create_rejects_bad_arguments_on_host(lib):
    h = ctypes.c_void_p()
    assert lib.mla_query_create(None, 16, 16, 16, 16, 16, 1e-6) == B.MLA_EINVAL
    # heads out of range
    assert lib.mla_query_create(ctypes.byref(h), 0, 16, 16, 16, 16, 1e-6) == B.MLA_EINVAL
    assert lib.mla_query_create(ctypes.byref(h), 129, 16, 16, 16, 16, 1e-6) == B.MLA_EINVAL
    # null weight
    assert lib.mla_query_create(ctypes.byref(h), 16, None, 16, 16, 16, 1e-6) == B.MLA_EINVAL
    # misaligned weight
    assert lib.mla_query_create(ctypes.byref(h), 16, 24, 16, 16, 16, 1e-6) == B.MLA_EINVAL
    # negative eps
    assert lib.mla_query_create(ctypes.byref(h), 16, 16, 16, 16, 16, -1.0) == B.MLA_EINVAL
    assert h.value is None


def test_decode_rejects_null_handle(lib):
    rc = B.mla_query_decode(None, 1, 16, 0, 16, 0, 16, 0, 16, 16, 8, 64, 0, 16, 16, 16, None, None)
    assert rc == B.MLA_EINVAL


def test_other_entry_points_reject_null_handle(lib):
    assert B.mla_query_set_path(None, B.MLA_PATH_FMA) == B.MLA_EINVAL
    assert B.mla_query_path_for(None, 1) == B.MLA_EINVAL
    with pytest.raises(B.MlaError):
        B.mla_query_get_error(None)
    B.mla_query_destroy(None)  # no-op


def test_qkv_a_rejects_bad_arguments_on_host(lib):
    """The down-projection's host checks run before any device call."""
    h = ctypes.c_void_p()
    assert lib.mla_qkv_a_create(None, 2112, 7168, 16) == B.MLA_EINVAL
    assert lib.mla_qkv_a_create(ctypes.byref(h), 2112, 7168, None) == B.MLA_EINVAL
    assert lib.mla_qkv_a_create(ctypes.byref(h), 2112, 7168, 24) == B.MLA_EINVAL  # misaligned
    assert lib.mla_qkv_a_create(ctypes.byref(h), 0, 7168, 16) == B.MLA_EINVAL
    assert lib.mla_qkv_a_create(ctypes.byref(h), 2112, 7000, 16) == B.MLA_EINVAL  # k % 512
    assert lib.mla_qkv_a_create(ctypes.byref(h), 2112, 256, 16) == B.MLA_EINVAL  # k < 512
    assert lib.mla_qkv_a_create(ctypes.byref(h), 2112, 8192, 16) == B.MLA_EUNSUPPORTED
    assert h.value is None
    assert lib.mla_qkv_a_run(None, 1, 16, 0, 16, 0, None) == B.MLA_EINVAL
    lib.mla_qkv_a_destroy(None)


def test_gathered_rows_reject_bad_arguments_on_host(lib):
    """Host checks of the gathered-row entry points, before any device call."""
    # null handle / buffer
    assert B.mla_query_rows_wait(None, 16, 1, 64, 64, 1, 1000, None) == B.MLA_EINVAL
    assert B.mla_query_rows_arm(None, 1, 64, 1, None) == B.MLA_EINVAL
    assert B.mla_query_rows_arm(16, 0, 64, 1, None) == B.MLA_EINVAL  # batch
    assert B.mla_query_rows_arm(16, 1, 0, 1, None) == B.MLA_EINVAL  # q_heads
    assert B.mla_query_rows_arm(16, 1, B.MLA_MAX_ROW_HEADS + 1, 1, None) == B.MLA_EINVAL
    assert B.mla_query_rows_arm(16, 1, 64, 4, None) == B.MLA_EINVAL  # element size
    assert B.mla_query_rows_arm(24, 1, 64, 1, None) == B.MLA_EINVAL  # misaligned
    assert B.mla_query_decode_rows(None, 1, 16, 0, 16, 0, 16, 0, 16, 16, 1, 64, 0, 16, None, 16,
                                   64, 0, None, None) == B.MLA_EINVAL


def test_kernel_for_rejects_a_null_handle(lib):
    assert B.mla_query_kernel_for(None, 1) is None
