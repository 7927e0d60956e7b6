"""ctypes binding of ``libmla_query.so`` (include/mla_query.h).

Argument marshalling only: torch tensors (or raw integer addresses) become the
plain pointers and sizes of the C ABI; every step of the decode runs in the
library's CUDA kernels.  There is no fallback: if the shared library is
missing, loading raises.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_query.so")

MLA_OK = 0
MLA_EINVAL = -1
MLA_ENOMEM = -2
MLA_ECUDA = -3
MLA_EUNSUPPORTED = -4
MLA_KV_FP8_E4M3 = 0
MLA_KV_FP8_DS_MLA = 1
MLA_KV_NVFP4_DS_MLA = 2
MLA_DEVERR_BAD_SLOT = 1
MLA_DEVERR_TIMEOUT = 2
MLA_DEVERR_CHECK = 4  # checks builds only: a bounds check failed (bit 8 + site names it)
MLA_PATH_AUTO = 0
MLA_PATH_FMA = 1
MLA_PATH_MMA = 2
MLA_MAX_BATCH = 256
MLA_MAX_HEADS = 128
MLA_NOALLOC_MAX_BATCH = 64
MLA_MAX_ROW_HEADS = 1024
MLA_ROWS_WAIT_MAX_NS = 2000000000

_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library once; raises if it has not been built.  The path
    defaults to the in-tree build; $MLA_QUERY_LIB selects another build of
    the same sources (for example an instrumented one)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = os.environ.get("MLA_QUERY_LIB", LIB_PATH)
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} not found: build it with `python -m mla_query_projection_gb300.build` "
            "(the MLA query path has no CPU fallback)"
        )
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.mla_query_create.argtypes = [ctypes.POINTER(vp), i32, vp, vp, vp, vp, f32]
    lib.mla_query_create.restype = i32
    lib.mla_query_decode.argtypes = [
        vp, i32, vp, i64, vp, i64, vp, i64, vp, vp, i64, i32, i32, vp, vp, vp, vp, vp,
    ]
    lib.mla_query_decode.restype = i32
    lib.mla_query_decode_fp8q.argtypes = [
        vp, i32, vp, i64, vp, i64, vp, i64, vp, vp, i64, i32, i32, vp, vp, vp, vp, vp, vp,
    ]
    lib.mla_query_decode_fp8q.restype = i32
    lib.mla_query_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint), vp]
    lib.mla_query_get_error.restype = i32
    lib.mla_query_set_path.argtypes = [vp, i32]
    lib.mla_query_set_path.restype = i32
    lib.mla_query_path_for.argtypes = [vp, i32]
    lib.mla_query_path_for.restype = i32
    lib.mla_query_decode_noalloc.argtypes = [
        i32, vp, vp, vp, vp, f32, i32, vp, i64, vp, i64, vp, i64, vp, vp, i64, i32, i32, vp, vp,
        vp, vp, vp, vp,
    ]
    lib.mla_query_decode_noalloc.restype = i32
    lib.mla_query_destroy.argtypes = [vp]
    lib.mla_query_destroy.restype = None
    lib.mla_query_kernel_for.argtypes = [vp, i32]
    lib.mla_query_kernel_for.restype = ctypes.c_char_p
    lib.mla_query_strerror.argtypes = [i32]
    lib.mla_query_strerror.restype = ctypes.c_char_p
    lib.mla_query_decode_rows.argtypes = [
        vp, i32, vp, i64, vp, i64, vp, i64, vp, vp, i64, i32, i32, vp, vp, vp, i32, i32, vp, vp,
    ]
    lib.mla_query_decode_rows.restype = i32
    lib.mla_query_rows_arm.argtypes = [vp, i32, i32, i32, vp]
    lib.mla_query_rows_arm.restype = i32
    lib.mla_query_rows_wait.argtypes = [vp, vp, i32, i32, i32, i32, i64, vp]
    lib.mla_query_rows_wait.restype = i32
    lib.mla_qkv_a_create.argtypes = [ctypes.POINTER(vp), i32, i32, vp]
    lib.mla_qkv_a_create.restype = i32
    lib.mla_qkv_a_run.argtypes = [vp, i32, vp, i64, vp, i64, vp]
    lib.mla_qkv_a_run.restype = i32
    lib.mla_qkv_a_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint), vp]
    lib.mla_qkv_a_get_error.restype = i32
    lib.mla_qkv_a_destroy.argtypes = [vp]
    lib.mla_qkv_a_destroy.restype = None
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    """A torch tensor's device address, an int address, or None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def strerror(code: int) -> str:
    return load().mla_query_strerror(code).decode()


def mla_query_create(num_heads, w_qb, w_uk, gamma_q, gamma_kv, eps) -> int:
    """Returns the handle (an opaque integer); raises MlaError on failure."""
    h = ctypes.c_void_p()
    rc = load().mla_query_create(
        ctypes.byref(h), int(num_heads), _ptr(w_qb), _ptr(w_uk), _ptr(gamma_q), _ptr(gamma_kv),
        float(eps),
    )
    if rc != MLA_OK:
        raise MlaError(rc, "mla_query_create")
    return h.value


def mla_query_decode(
    handle, batch, q_a, q_a_stride, kv_c, kv_c_stride, k_pe, k_pe_stride, slot_mapping,
    kv_cache, num_pages, page_size, layout, k_scale, q_latent, q_pe, q_c, stream,
) -> int:
    """Returns the C return code (MLA_OK on success)."""
    return load().mla_query_decode(
        handle, int(batch), _ptr(q_a), int(q_a_stride), _ptr(kv_c), int(kv_c_stride),
        _ptr(k_pe), int(k_pe_stride), _ptr(slot_mapping), _ptr(kv_cache), int(num_pages),
        int(page_size), int(layout), _ptr(k_scale), _ptr(q_latent), _ptr(q_pe), _ptr(q_c),
        _stream(stream),
    )


def mla_query_decode_fp8q(
    handle, batch, q_a, q_a_stride, kv_c, kv_c_stride, k_pe, k_pe_stride, slot_mapping,
    kv_cache, num_pages, page_size, layout, k_scale, q_scale_inv, q_latent_fp8, q_pe_fp8, q_c,
    stream,
) -> int:
    """The decode step with per-tensor FP8 query outputs; returns the C return code."""
    return load().mla_query_decode_fp8q(
        handle, int(batch), _ptr(q_a), int(q_a_stride), _ptr(kv_c), int(kv_c_stride),
        _ptr(k_pe), int(k_pe_stride), _ptr(slot_mapping), _ptr(kv_cache), int(num_pages),
        int(page_size), int(layout), _ptr(k_scale), _ptr(q_scale_inv), _ptr(q_latent_fp8),
        _ptr(q_pe_fp8), _ptr(q_c), _stream(stream),
    )


def mla_query_decode_noalloc(
    num_heads, w_qb, w_uk, gamma_q, gamma_kv, eps, batch, q_a, q_a_stride, kv_c, kv_c_stride,
    k_pe, k_pe_stride, slot_mapping, kv_cache, num_pages, page_size, layout, k_scale, q_latent,
    q_pe, q_c, device_flags, stream,
) -> int:
    """The handle-free decode for callers that must not allocate device
    memory; returns the C return code."""
    return load().mla_query_decode_noalloc(
        int(num_heads), _ptr(w_qb), _ptr(w_uk), _ptr(gamma_q), _ptr(gamma_kv), float(eps),
        int(batch), _ptr(q_a), int(q_a_stride), _ptr(kv_c), int(kv_c_stride), _ptr(k_pe),
        int(k_pe_stride), _ptr(slot_mapping), _ptr(kv_cache), int(num_pages), int(page_size),
        int(layout), _ptr(k_scale), _ptr(q_latent), _ptr(q_pe), _ptr(q_c), _ptr(device_flags),
        _stream(stream),
    )


def mla_query_get_error(handle, stream=None) -> int:
    v = ctypes.c_uint(0)
    rc = load().mla_query_get_error(handle, ctypes.byref(v), _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_query_get_error")
    return v.value


def mla_query_set_path(handle, path) -> int:
    return load().mla_query_set_path(handle, int(path))


def mla_query_path_for(handle, batch) -> int:
    return load().mla_query_path_for(handle, int(batch))


def mla_query_kernel_for(handle, batch) -> str | None:
    """Names of the kernels a decode of `batch` tokens launches ("a+b")."""
    r = load().mla_query_kernel_for(handle, int(batch))
    return r.decode() if r is not None else None


def mla_query_destroy(handle) -> None:
    load().mla_query_destroy(handle)


def mla_query_decode_rows(
    handle, batch, q_a, q_a_stride, kv_c, kv_c_stride, k_pe, k_pe_stride, slot_mapping,
    kv_cache, num_pages, page_size, layout, k_scale, q_scale_inv, q_rows, q_heads, head_offset,
    q_c, stream,
) -> int:
    return load().mla_query_decode_rows(
        handle, int(batch), _ptr(q_a), int(q_a_stride), _ptr(kv_c), int(kv_c_stride), _ptr(k_pe),
        int(k_pe_stride), _ptr(slot_mapping), _ptr(kv_cache), int(num_pages), int(page_size),
        int(layout), _ptr(k_scale), _ptr(q_scale_inv), _ptr(q_rows), int(q_heads),
        int(head_offset), _ptr(q_c), _stream(stream),
    )


def mla_query_rows_arm(q_rows, batch, q_heads, elem_bytes, stream) -> int:
    return load().mla_query_rows_arm(_ptr(q_rows), int(batch), int(q_heads), int(elem_bytes),
                                     _stream(stream))


def mla_query_rows_wait(handle, q_rows, batch, q_heads, wait_heads, elem_bytes, limit_ns,
                        stream) -> int:
    return load().mla_query_rows_wait(handle, _ptr(q_rows), int(batch), int(q_heads),
                                      int(wait_heads), int(elem_bytes), int(limit_ns),
                                      _stream(stream))


def mla_qkv_a_create(n, k, w) -> int:
    """Handle of the qkv_a down-projection y = x @ W^T (W [n][k] BF16 on the
    device, borrowed); raises MlaError on failure."""
    h = ctypes.c_void_p()
    rc = load().mla_qkv_a_create(ctypes.byref(h), int(n), int(k), _ptr(w))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_qkv_a_create")
    return h.value


def mla_qkv_a_run(handle, batch, x, x_stride, y, y_stride, stream) -> int:
    return load().mla_qkv_a_run(
        handle, int(batch), _ptr(x), int(x_stride), _ptr(y), int(y_stride), _stream(stream)
    )


def mla_qkv_a_get_error(handle, stream=None) -> int:
    v = ctypes.c_uint(0)
    rc = load().mla_qkv_a_get_error(handle, ctypes.byref(v), _stream(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_qkv_a_get_error")
    return v.value


def mla_qkv_a_destroy(handle) -> None:
    load().mla_qkv_a_destroy(handle)


def exported_symbols() -> list[str]:
    """Function names the public header declares."""
    import re

    hdr = os.path.join(os.path.dirname(HERE), "include", "mla_query.h")
    with open(hdr) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(mla_(?:query|qkv_a)_[a-z_0-9]+)\s*\(", text)))
