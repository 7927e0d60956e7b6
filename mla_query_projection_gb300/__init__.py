"""GB300-native decode-step MLA query path.

``binding`` holds the ctypes binding of ``libmla_query.so`` (the C ABI in
``include/mla_query.h``); ``runner`` wraps it for torch tensors;
``synthetic`` draws the seeded workloads.  Importing the package does not load
the library; the first binding call does, and fails loudly if it is missing.
"""

from .binding import (  # noqa: F401
    MLA_DEVERR_BAD_SLOT,
    MLA_DEVERR_TIMEOUT,
    MLA_KV_FP8_DS_MLA,
    MLA_KV_FP8_E4M3,
    MLA_KV_NVFP4_DS_MLA,
    MLA_OK,
    MLA_PATH_AUTO,
    MLA_PATH_FMA,
    MLA_PATH_MMA,
    MlaError,
    mla_query_create,
    mla_query_decode,
    mla_query_decode_fp8q,
    mla_query_decode_rows,
    mla_query_rows_arm,
    mla_query_rows_wait,
    mla_query_destroy,
    mla_query_get_error,
    mla_query_kernel_for,
    mla_query_path_for,
    mla_query_set_path,
    mla_qkv_a_create,
    mla_qkv_a_destroy,
    mla_qkv_a_get_error,
    mla_qkv_a_run,
)
