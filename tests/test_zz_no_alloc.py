"""The allocation-free entry point, mla_query_decode_noalloc.

Some callers may not allocate device memory at all: a serving runtime that
hands every byte of the GPU to its own pool at start-up, or a plugin inside a
framework whose allocator owns the device.  For them the library offers a
decode that keeps its scratch in one fixed array inside the library.  This
test calls it through the C ABI and checks that, on two calls in a row, its
results pass the parity checks against the oracle and are bit-identical to
each other.  The file name makes pytest collect it last.
"""

import numpy as np
import pytest
import torch

from mla_query_projection_gb300 import binding as B
from mla_query_projection_gb300 import synthetic as S
from mla_query_projection_gb300.runner import DecodeStep

from .parity_util import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()
    torch.cuda.set_device(0)
    yield


def _noalloc_call(st: DecodeStep, flags: torch.Tensor, q_latent, q_pe, q_c, cache):
    return B.mla_query_decode_noalloc(
        st.heads, st.w_qb, st.w_uk, st.gamma_q, st.gamma_kv, st.eps, st.batch,
        st.q_a, st.strides[0], st.kv_c, st.strides[1], st.k_pe, st.strides[2], st.slots,
        cache, st.num_pages, st.page_size, st.layout, st.k_scale, q_latent, q_pe, q_c, flags,
        torch.cuda.current_stream(),
    )


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize(
    "batch,heads,layout",
    [(1, 64, S.LAYOUT_E4M3), (2, 128, S.LAYOUT_E4M3), (8, 128, S.LAYOUT_E4M3),
     (33, 32, S.LAYOUT_DS_MLA), (5, 16, S.LAYOUT_NVFP4_DS_MLA),
     (64, 128, S.LAYOUT_DS_MLA)],
)
def test_noalloc_matches_oracle_twice(batch, heads, layout):
    """Batch 2 takes the FP32-FMA flavour of the hand-off kernel (its only
    caller); batch 64 at 128 heads fills the fixed array exactly (four groups
    of 16 tokens: every counter and every hand-off row)."""
    inp = S.make_inputs(batch=batch, heads=heads, layout=layout, pages=64, seed=1200 + batch)
    st = DecodeStep(inp)
    cache0 = st.cache.clone()
    dev = st.q_a.device
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    runs = []
    for _ in range(2):  # two calls in a row: the shared array must re-arm
        q_latent = torch.full_like(st.q_latent, float("nan"))
        q_pe = torch.full_like(st.q_pe, float("nan"))
        q_c = torch.full_like(st.q_c, float("nan"))
        cache = cache0.clone()
        assert _noalloc_call(st, flags, q_latent, q_pe, q_c, cache) == B.MLA_OK
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        gpu = {"q_latent": _bits(q_latent), "q_pe": _bits(q_pe), "q_c": _bits(q_c),
               "cache": cache.cpu().numpy()}
        check_against_oracle(gpu, inp)
        runs.append(gpu)
    for k in runs[0]:  # the same kernel on the same inputs: bit-identical
        assert np.array_equal(runs[0][k], runs[1][k]), k
    st.close()


def test_noalloc_rejects_batches_beyond_its_array():
    inp = S.make_inputs(batch=B.MLA_NOALLOC_MAX_BATCH + 1, heads=4, layout=S.LAYOUT_E4M3,
                        pages=8, seed=1300)
    st = DecodeStep(inp)
    flags = torch.zeros(1, dtype=torch.int32, device=st.q_a.device)
    rc = _noalloc_call(st, flags, st.q_latent, st.q_pe, st.q_c, st.cache)
    assert rc == B.MLA_EUNSUPPORTED
    st.close()
