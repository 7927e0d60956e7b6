"""Per-tensor FP8 query outputs (mla_query_decode_fp8q), on every path.

The FP8 variant runs the same kernels with a different epilogue (page
"mla.query", method kernel: q_latent and q_pe stored as E4M3 codes of
bf16(v) * q_scale_inv).  So its codes must equal, bit for bit, the oracle's
FP8 conversion (query_fp8) applied to the same kernels' BF16 outputs, which are
themselves checked against the oracle here; and they must meet the FP8 bar
against the oracle's own FP8 outputs (at least 99.9% of codes identical, the
rest within one code of the codes the oracle allows: its own, or for q_latent
elements fed by a nope Q_B value of ambiguous rounding, the codes of that
rounding's range).
"""

import numpy as np
import pytest
import torch

from mla_query_projection_gb300 import binding as B
from mla_query_projection_gb300 import synthetic as S
from mla_query_projection_gb300.runner import DecodeStep
from oracle import mla_oracle as O

from .parity_util import check_against_oracle, check_fp8_query, latent_slack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()
    torch.cuda.set_device(0)
    yield


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize(
    "batch,heads,layout,path",
    [
        (1, 64, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),    # paired kernel, 8 tokens
        (16, 128, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),  # paired kernel, 16 tokens
        (48, 64, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),   # wide tcgen05 kernel
        (70, 16, S.LAYOUT_DS_MLA, B.MLA_PATH_AUTO), # wide kernel, two 64-token slices
        (4, 16, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),    # partials + closing kernel (small H)
        (2, 32, S.LAYOUT_E4M3, B.MLA_PATH_FMA),     # FP32-FMA absorbing kernel
        (8, 64, S.LAYOUT_NVFP4_DS_MLA, B.MLA_PATH_AUTO),   # FP8 query + nvfp4_ds_mla rows
        (40, 32, S.LAYOUT_NVFP4_DS_MLA, B.MLA_PATH_AUTO),  # the same on the wide kernel
    ],
)
def test_fp8_query_codes_follow_the_bf16_outputs(batch, heads, layout, path):
    inp = S.make_inputs(batch=batch, heads=heads, layout=layout, pages=64, seed=1500 + batch)
    st = DecodeStep(inp)
    assert st.set_path(path) == B.MLA_OK
    cache0 = st.cache.clone()
    # BF16 run, checked against the oracle
    assert st.decode() == B.MLA_OK
    bf = st.results()
    ref = check_against_oracle(bf, inp)
    # FP8 run on the same inputs and a fresh copy of the cache
    dev = st.q_a.device
    qsi = torch.tensor([3.0], dtype=torch.float32, device=dev)
    ql8 = torch.full((batch, heads, 512), 0x7F, dtype=torch.uint8, device=dev)
    qp8 = torch.full((batch, heads, 64), 0x7F, dtype=torch.uint8, device=dev)
    qc = torch.full_like(st.q_c, float("nan"))
    cache = cache0.clone()
    rc = B.mla_query_decode_fp8q(
        st.handle, batch, st.q_a, st.strides[0], st.kv_c, st.strides[1], st.k_pe,
        st.strides[2], st.slots, cache, st.num_pages, st.page_size, st.layout, st.k_scale, qsi,
        ql8, qp8, qc, torch.cuda.current_stream())
    assert rc == B.MLA_OK
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    np.testing.assert_array_equal(ql8.cpu().numpy(), O.query_fp8(bf["q_latent"], 3.0))
    np.testing.assert_array_equal(qp8.cpu().numpy(), O.query_fp8(bf["q_pe"], 3.0))
    # directly against the oracle's FP8 outputs (the oracle's step for the
    # q_c rounding the GPU took, with q_scale_inv = 3)
    rep = {}
    check_fp8_query("q_latent_fp8", ql8.cpu().numpy(), ref["q_latent"], 3.0, rep,
                    slack=latent_slack(ref, inp))
    check_fp8_query("q_pe_fp8", qp8.cpu().numpy(), ref["q_pe"], 3.0, rep)
    print(batch, heads, rep)
    np.testing.assert_array_equal(_bits(qc), bf["q_c"])
    np.testing.assert_array_equal(cache.cpu().numpy(), bf["cache"])
    st.close()


def test_fp8_query_requires_a_scale():
    inp = S.make_inputs(batch=1, heads=4, layout=S.LAYOUT_E4M3, pages=4, seed=1600)
    st = DecodeStep(inp)
    rc = B.mla_query_decode_fp8q(
        st.handle, 1, st.q_a, 0, st.kv_c, 0, st.k_pe, 0, st.slots, st.cache, st.num_pages,
        st.page_size, st.layout, st.k_scale, None, st.q_latent, st.q_pe, st.q_c,
        torch.cuda.current_stream())
    assert rc == B.MLA_EINVAL
    st.close()
