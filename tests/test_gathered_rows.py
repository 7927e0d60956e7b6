"""Gathered query rows (page "mla.query", class MlaQuery, methods publish and
gathered): decode context parallel ranks, simulated as decode calls on one
stream, write their heads' query rows [576] into head block rank * H of one
sentinel-armed [B][q_heads][576] buffer; a bounded poll then finds no
sentinel.  Each rank's rows must equal, bit for bit, the same kernels'
contiguous outputs, which are themselves checked against the oracle."""

import numpy as np
import pytest
import torch

from mla_query_projection_gb300 import binding as B
from mla_query_projection_gb300 import synthetic as S
from mla_query_projection_gb300.runner import DecodeStep
from oracle import mla_oracle as O

from .parity_util import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()
    torch.cuda.set_device(0)
    yield


def _ranks(inp, dcp):
    """Each rank's inputs: its H heads' slices of W_QB and W_UK, the rest shared."""
    H = inp["w_uk"].shape[0] // dcp
    return [dict(inp, w_qb=inp["w_qb"][r * H * 192:(r + 1) * H * 192],
                 w_uk=inp["w_uk"][r * H:(r + 1) * H]) for r in range(dcp)]


def _publish(st, rows, q_heads, offset, qsi, s):
    return B.mla_query_decode_rows(
        st.handle, st.batch, st.q_a, 0, st.kv_c, 0, st.k_pe, 0, st.slots, st.cache, st.num_pages,
        st.page_size, st.layout, st.k_scale, qsi, rows, q_heads, offset, st.q_c, s)


@pytest.mark.parametrize(
    "batch,heads,fp8,layout,path",
    [
        (1, 64, False, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),        # paired kernel
        (8, 32, True, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),         # paired kernel, E4M3 rows
        (16, 64, False, S.LAYOUT_DS_MLA, B.MLA_PATH_AUTO),     # 16-token paired kernel
        (40, 32, True, S.LAYOUT_NVFP4_DS_MLA, B.MLA_PATH_AUTO),  # wide kernel
        (70, 16, False, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),       # wide kernel, two slices
        (4, 8, False, S.LAYOUT_E4M3, B.MLA_PATH_AUTO),         # partials + closing kernel
        (2, 16, True, S.LAYOUT_E4M3, B.MLA_PATH_FMA),          # FMA kernel + closing kernel
    ],
)
def test_ranks_gather_their_rows(batch, heads, fp8, layout, path):
    dcp, pad = 2, 3
    q_heads = dcp * heads + pad
    E = 1 if fp8 else 2
    inp = S.make_inputs(batch=batch, heads=dcp * heads, layout=layout, pages=64,
                        seed=2500 + batch + heads)
    dev, s = torch.device("cuda", 0), torch.cuda.current_stream()
    rows = torch.empty(batch * q_heads * 576 * E, dtype=torch.uint8, device=dev)
    assert B.mla_query_rows_arm(rows, batch, q_heads, E, s) == B.MLA_OK
    steps = [DecodeStep(r_inp) for r_inp in _ranks(inp, dcp)]
    for st in steps:
        assert st.set_path(path) == B.MLA_OK
    qsi = torch.tensor([3.0], dtype=torch.float32, device=dev) if fp8 else None
    for r, st in enumerate(steps):
        assert _publish(st, rows, q_heads, r * heads, qsi, s) == B.MLA_OK
    assert B.mla_query_rows_wait(steps[0].handle, rows, batch, q_heads, dcp * heads, E,
                                 100_000_000, s) == 0
    torch.cuda.synchronize()
    assert steps[0].error_flags() == 0
    got = rows.cpu().numpy().reshape(batch, q_heads, 576 * E)
    assert np.all(got[:, dcp * heads:, :] == 0xFF), "padding heads were written"
    if not fp8:
        got = got.view(np.uint16).reshape(batch, q_heads, 576)
    for r, (st, r_inp) in enumerate(zip(steps, _ranks(inp, dcp))):
        assert st.decode() == B.MLA_OK  # the same kernels, contiguous BF16 outputs
        out = st.results()
        check_against_oracle(out, r_inp)
        want_l, want_p = out["q_latent"], out["q_pe"]
        if fp8:
            want_l, want_p = O.query_fp8(want_l, 3.0), O.query_fp8(want_p, 3.0)
        block = got[:, r * heads:(r + 1) * heads, :]
        np.testing.assert_array_equal(block[:, :, :512], want_l)
        np.testing.assert_array_equal(block[:, :, 512:], want_p)
        st.close()


def test_wait_reports_a_missing_rank_and_the_context_survives():
    """Only rank 0 publishes: the poll runs out after its 2 ms limit and sets
    MLA_DEVERR_TIMEOUT.  Rank 1 then publishes and a second wait passes."""
    heads, batch, dcp = 8, 3, 2
    inp = S.make_inputs(batch=batch, heads=dcp * heads, layout=S.LAYOUT_E4M3, pages=16,
                        seed=2600)
    dev, s = torch.device("cuda", 0), torch.cuda.current_stream()
    rows = torch.empty(batch * dcp * heads * 576 * 2, dtype=torch.uint8, device=dev)
    assert B.mla_query_rows_arm(rows, batch, dcp * heads, 2, s) == B.MLA_OK
    steps = [DecodeStep(r_inp) for r_inp in _ranks(inp, dcp)]
    assert _publish(steps[0], rows, dcp * heads, 0, None, s) == B.MLA_OK
    assert B.mla_query_rows_wait(steps[0].handle, rows, batch, dcp * heads, dcp * heads, 2,
                                 2_000_000, s) == 0
    torch.cuda.synchronize()
    assert steps[0].error_flags() == B.MLA_DEVERR_TIMEOUT
    assert _publish(steps[1], rows, dcp * heads, heads, None, s) == B.MLA_OK
    assert B.mla_query_rows_wait(steps[0].handle, rows, batch, dcp * heads, dcp * heads, 2,
                                 100_000_000, s) == 0
    torch.cuda.synchronize()
    assert steps[0].error_flags() == 0
    for st in steps:
        st.close()


def test_rows_argument_errors():
    inp = S.make_inputs(batch=2, heads=8, layout=S.LAYOUT_E4M3, pages=4, seed=2700)
    st = DecodeStep(inp)
    dev, s = torch.device("cuda", 0), torch.cuda.current_stream()
    rows = torch.empty(2 * 16 * 576 * 2, dtype=torch.uint8, device=dev)
    assert _publish(st, rows, 16, 9, None, s) == B.MLA_EINVAL  # 9 + 8 heads > 16
    assert _publish(st, rows, 16, -1, None, s) == B.MLA_EINVAL
    assert _publish(st, rows, B.MLA_MAX_ROW_HEADS + 1, 0, None, s) == B.MLA_EINVAL
    assert _publish(st, rows, 16, 8, None, s) == B.MLA_OK
    too_long = B.MLA_ROWS_WAIT_MAX_NS + 1
    assert B.mla_query_rows_wait(st.handle, rows, 2, 16, 16, 2, too_long, s) == B.MLA_EINVAL
    assert B.mla_query_rows_wait(st.handle, rows, 2, 16, 16, 2, -1, s) == B.MLA_EINVAL
    assert B.mla_query_rows_wait(st.handle, rows, 2, 16, 17, 2, 1000, s) == B.MLA_EINVAL
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    st.close()
