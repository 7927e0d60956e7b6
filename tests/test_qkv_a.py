"""GPU parity of the qkv_a down-projection (the step that makes the fused
q_a | kv_c | k_pe row; pages "ws_gemm", class WsGemm, and "mla.query",
method kernel) against the FP64 oracle, and of the chained step: the
projection, then the decode step reading its output row."""

import numpy as np
import pytest
import torch

from mla_query_projection_gb300 import binding as B
from mla_query_projection_gb300 import synthetic as S
from mla_query_projection_gb300.runner import DecodeStep, bf16_bits, bf16_tensor
from oracle import mla_oracle as O

from .parity_util import check_against_oracle, check_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()
    torch.cuda.set_device(0)
    yield


def _draw(batch, n, k, seed):
    rng = np.random.default_rng(seed)
    w = S.qkv_a_weights(rng, n=n, k=k)["w_qkv_a"]
    x = S.hidden_rows(batch, rng, k=k)
    return w, x


def _run(w, x, x_pad=0, y_pad=0, repeat=1):
    dev = torch.device("cuda", 0)
    (n, k), batch = w.shape, x.shape[0]
    wd = bf16_tensor(w, dev)
    xs = np.zeros((batch, k + x_pad), dtype=np.uint16)
    xs[:, :k] = x
    xd = bf16_tensor(xs, dev)
    h = B.mla_qkv_a_create(n, k, wd)
    outs = []
    for _ in range(repeat):
        yd = torch.full((batch, n + y_pad), float("nan"), dtype=torch.bfloat16, device=dev)
        rc = B.mla_qkv_a_run(h, batch, xd, k + x_pad, yd, n + y_pad, torch.cuda.current_stream())
        assert rc == B.MLA_OK
        torch.cuda.synchronize()
        outs.append(bf16_bits(yd))
    assert B.mla_qkv_a_get_error(h, torch.cuda.current_stream()) == 0
    B.mla_qkv_a_destroy(h)
    return outs


def _check(y, w, x, report=None):
    ref, exact, cond = O.qkv_a_projection(x, w)
    check_bf16("y", y, ref, cond, report=report)


@pytest.mark.parametrize(
    "batch,n,k",
    [
        (1, 2112, 7168),   # the fused row of one token: 14 rows per CTA
        (8, 2112, 7168),   # one full 8-token launch
        (3, 2112, 7168),   # a partial n8 tile
        (9, 2112, 7168),   # two launches, the second with one token
        (33, 2112, 7168),  # five launches
        (2, 2280, 7168),   # 15 rows per CTA: the largest share
        (5, 16, 512),      # one row per CTA, the smallest K
        (4, 100, 1536),    # a ragged last CTA
        (7, 300, 4096),
    ],
)
def test_qkv_a_matches_oracle(batch, n, k):
    w, x = _draw(batch, n, k, seed=2000 + batch + n)
    (y,) = _run(w, x)
    rep = {}
    _check(y, w, x, report=rep)
    print(batch, n, k, rep)


def test_qkv_a_strides_and_untouched_padding():
    """Row strides above the widths: x's padding is not read (it holds NaN
    patterns), y's padding is not written."""
    w, x = _draw(6, 2112, 7168, seed=2100)
    dev = torch.device("cuda", 0)
    xs = np.full((6, 7168 + 64), 0x7FC0, dtype=np.uint16)
    xs[:, :7168] = x
    yd = torch.full((6, 2112 + 24), 3.0, dtype=torch.bfloat16, device=dev)
    h = B.mla_qkv_a_create(2112, 7168, bf16_tensor(w, dev))
    xd = bf16_tensor(xs, dev)
    assert B.mla_qkv_a_run(h, 6, xd, 7168 + 64, yd, 2112 + 24, torch.cuda.current_stream()) == 0
    torch.cuda.synchronize()
    y = bf16_bits(yd)
    _check(y[:, :2112], w, x)
    assert np.all(y[:, 2112:] == bf16_bits(torch.tensor([3.0], dtype=torch.bfloat16))[0])
    B.mla_qkv_a_destroy(h)


def test_qkv_a_deterministic():
    w, x = _draw(5, 2112, 7168, seed=2200)
    a, b = _run(w, x, repeat=2)
    assert np.array_equal(a, b)


def test_qkv_a_argument_errors_on_device_buffers():
    dev = torch.device("cuda", 0)
    w = torch.zeros((2112, 7168), dtype=torch.bfloat16, device=dev)
    x = torch.zeros((2, 7168), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((2, 2112), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.current_stream()
    h = B.mla_qkv_a_create(2112, 7168, w)
    assert B.mla_qkv_a_run(h, 0, x, 0, y, 0, s) == B.MLA_EINVAL
    assert B.mla_qkv_a_run(h, B.MLA_MAX_BATCH + 1, x, 0, y, 0, s) == B.MLA_EINVAL
    assert B.mla_qkv_a_run(h, 2, x.data_ptr() + 2, 0, y, 0, s) == B.MLA_EINVAL  # misaligned x
    assert B.mla_qkv_a_run(h, 2, x, 7160, y, 0, s) == B.MLA_EINVAL  # x stride below k
    assert B.mla_qkv_a_run(h, 2, x, 7172, y, 0, s) == B.MLA_EINVAL  # x stride not a multiple of 8
    assert B.mla_qkv_a_run(h, 2, x, 0, y, 2000, s) == B.MLA_EINVAL  # y stride below n
    assert B.mla_qkv_a_run(h, 2, x, 0, y, 0, s) == B.MLA_OK
    torch.cuda.synchronize()
    assert B.mla_qkv_a_get_error(h, s) == 0
    B.mla_qkv_a_destroy(h)
    with pytest.raises(B.MlaError):
        B.mla_qkv_a_create(2432, 7168, w)  # 16 rows per CTA: beyond the limit


@pytest.mark.parametrize("batch,heads,layout", [(1, 64, S.LAYOUT_E4M3), (12, 32, S.LAYOUT_DS_MLA),
                                                (40, 16, S.LAYOUT_NVFP4_DS_MLA)])
def test_hidden_row_then_decode_step(batch, heads, layout):
    """The chained step on one stream: the projection writes the fused row,
    the decode step reads it (its weight streaming overlaps the projection's
    tail).  The row is held to the oracle's projection; the decode outputs to
    the oracle's step on that row."""
    inp = S.make_inputs(batch=batch, heads=heads, layout=layout, pages=64, seed=2300 + batch,
                        hidden=True)
    st = DecodeStep(inp, hidden=True)
    assert st.decode() == B.MLA_OK
    out = st.results()
    assert st.error_flags() == 0
    assert B.mla_qkv_a_get_error(st.qkv_a, torch.cuda.current_stream()) == 0
    _check(out["qkv_row"], inp["w_qkv_a"], inp["hidden"])
    row = out["qkv_row"]
    step_inp = dict(inp, q_a=row[:, :1536], kv_c=row[:, 1536:2048], k_pe=row[:, 2048:])
    check_against_oracle(out, step_inp)
    st.close()
