"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle, on
the same seeded inputs, element by element.  Every test needs a GB300."""

import os

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


def run_case(inp, path=B.MLA_PATH_AUTO, fused_row=False, q_c=True, repeat=1):
    step = DecodeStep(inp, fused_row=fused_row, q_c=q_c)
    assert step.set_path(path) == B.MLA_OK
    for _ in range(repeat):
        assert step.decode() == B.MLA_OK
    out = step.results()
    flags = step.error_flags()
    step.close()
    return out, flags


def assert_parity(inp, report=None, **kw):
    out, flags = run_case(inp, **kw)
    name = os.environ.get("PYTEST_CURRENT_TEST", "case").split(" ")[0].split("::")[-1]
    ref = check_against_oracle(out, inp, report=report, q_c=kw.get("q_c", True), dump_name=name)
    want_flag = B.MLA_DEVERR_BAD_SLOT if ref["bad_slots"] else 0
    assert flags == want_flag, f"device flags {flags}"
    return out, ref


@pytest.mark.parametrize("name", list(S.WORKLOADS))
def test_named_workloads(name):
    inp = S.workload_inputs(name)
    rep = {}
    assert_parity(inp, report=rep)
    print(name, rep)


@pytest.mark.parametrize("layout", [S.LAYOUT_E4M3, S.LAYOUT_DS_MLA])
@pytest.mark.parametrize("heads", [64, 128])
@pytest.mark.parametrize("batch", [1, 2, 4, 8, 16, 32, 64])
def test_sweep(batch, heads, layout):
    inp = S.make_inputs(**S.sweep_workload(batch, heads, layout))
    assert_parity(inp)


@pytest.mark.parametrize("heads", [64, 128])
@pytest.mark.parametrize("batch", [1, 2, 8, 16, 17, 64, 70])
def test_nvfp4_ds_mla_rows(batch, heads):
    """The nvfp4_ds_mla cache layout on every kernel the batch selects
    (paired 8 and 16 tokens, wide, wide in two slices), 1% kv_c outliers."""
    inp = S.make_inputs(**S.sweep_workload(batch, heads, S.LAYOUT_NVFP4_DS_MLA))
    rep = {}
    assert_parity(inp, report=rep)
    print(batch, heads, rep)


@pytest.mark.parametrize("path", [B.MLA_PATH_FMA, B.MLA_PATH_MMA])
def test_nvfp4_zero_rows_and_bad_slots(path):
    """kv_c rows of zeros normalise to zeros: every block takes the scale floor
    2**-9 (E4M3 0x01) and code 0; a skipped and an out-of-range slot leave
    their rows alone."""
    inp = S.make_inputs(batch=2, heads=16, layout=S.LAYOUT_NVFP4_DS_MLA, pages=4, seed=650)
    inp["kv_c"][0, :] = 0
    out, ref = assert_parity(inp, path=path)
    s = int(inp["slots"][0])
    row = out["cache"][s // 64, s % 64]
    assert np.all(row[:256] == 0) and np.all(row[256:288] == 0x01)
    inp = S.make_inputs(batch=4, heads=8, layout=S.LAYOUT_NVFP4_DS_MLA, pages=4, seed=651)
    inp["slots"] = np.array([-1, 7, 4 * 64, 200], dtype=np.int64)
    out, ref = assert_parity(inp)
    assert ref["bad_slots"] == [2]


@pytest.mark.parametrize("batch", [3, 5, 7, 9, 15, 17, 31, 33, 63, 65, 100, 200, 256])
def test_ragged_batches(batch):
    layout = S.LAYOUT_DS_MLA if batch % 2 else S.LAYOUT_E4M3
    inp = S.make_inputs(batch=batch, heads=16, layout=layout, pages=64, seed=100 + batch,
                        outliers=0.01)
    assert_parity(inp)


def test_empty_and_oversize_batches_write_nothing():
    """An empty step (B = 0), a negative batch and one above MLA_MAX_BATCH
    are host errors: the call returns MLA_EINVAL, launches nothing and leaves
    every output and cache byte as it was; a valid call afterwards meets the
    oracle."""
    inp = S.make_inputs(batch=3, heads=4, layout=S.LAYOUT_E4M3, pages=4, seed=661)
    step = DecodeStep(inp)
    before = step.results()
    for b in (0, -3, B.MLA_MAX_BATCH + 1):
        assert step.decode(batch=b) == B.MLA_EINVAL, b
    after = step.results()
    for k in before:
        assert np.array_equal(before[k], after[k]), k
    assert step.error_flags() == 0
    step.close()
    assert_parity(inp)


@pytest.mark.parametrize("heads", [1, 2, 3, 5, 127, 128])
@pytest.mark.parametrize("batch", [1, 2, 16])
def test_head_counts(heads, batch):
    inp = S.make_inputs(batch=batch, heads=heads, layout=S.LAYOUT_E4M3, pages=16, seed=200 + heads)
    assert_parity(inp)


@pytest.mark.parametrize("batch,heads", [(1, 40), (1, 96), (2, 96), (4, 40), (8, 80), (16, 96),
                                         (16, 40), (8, 16)])
def test_paired_kernel_unbalanced_head_counts(batch, heads):
    """Head counts where whole half-heads leave the paired kernel's CTAs
    unbalanced (some pairs two heads, or none) still take it: it meets the
    oracle there, with the heads on the first pairs (up to 8 tokens, fewer
    heads than pairs) or spread evenly (16 tokens, or more heads than
    pairs)."""
    inp = S.make_inputs(batch=batch, heads=heads, layout=S.LAYOUT_DS_MLA, pages=16,
                        seed=800 + heads + batch)
    st = DecodeStep(inp)
    assert B.mla_query_kernel_for(st.handle, batch).startswith("mla_absorb_pair_kernel")
    st.close()
    assert_parity(inp)


@pytest.mark.parametrize("heads", [1, 3, 5, 61, 64, 113, 127])
@pytest.mark.parametrize("batch", [24, 64])
def test_wide_kernel_head_counts(heads, batch):
    """The wide tcgen05 kernel with odd head counts: pairs without a head, a
    last two-head rope unit whose second head does not exist; and head counts
    whose split takes single-head rope units (64-row tiles: 61, 64, 113)."""
    inp = S.make_inputs(batch=batch, heads=heads, layout=S.LAYOUT_DS_MLA, pages=16,
                        seed=250 + heads + batch)
    assert_parity(inp)


@pytest.mark.parametrize("batch,heads", [(b, h) for b in (1, 2) for h in (16, 32, 64, 128)]
                         + [(3, 16), (4, 64), (5, 128), (8, 16), (8, 128)])
def test_fma_and_mma_paths_agree(batch, heads):
    """The small-batch FMA kernel (1, 2, 4 or 8 tokens a CTA; clusters of 4
    at 16 heads, of 2 above) and the tensor-core kernels meet the oracle on
    the same inputs, ragged token counts included; the KV insert is computed
    alike, bit for bit."""
    inp = S.make_inputs(batch=batch, heads=heads, layout=S.LAYOUT_DS_MLA, pages=16,
                        seed=300 + heads)
    fma, ref = assert_parity(inp, path=B.MLA_PATH_FMA)
    mma, _ = assert_parity(inp, path=B.MLA_PATH_MMA)
    # The two kernels add the squares of q_a in different orders, so a q_c
    # element may take the other rounding of a tie, and only there.
    diff = fma["q_c"] != mma["q_c"]
    near = O.bf16_midpoint_distance(ref["xq_exact"]) <= O.XQ_TIE_REL * np.abs(ref["xq_exact"])
    assert not (diff & ~near).any()
    # the KV insert sums in one order on every kernel: bit-identical rows
    assert np.array_equal(fma["cache"], mma["cache"])


def test_fma_path_refuses_large_batch():
    inp = S.make_inputs(batch=9, heads=4, layout=S.LAYOUT_E4M3, pages=4, seed=301)
    step = DecodeStep(inp)
    assert step.set_path(B.MLA_PATH_FMA) == B.MLA_OK
    assert step.decode() == B.MLA_EUNSUPPORTED
    step.close()


@pytest.mark.parametrize("batch", [1, 8, 24])
def test_fused_qkv_row_strides(batch):
    layout = S.LAYOUT_NVFP4_DS_MLA if batch == 8 else S.LAYOUT_E4M3
    inp = S.make_inputs(batch=batch, heads=16, layout=layout, pages=8, seed=400 + batch)
    assert_parity(inp, fused_row=True)


def test_q_c_optional():
    """q_c = NULL computes the same step without writing q_c: bit-identical to
    the run that writes it, which is checked against the oracle."""
    inp = S.make_inputs(batch=4, heads=8, layout=S.LAYOUT_E4M3, pages=8, seed=500)
    with_qc, _ = assert_parity(inp)
    without, flags = run_case(inp, q_c=False)
    assert flags == 0
    for k in ("q_latent", "q_pe", "cache"):
        assert np.array_equal(with_qc[k], without[k])


def test_negative_slots_skip_and_bad_slots_flag():
    inp = S.make_inputs(batch=6, heads=8, layout=S.LAYOUT_DS_MLA, pages=4, seed=600)
    cap = 4 * 64
    inp["slots"] = np.array([-1, 3, cap, 17, cap + 1000, -5], dtype=np.int64)
    out, ref = assert_parity(inp)
    assert ref["bad_slots"] == [2, 4]


def test_repeated_calls_rearm_and_match():
    """Back-to-back calls on one handle: the hand-off counters re-arm (no
    timeout flag) and every call gives the same bits."""
    inp = S.make_inputs(batch=16, heads=64, layout=S.LAYOUT_E4M3, pages=64, seed=700)
    step = DecodeStep(inp)
    outs = []
    for _ in range(5):
        assert step.decode() == B.MLA_OK
        outs.append(step.results())
    assert step.error_flags() == 0
    for o in outs[1:]:
        for k in ("q_latent", "q_pe", "q_c"):
            assert np.array_equal(o[k], outs[0][k])
    step.close()


def test_small_head_count_repeated_calls_close_every_head():
    """Small head counts run the partials kernel, whose last CTA per head adds
    the head's partials: the per-head counters must re-arm, so repeated calls
    give the same bits and no timeout flag."""
    inp = S.make_inputs(batch=4, heads=16, layout=S.LAYOUT_E4M3, pages=8, seed=710)
    st = DecodeStep(inp)
    assert B.mla_query_kernel_for(st.handle, 4) == "mla_absorb_mma_kernel<8>"
    outs = []
    for _ in range(4):
        assert st.decode() == B.MLA_OK
        outs.append(st.results())
    assert st.error_flags() == 0
    check_against_oracle(outs[0], inp)
    for o in outs[1:]:
        for k in ("q_latent", "q_pe", "q_c"):
            assert np.array_equal(o[k], outs[0][k])
    st.close()


@pytest.mark.parametrize(
    "batch,heads,path,want",
    [
        (1, 64, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<8>"),
        (2, 128, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<8>"),
        (1, 64, B.MLA_PATH_FMA, "mla_small_kernel<1,2>"),
        (2, 128, B.MLA_PATH_FMA, "mla_small_kernel<2,2>"),
        (3, 64, B.MLA_PATH_FMA, "mla_small_kernel<4,2>"),
        (8, 128, B.MLA_PATH_FMA, "mla_small_kernel<8,2>"),
        (12, 64, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<16>"),
        (40, 64, B.MLA_PATH_AUTO, "mla_wide_norm_kernel+mla_wide_kernel"),
        (1, 16, B.MLA_PATH_AUTO, "mla_small_kernel<1,"),
        (2, 16, B.MLA_PATH_AUTO, "mla_absorb_mma_kernel<8>"),
        (8, 16, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<8>"),
        (16, 16, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<16>"),
        (1, 32, B.MLA_PATH_AUTO, "mla_small_kernel<1,"),
        (1, 40, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<8>"),
        (1, 96, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<8>"),
        (2, 96, B.MLA_PATH_AUTO, "mla_absorb_pair_kernel<8>"),
        (1, 96, B.MLA_PATH_MMA, "mla_absorb_pair_kernel<8>"),
        (1, 16, B.MLA_PATH_FMA, "mla_small_kernel<1,"),
        (2, 16, B.MLA_PATH_FMA, "mla_small_kernel<2,"),
    ],
)
def test_kernel_for_names_the_split(batch, heads, path, want):
    inp = S.make_inputs(batch=1, heads=heads, layout=S.LAYOUT_E4M3, pages=2, seed=720)
    st = DecodeStep(inp)
    assert st.set_path(path) == B.MLA_OK
    got = B.mla_query_kernel_for(st.handle, batch)
    # the small-batch kernel's cluster size depends on the device's SM groups
    assert got == want or (want.endswith(",") and got.startswith(want)), got
    assert B.mla_query_kernel_for(st.handle, 0) is None
    st.close()


def test_all_paths_deterministic_across_handles():
    inp = S.make_inputs(batch=2, heads=16, layout=S.LAYOUT_E4M3, pages=8, seed=800)
    a, _ = run_case(inp)
    b, _ = run_case(inp)
    for k in ("q_latent", "q_pe", "q_c", "cache"):
        assert np.array_equal(a[k], b[k])


def test_decode_argument_errors_on_device_buffers():
    inp = S.make_inputs(batch=2, heads=4, layout=S.LAYOUT_E4M3, pages=4, seed=900)
    st = DecodeStep(inp)
    s = torch.cuda.current_stream()
    args = [st.handle, 2, st.q_a, 0, st.kv_c, 0, st.k_pe, 0, st.slots, st.cache, st.num_pages,
            st.page_size, st.layout, st.k_scale, st.q_latent, st.q_pe, st.q_c, s]

    def call(**over):
        a = list(args)
        names = ["h", "batch", "q_a", "qs", "kv_c", "ks", "k_pe", "ps", "slots", "cache", "pages",
                 "psize", "layout", "k_scale", "q_latent", "q_pe", "q_c", "stream"]
        for k, v in over.items():
            a[names.index(k)] = v
        return B.mla_query_decode(*a)

    assert call() == B.MLA_OK
    assert call(batch=0) == B.MLA_EINVAL
    assert call(batch=B.MLA_MAX_BATCH + 1) == B.MLA_EINVAL
    assert call(q_a=None) == B.MLA_EINVAL
    assert call(q_a=st.q_a.data_ptr() + 2) == B.MLA_EINVAL  # misaligned
    assert call(qs=1530) == B.MLA_EINVAL  # stride below the row width
    assert call(qs=1540) == B.MLA_EINVAL  # stride not a multiple of 8
    assert call(layout=7) == B.MLA_EINVAL
    assert call(k_scale=None) == B.MLA_EINVAL  # per-tensor layout needs k_scale
    assert call(pages=0) == B.MLA_EINVAL
    assert call() == B.MLA_OK
    torch.cuda.synchronize()
    assert st.error_flags() == 0
    st.close()


def test_weights_bound_at_create_are_read_each_call():
    """Small batches read the borrowed W_QB in place: changing it between
    calls changes the result."""
    inp = S.make_inputs(batch=1, heads=4, layout=S.LAYOUT_E4M3, pages=4, seed=1000)
    st = DecodeStep(inp)
    assert st.decode() == B.MLA_OK
    first = st.results()
    st.w_qb.mul_(2.0)
    assert st.decode() == B.MLA_OK
    second = st.results()
    inp2 = dict(inp)
    inp2["w_qb"] = (O.f64_to_bf16_bits(2.0 * O.bf16_bits_to_f64(inp["w_qb"])))
    check_against_oracle(second, inp2)
    assert not np.array_equal(first["q_pe"], second["q_pe"])
    st.close()


def test_per_tensor_insert_divides_by_k_scale():
    """k_pe goes into the per-tensor row divided by k_scale, with no norm.
    With k_scale = 7 and k_pe = 91 * 2**-10 the quotient 13 * 2**-10 is an
    E4M3 tie that rounds to the even code 0x06; multiplying by the binary32
    reciprocal of 7 would give 0x07.  The oracle pins the same case."""
    inp = S.make_inputs(batch=2, heads=4, layout=S.LAYOUT_E4M3, pages=4, seed=1100)
    v = O.f64_to_bf16_bits(np.array([91 * 2.0**-10, -91 * 2.0**-10]))
    inp["k_pe"][0, :] = v[0]
    inp["k_pe"][1, :] = v[1]
    inp["k_scale"] = 7.0
    out, ref = assert_parity(inp)
    for b, want in ((0, 0x06), (1, 0x86)):
        s = int(inp["slots"][b])
        row = out["cache"][s // 64, s % 64]
        assert np.all(row[512:] == want), (b, row[512:520])


def test_batches_above_16_read_the_create_time_copy():
    """Batches above 16 tokens run the wide kernel, which reads the W_QB and
    W_UK^T tiles copied at create: changing W_QB in place afterwards leaves
    their results as they were (still the oracle's for the weights at create),
    while a batch of up to 16 tokens reads the changed W_QB."""
    inp = S.make_inputs(batch=24, heads=8, layout=S.LAYOUT_E4M3, pages=8, seed=1010)
    st = DecodeStep(inp)
    assert B.mla_query_kernel_for(st.handle, 24) == "mla_wide_norm_kernel+mla_wide_kernel"
    assert st.decode() == B.MLA_OK
    first = st.results()
    check_against_oracle(first, inp)
    st.w_qb.mul_(2.0)
    assert st.decode() == B.MLA_OK
    second = st.results()
    for k in ("q_latent", "q_pe", "q_c"):
        assert np.array_equal(first[k], second[k]), k
    assert st.decode(batch=4) == B.MLA_OK  # four tokens: W_QB read in place
    small = st.results()
    assert not np.array_equal(small["q_pe"][:4], first["q_pe"][:4])
    st.close()


@pytest.mark.parametrize("heads", [64, 128])
def test_create_allocates_only_what_the_dispatch_reaches(heads):
    """On a GB300 at 64 or 128 heads every batch takes the paired kernel (up
    to 16 tokens, weights read in place) or the wide kernel (its tiled copies
    of W_QB and W_UK^T, H * 704 KiB): create allocates those copies and a few
    hundred KiB besides, not the partials buffer (H * 256 KiB), the packed
    W_UK (H * 128 KiB) or the hand-off q buffer."""
    inp = S.make_inputs(batch=1, heads=heads, layout=S.LAYOUT_E4M3, pages=2, seed=1020)
    dev = torch.device("cuda", 0)
    from mla_query_projection_gb300.runner import bf16_tensor

    w = [bf16_tensor(inp[k], dev) for k in ("w_qb", "w_uk", "gamma_q", "gamma_kv")]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    h = B.mla_query_create(heads, *w, float(inp["eps"]))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    used = free0 - free1
    wide = heads * 704 * 1024
    assert B.mla_query_kernel_for(h, 1) == "mla_absorb_pair_kernel<8>"
    assert B.mla_query_kernel_for(h, 64) == "mla_wide_norm_kernel+mla_wide_kernel"
    # allocations are rounded to 2 MiB pages
    assert used <= wide + 6 * 1024 * 1024, (used, wide)
    B.mla_query_destroy(h)
