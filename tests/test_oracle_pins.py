"""Pins of the FP64 oracle to things other than itself.

Each test fixes one part of the oracle against hand-worked encodings of the
number formats, brute force on tiny inputs, invariants of the method, or an
independent library conversion, so that a dropped term, a wrong sign or index
or a transposed operand fails at least one of them.  CPU only.
"""

import math
import os

import numpy as np
import pytest
import torch

from mla_query_projection_gb300 import synthetic as S
from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- bfloat16


@pytest.mark.parametrize(
    "value,bits",
    [
        (1.0, 0x3F80),
        (-2.0, 0xC000),
        (3.0, 0x4040),
        (0.1, 0x3DCD),  # 1.6 * 2**-4: mantissa 76.8 -> 77
        (1.0 + 2.0**-8, 0x3F80),  # tie -> even
        (1.0 + 3 * 2.0**-8, 0x3F82),  # tie -> even
        (1.0 + 2.0**-8 + 2.0**-30, 0x3F81),  # just above the tie
        ((2.0 - 2.0**-7) * 2.0**127, 0x7F7F),  # largest finite
        (2.0**-133, 0x0001),  # smallest subnormal
        (2.0**-134, 0x0000),  # tie with zero -> even
        (3 * 2.0**-134, 0x0002),  # tie -> even
        (-0.0, 0x8000),
    ],
)
def test_bf16_hand_worked(value, bits):
    assert int(O.f64_to_bf16_bits(np.array([value]))[0]) == bits


def test_bf16_matches_torch_cast_on_binary32_values():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-30, 30, 200_000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_decode_roundtrip():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    assert np.array_equal(O.f64_to_bf16_bits(vals[finite]), bits[finite])


# ---------------------------------------------------------------- E4M3


def test_e4m3_hand_worked_table():
    for value, code in _read_table("e4m3_codes.txt"):
        got = int(O.e4m3_satfinite(np.array([float(value)]))[0])
        assert got == int(code, 16), (value, hex(got), code)


def test_e4m3_decode_matches_torch_and_roundtrips():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = O.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin].astype(np.float64))
    assert np.array_equal(O.e4m3_satfinite(got[fin]), codes[fin])


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-12, 6.5, 200_000))).astype(np.float32)
    x = x[np.abs(x) < 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_satfinite(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_saturates_never_nan():
    big = np.array([448.0, 463.99, 464.0, 500.0, 1e6, -1e6, -470.0])
    codes = O.e4m3_satfinite(big)
    assert set(codes.tolist()) <= {0x7E, 0xFE}


# ---------------------------------------------------------------- pow2_ceil


def _page_pow2_ceil(v32: np.ndarray) -> np.ndarray:
    """The integer form printed with pow2_ceil: take the binary32 bits, keep the
    exponent field, add one if any mantissa bit is set, shift back."""
    bits = v32.astype(np.float32).view(np.uint32)
    e = bits >> np.uint32(23)
    e = e + (bits & np.uint32(0x7FFFFF) != 0).astype(np.uint32)
    return (e << np.uint32(23)).view(np.float32).astype(np.float64)


def test_pow2_ceil_table():
    for kind, v, want in _read_table("pow2_ceil.txt"):
        v, want = float(v), float(want)
        got = O.pow2_ceil(np.float32(v)) if kind == "p2c" else O.ds_tile_scale(v)
        assert float(got) == want, (kind, v, float(got), want)


def test_pow2_ceil_matches_integer_form():
    rng = np.random.default_rng(13)
    v = np.exp2(rng.uniform(-120, 120, 300_000)).astype(np.float32)
    v = np.concatenate([v, np.exp2(np.arange(-126, 127)).astype(np.float32)])
    assert np.array_equal(O.pow2_ceil(v.astype(np.float64)), _page_pow2_ceil(v))


def test_ds_tile_scale_uses_division_by_448():
    # amax = 1.75 * 2**k gives exactly 2**(k-8) only with a correctly rounded
    # division; every such scale must be the exact power of two.
    for k in range(-10, 12):
        assert float(O.ds_tile_scale(1.75 * 2.0**k)) == max(2.0 ** (k - 8), 2.0**-13)


# ---------------------------------------------------------------- RMSNorm


def test_rmsnorm_worked_example():
    out = O.rmsnorm(np.array([[3.0, 4.0]]), np.ones(2), 0.0)
    assert np.allclose(out, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=0, atol=1e-15)
    assert abs(out[0, 0] - 0.848528137423857) < 1e-14
    assert abs(out[0, 1] - 1.131370849898476) < 1e-14


def test_rmsnorm_gamma_and_eps():
    out = O.rmsnorm(np.array([[3.0, 4.0]]), np.array([2.0, 0.5]), 0.0)
    assert np.allclose(out, [[6 / math.sqrt(12.5), 2 / math.sqrt(12.5)]], atol=1e-15)
    # eps is added to the mean of squares, not to the root
    out = O.rmsnorm(np.array([[1.0, 1.0]]), np.ones(2), 3.0)
    assert np.allclose(out, [[0.5, 0.5]], atol=1e-15)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((4, 1536))
    g = 1 + 0.1 * rng.standard_normal(1536)
    a = O.rmsnorm(x, g, 0.0)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    for c in (0.1, 3.0, 10.0):
        # without eps the norm is exactly scale-free
        assert np.max(np.abs(a - O.rmsnorm(c * x, g, 0.0)) / np.abs(a)) < 1e-13
        # with eps the change is the closed-form factor sqrt((ms+eps)/(ms+eps/c^2))
        b = O.rmsnorm(c * x, g, 1e-6)
        ratio = np.sqrt((ms + 1e-6) / (ms + 1e-6 / c**2))
        assert np.max(np.abs(b / O.rmsnorm(x, g, 1e-6) - ratio)) < 1e-13


# ---------------------------------------------------------------- Q_B and W_UK


def test_q_projection_brute_force():
    rng = np.random.default_rng(15)
    B, H = 2, 2
    xq = rng.standard_normal((B, 1536))
    w = rng.standard_normal((H * 192, 1536))
    q, cond = O.q_projection(xq, w, H)
    for b in range(B):
        for h in range(H):
            for p in (0, 1, 77, 127, 128, 150, 191):
                s = 0.0
                a = 0.0
                for k in range(1536):
                    s += xq[b, k] * w[h * 192 + p, k]
                    a += abs(xq[b, k] * w[h * 192 + p, k])
                assert abs(q[b, h, p] - s) <= 1e-12 * a
                assert abs(cond[b, h, p] - a) <= 1e-12 * a


def test_q_projection_one_hot_indexing():
    H = 3
    w = np.arange(H * 192 * 1536, dtype=np.float64).reshape(H * 192, 1536)
    for k in (0, 5, 1535):
        xq = np.zeros((1, 1536))
        xq[0, k] = 1.0
        q, _ = O.q_projection(xq, w, H)
        for h in range(H):
            for p in (0, 127, 128, 191):
                assert q[0, h, p] == w[h * 192 + p, k]


def test_absorb_brute_force_and_one_hot():
    rng = np.random.default_rng(16)
    B, H = 2, 2
    qn = rng.standard_normal((B, H, 128))
    w = rng.standard_normal((H, 128, 512))
    lat, cond = O.absorb(qn, w)
    for b in range(B):
        for h in range(H):
            for c in (0, 1, 255, 511):
                s = sum(qn[b, h, p] * w[h, p, c] for p in range(128))
                a = sum(abs(qn[b, h, p] * w[h, p, c]) for p in range(128))
                assert abs(lat[b, h, c] - s) <= 1e-12 * a
                assert abs(cond[b, h, c] - a) <= 1e-12 * a
    e = np.zeros((1, H, 128))
    e[0, 1, 37] = 1.0
    lat, _ = O.absorb(e, w)
    assert np.array_equal(lat[0, 1], w[1, 37])
    assert np.all(lat[0, 0] == 0)


def test_absorb_equals_unabsorbed_score():
    """q_nope . (W_UK[h] @ c) == (absorbed q) . c for any latent vector c: the
    absorbed query scores a latent KV row exactly as the unabsorbed query scores
    the key it up-projects to."""
    rng = np.random.default_rng(17)
    H = 3
    qn = rng.standard_normal((2, H, 128))
    w = rng.standard_normal((H, 128, 512))
    lat, _ = O.absorb(qn, w)
    c = rng.standard_normal(512)
    for b in range(2):
        for h in range(H):
            k_nope = w[h] @ c
            lhs = qn[b, h] @ k_nope
            rhs = lat[b, h] @ c
            assert abs(lhs - rhs) <= 1e-12 * (np.abs(qn[b, h]) @ np.abs(w[h]) @ np.abs(c))


# ---------------------------------------------------------------- KV rows


def _bf16(vals):
    return O.f64_to_bf16_bits(np.asarray(vals, dtype=np.float64))


def _hand_inputs(layout, pages=2, page_size=4, slots=(5,), H=1):
    B = len(slots)
    row = O.ROW_BYTES[layout]
    rng = np.random.default_rng(18)
    cache = rng.integers(0, 256, (pages, page_size, row), dtype=np.uint8)
    return dict(
        w_qb=_bf16(np.zeros((H * 192, 1536))),
        w_uk=_bf16(np.zeros((H, 128, 512))),
        gamma_q=_bf16(np.ones(1536)),
        gamma_kv=_bf16(np.ones(512)),
        q_a=_bf16(np.ones((B, 1536))),
        kv_c=_bf16(np.ones((B, 512))),
        k_pe=_bf16(np.full((B, 64), 2.0)),
        slots=np.array(slots, dtype=np.int64),
        cache=cache,
        layout=layout,
        k_scale=0.05,
        eps=1e-6,
    )


def test_kv_row_per_tensor_worked():
    # kv_c = 1 -> normed = bf16(1/sqrt(1 + 1e-6)) = 1.0; 1.0 / fp32(0.05) rounds
    # to 20.0 -> E4M3 0x5A; k_pe 2.0 / 0.05 -> 40.0 -> 0x62.
    inp = _hand_inputs(0)
    out = O.decode_step(inp)
    row = out["cache"][1, 1]  # slot 5, page size 4
    assert np.all(row[:512] == 0x5A)
    assert np.all(row[512:] == 0x62)
    other = np.ones(inp["cache"].shape[:2], bool)
    other[1, 1] = False
    assert np.array_equal(out["cache"][other], inp["cache"][other])


def test_kv_row_per_tensor_divides_by_k_scale():
    """The per-tensor row divides by k_scale; multiplying by the binary32
    reciprocal gives a different byte here.  k_scale = 7 and the value
    91 * 2**-10 (BF16, seven significant bits): the quotient is exactly
    13 * 2**-10 = 6.5 * 2**-9, halfway between the E4M3 subnormals 6 * 2**-9
    (0x06) and 7 * 2**-9 (0x07); ties go to the even code, 0x06.  The binary32
    reciprocal of 7 is 9586981 * 2**-26 > 1/7, so the product lands above the
    midpoint and would round to 0x07.  With k_scale = 0.05 both forms give the
    same bytes on every BF16 value, so the workloads' scale cannot tell them
    apart; this case does."""
    v = 91 * 2.0**-10
    assert O.round_to_bf16(v) == v
    assert np.float32(1.0) / np.float32(7.0) == np.float32(9586981 * 2.0**-26)
    normed = np.full(512, v)
    k_pe = np.full(64, -v)
    row = O.kv_row_e4m3(normed, k_pe, 7.0)
    assert np.all(row[:512] == 0x06)
    assert np.all(row[512:] == 0x86)
    # the other reading would have given 0x07: this pin tells the two apart
    prod = float(np.float32(v) * (np.float32(1.0) / np.float32(7.0)))
    assert O.e4m3_satfinite(prod) == 0x07


def test_kv_row_ds_worked():
    # normed = 1.0 -> amax 1 -> 1/448 -> scale 2**-8; 1.0 * 256 -> E4M3 0x78;
    # scale bits 0x3B800000 little-endian; k_pe BF16 2.0 = 0x4000 little-endian.
    inp = _hand_inputs(1)
    out = O.decode_step(inp)
    row = out["cache"][1, 1]
    assert np.all(row[:512] == 0x78)
    assert list(row[512:528]) == [0x00, 0x00, 0x80, 0x3B] * 4
    assert list(row[528:]) == [0x00, 0x40] * 64


def test_kv_ds_scale_per_tile_and_k_pe_raw():
    inp = _hand_inputs(1)
    kv = np.ones((1, 512))
    kv[0, 128:256] *= 8.0  # tile 1 larger
    kv[0, 300] = 64.0  # one big value in tile 2
    inp["kv_c"] = _bf16(kv)
    kpe = np.linspace(-3, 3, 64)[None]
    inp["k_pe"] = _bf16(kpe)
    out = O.decode_step(inp)
    row = out["cache"][1, 1]
    scales = row[512:528].view("<f4").astype(np.float64)
    n = out["kv_normed"][0]
    for t in range(4):
        want = O.pow2_ceil(max(np.float32(np.max(np.abs(n[128 * t:128 * t + 128])) / 448), np.float32(1e-4)))
        assert scales[t] == want
    assert scales[1] > scales[0] and scales[2] > scales[1]
    assert np.array_equal(row[528:].view("<u2"), inp["k_pe"][0])
    # the element holding a tile's amax maps near the top of the E4M3 range
    assert O.e4m3_to_f64(row[300:301])[0] * scales[2] == pytest.approx(n[300], rel=2**-3)


def test_slot_math_every_slot():
    pages, ps = 3, 4
    slots = list(range(pages * ps)) + [-1]
    for layout in (0, 1, 2):
        inp = _hand_inputs(layout, pages=pages, page_size=ps, slots=slots)
        kv = np.tile(np.linspace(0.5, 2.0, 512), (len(slots), 1)) * np.arange(1, len(slots) + 1)[:, None]
        inp["kv_c"] = _bf16(kv)
        out = O.decode_step(inp)
        for b, s in enumerate(slots[:-1]):
            one = dict(inp)
            one.update(
                kv_c=inp["kv_c"][b:b + 1], k_pe=inp["k_pe"][b:b + 1],
                q_a=inp["q_a"][b:b + 1], slots=np.array([s]),
            )
            row = O.decode_step(one)["cache"][s // ps, s % ps]
            assert np.array_equal(out["cache"][s // ps, s % ps], row)
            if layout == 0:
                # one byte the hand derivation fixes: normed = bf16 of the row/rms
                assert row.shape == (576,)


def test_negative_and_out_of_range_slots_are_skipped():
    inp = _hand_inputs(0, pages=2, page_size=4, slots=(-1, 8, 100))
    out = O.decode_step(inp)
    assert np.array_equal(out["cache"], inp["cache"])
    assert out["bad_slots"] == [1, 2]


# ---------------------------------------------------------------- whole step


def test_decode_step_constructed_example():
    """A step whose every output follows by hand: q_a = 1 and gamma = 1 give
    xq = bf16(1/sqrt(1+eps)) = 1; row p of every head is constant
    (p+1) * 2**-12, so q[p] = bf16(0.375 (p+1)); W_UK[h, p, c] = 3 * 2**-8 when
    p == c % 128, so q_latent[c] = bf16(3 * 2**-8 * q[c % 128]) (the rounded q)."""
    H = 2
    inp = _hand_inputs(0, H=H, slots=(2,))
    w_qb = np.zeros((H * 192, 1536))
    for h in range(H):
        for p in range(192):
            w_qb[h * 192 + p, :] = (p + 1) * 2.0**-12 * (1 + h)
    w_uk = np.zeros((H, 128, 512))
    for c in range(512):
        w_uk[:, c % 128, c] = 3 * 2.0**-8
    inp["w_qb"] = _bf16(w_qb)
    inp["w_uk"] = _bf16(w_uk)
    out = O.decode_step(inp)
    assert np.all(out["q_c"] == 0x3F80)
    for h in range(H):
        q = O.round_to_bf16(0.375 * np.arange(1, 193) * (1 + h))
        assert np.array_equal(O.bf16_bits_to_f64(out["q_pe"][0, h]), q[128:])
        want = O.round_to_bf16(3 * 2.0**-8 * q[np.arange(512) % 128])
        assert np.array_equal(O.bf16_bits_to_f64(out["q_latent"][0, h]), want)
    # the unrounded q would give a different latent for some columns
    qx = 0.375 * np.arange(1, 129)
    assert np.any(O.round_to_bf16(3 * 2.0**-8 * qx) != O.round_to_bf16(3 * 2.0**-8 * O.round_to_bf16(qx)))


def test_decode_step_shapes_on_a_workload():
    from mla_query_projection_gb300 import synthetic as S

    inp = S.workload_inputs("tiny_b1_h16_e4m3")
    out = O.decode_step(inp)
    assert out["q_c"].shape == (1, 1536)
    assert out["q_pe"].shape == (1, 16, 64)
    assert out["q_latent"].shape == (1, 16, 512)
    assert out["cache"].shape == (8, 64, 576)
    changed = np.any(out["cache"] != inp["cache"], axis=-1)
    s = int(inp["slots"][0])
    assert changed.sum() == 1 and changed[s // 64, s % 64]


# ---------------------------------------------------------------- tie zones


def test_bf16_midpoint_helpers_hand_worked():
    x = np.array([1.0 + 2.0**-8, 1.0 + 2.0**-9, 3.0, -0.95117186, 2.0**-140])
    d = O.bf16_midpoint_distance(x)
    assert d[0] == 0.0  # exactly halfway between 1.0 and 1 + 2**-7
    assert d[1] == 2.0**-9  # a quarter quantum from 1.0, a quarter from the midpoint
    assert d[2] == 2.0**-7  # representable (quantum 2**-6 in [2, 4)): half a quantum away
    assert abs(d[3] - 1.5e-8) < 1e-15
    other = O.bf16_other_rounding(x)
    assert other[0] == 1.0078125 and O.round_to_bf16(x[0]) == 1.0
    assert other[1] == 1.0078125
    assert other[2] == 3.0
    assert other[3] == -0.953125 and O.round_to_bf16(x[3]) == -0.94921875


def test_decode_step_alternate_rounding_of_a_tie():
    """Marking the normalised element nearest a BF16 tie moves only that q_c
    element, by one quantum; marking an element far from a tie is refused."""
    inp = _hand_inputs(0, H=1, slots=(1,))
    rng = np.random.default_rng(19)
    inp["q_a"] = _bf16(rng.standard_normal((1, 1536)))
    ref = O.decode_step(inp)
    dist = O.bf16_midpoint_distance(ref["xq_exact"]) / np.abs(ref["xq_exact"])
    k = int(np.argmin(dist))
    if dist[0, k] <= O.XQ_TIE_REL:
        alt = np.zeros((1, 1536), bool)
        alt[0, k] = True
        out = O.decode_step(inp, xq_alt=alt)
        moved = out["q_c"] != ref["q_c"]
        assert moved.sum() == 1 and moved[0, k]
        q = O.bf16_quantum(ref["xq_exact"][0, k])
        assert abs(O.bf16_bits_to_f64(out["q_c"])[0, k] - O.bf16_bits_to_f64(ref["q_c"])[0, k]) == q
    far = int(np.argmax(dist))
    alt = np.zeros((1, 1536), bool)
    alt[0, far] = True
    with pytest.raises(ValueError):
        O.decode_step(inp, xq_alt=alt)


# --------------------------------------------------------------- FP8 query
# Page "mla.query", method kernel (FP8 query epilogue): fp8(bf16(v) * q_scale_inv).


@pytest.mark.parametrize(
    "value,qsi,code",
    [
        (1.0, 2.0, 0x40),      # 2.0
        (0.5, 0.25, 0x20),     # 0.125 = 2^-3: exponent field 4
        (-1.5, 1.0, 0xBC),     # -1.5: sign, exponent 7, mantissa 100
        (300.0, 2.0, 0x7E),    # 600 saturates to 448
        (-300.0, 2.0, 0xFE),
        (1.0625, 1.0, 0x38),   # tie between 1.0 and 1.125: to even
        (1.1875, 1.0, 0x3A),   # tie between 1.125 and 1.25: to even
        (0.0, 5.0, 0x00),
    ],
)
def test_query_fp8_hand_worked(value, qsi, code):
    bits = O.f64_to_bf16_bits(np.array([value]))
    assert int(O.query_fp8(bits, qsi)[0]) == code


def test_query_fp8_rounds_the_output_to_bf16_first():
    """The scale multiplies the BF16 output, not the exact value: a value just
    above a BF16 midpoint scales to a different FP8 code than its rounding."""
    # exact 1.0 + 2^-8 + tiny rounds (BF16, 8 bits) to 1.0078125; times 1.0 the
    # FP8 code then follows the rounded value 1.0078125 -> 0x38 (nearest 1.0)
    bits = O.f64_to_bf16_bits(np.array([1.0 + 2.0**-8 + 2.0**-20]))
    assert float(O.bf16_bits_to_f64(bits)[0]) == 1.0078125
    assert int(O.query_fp8(bits, 1.0)[0]) == 0x38
    assert int(O.query_fp8(bits, 8.0)[0]) == 0x50  # 8.0625 -> 8 (0x50)


def test_decode_step_fp8_query_outputs_follow_the_bf16_outputs():
    inp = S.make_inputs(batch=2, heads=2, layout=S.LAYOUT_E4M3, pages=4, seed=77)
    inp["q_scale_inv"] = 4.0
    out = O.decode_step(inp)
    assert out["q_latent_fp8"].shape == out["q_latent"].shape
    assert out["q_pe_fp8"].shape == out["q_pe"].shape
    # each code decodes to the E4M3 value nearest 4 x the BF16 output
    for k in ("q_latent", "q_pe"):
        want = 4.0 * O.bf16_bits_to_f64(out[k])
        got = O.e4m3_to_f64(out[k + "_fp8"])
        step = np.abs(got) * 2.0**-3 + 2.0**-9
        assert np.all(np.abs(got - np.clip(want, -448, 448)) <= step)


# ---------------------------------------------------------------- nvfp4_ds_mla


E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # codes 0..7


def test_e2m1_hand_worked_table():
    for value, code in _read_table("e2m1_codes.txt"):
        got = int(O.e2m1_satfinite(np.array([float(value)]))[0])
        assert got == int(code, 16), (value, hex(got), code)


def test_e2m1_decode_and_roundtrip():
    codes = np.arange(16, dtype=np.uint8)
    want = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
    got = O.e2m1_to_f64(codes)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got[8:]), np.ones(8, bool))  # code 8 is -0
    assert np.array_equal(O.e2m1_satfinite(got), codes)


def test_e2m1_is_the_nearest_value_ties_to_even():
    """Brute force over the eight magnitudes: the nearest one, the one with
    mantissa bit 0 (an even code) on a tie, 6 beyond the range."""
    rng = np.random.default_rng(31)
    x = np.concatenate([rng.uniform(-8, 8, 20_000), np.arange(-32, 33) / 4.0])
    mags = np.array(E2M1_MAGNITUDES)
    got = O.e2m1_satfinite(x)
    for v, c in zip(x, got):
        d = np.abs(mags - min(abs(v), 6.0))
        best = np.flatnonzero(d == d.min())
        k = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        assert (int(c) & 7) == k, (v, int(c))
        assert (int(c) >> 3) == (1 if np.signbit(v) else 0), (v, int(c))


@pytest.mark.parametrize(
    "amax, code, value",
    [
        (6.0, 0x38, 1.0),  # 6 / 6 = 1: E4M3 E=7, m=0
        (3.0, 0x30, 0.5),  # 0.5: E=6
        (0.0, 0x01, 2.0**-9),  # floor 2**-9: the smallest E4M3 subnormal
        (6 * 2.0**-10, 0x01, 2.0**-9),  # 2**-10 is below the floor
        (7.0, 0x39, 1.125),  # 1.1667 -> nearer 1.125 (m=1) than 1.25
        (6.375, 0x38, 1.0),  # 1.0625: tie 1.0 / 1.125 -> even (m=0)
        (1.0, 0x23, 0.171875),  # 1/6 = 1.333 * 2**-3 -> m=3 (1.375): E=4
        (2688.0, 0x7E, 448.0),  # 448: the largest finite E4M3
        (1e5, 0x7E, 448.0),  # saturates
    ],
)
def test_nvfp4_block_scale_hand_worked(amax, code, value):
    c, v, inv = O.nvfp4_block_scale(amax)
    assert int(c) == code and float(v) == value
    assert float(inv) == float(np.float32(1.0) / np.float32(value))


def test_nvfp4_values_use_the_stored_scale():
    """Block amax 7: the stored scale is 1.125 (not 7/6), and 2.875 / 1.125 =
    2.556 rounds to E2M1 3 (code 5), where 2.875 / (7/6) = 2.464 would give 2.
    7 / 1.125 = 6.22 saturates to 6 (code 7)."""
    n = np.zeros(512)
    n[0], n[1] = 7.0, 2.875
    row, scales = O.kv_row_nvfp4(n, np.zeros(64))
    assert row[0] == 0x57  # value 0 in the low half, value 1 in the high half
    assert row[O.NVFP4_SCALES] == 0x39 and scales[0] == 1.125
    assert np.all(row[8:256] == 0x00)  # zero blocks: zero codes
    assert np.all(row[O.NVFP4_SCALES + 1:O.NVFP4_SCALES + 8] == 0x01)  # blocks 4, 8, ..: floor


def test_kv_row_nvfp4_worked():
    # kv_c = 1 -> normed 1.0 -> amax 1 -> scale code 0x23 (0.171875), reciprocal
    # 5.8181820 -> 1.0 * 5.818 rounds to E2M1 6 (code 7) -> byte 0x77; k_pe 2.0
    # stored unscaled -> E4M3 0x40.
    inp = _hand_inputs(2)
    out = O.decode_step(inp)
    row = out["cache"][1, 1]
    assert row.shape == (352,)
    assert np.all(row[:256] == 0x77)
    assert np.all(row[256:288] == 0x23)
    assert np.all(row[288:] == 0x40)


def test_nvfp4_nibble_order_and_scale_placement():
    """Block s of 16 values has amax 6 * 2**-(s % 7) * (1 + (s // 8) / 8), so its
    scale is exactly 2**-(s % 7) * (1 + (s // 8) / 8), a normal E4M3 value:
    code ((7 - s % 7) << 3) | (s // 8).  The scale of block s sits at byte
    256 + 8 * (s % 4) + s // 4; every scale byte is written once.  Within a
    block, values [6, -3, 1.5, 0.5, 4, 0, ...] times the scale give codes
    7, 0xD, 3, 1, 6, 0: bytes 0xD7, 0x13, 0x06."""
    n = np.zeros(512)
    pattern = np.array([6.0, -3.0, 1.5, 0.5, 4.0] + [0.0] * 11)
    for s in range(32):
        n[16 * s:16 * s + 16] = pattern * 2.0 ** -(s % 7) * (1 + (s // 8) / 8)
    row, _ = O.kv_row_nvfp4(n, np.zeros(64))
    placed = sorted(O.nvfp4_scale_byte(s) for s in range(32))
    assert placed == list(range(256, 288))
    assert O.nvfp4_scale_byte(5) == 265
    for s in range(32):
        assert row[256 + 8 * (s % 4) + s // 4] == ((7 - s % 7) << 3) | (s // 8), s
        assert list(row[8 * s:8 * s + 3]) == [0xD7, 0x13, 0x06], s
        assert np.all(row[8 * s + 3:8 * s + 8] == 0)


def test_nvfp4_dequantised_row_error_bound():
    """E2M1 code times the stored scale is within half an E2M1 step of the
    scaled value: |n - deq| <= sf * max(0.25, |n / sf| / 4), the slack of the
    top step (4..6, step 2) also covering saturation (|n / sf| <= 6 * 17/16
    after the scale's E4M3 rounding).  The bound holds while every scale is a
    normal E4M3 value below 448, as for RMS-normalised rows (|n| <= sqrt(512)
    times gamma)."""
    rng = np.random.default_rng(32)
    for trial in range(50):
        n = O.round_to_bf16(rng.standard_normal(512) * np.exp(rng.uniform(-1.5, 1.5)))
        n[rng.random(512) < 0.01] *= 20.0
        row, scales = O.kv_row_nvfp4(n, np.zeros(64))
        assert scales.min() >= 2.0**-6 and scales.max() < 448.0
        codes = np.empty(512, np.uint8)
        codes[0::2] = row[:256] & 0xF
        codes[1::2] = row[:256] >> 4
        sf = np.repeat(scales, 16)
        deq = O.e2m1_to_f64(codes) * sf
        bound = sf * np.maximum(0.25, np.abs(n / sf) / 4) * (1 + 2.0**-20)
        assert np.all(np.abs(n - deq) <= bound), trial
        # the decoded scale bytes are the returned scales
        for s in range(32):
            assert O.e4m3_to_f64(row[O.nvfp4_scale_byte(s):O.nvfp4_scale_byte(s) + 1])[0] == scales[s]


def test_nvfp4_power_of_two_scaling_moves_only_the_scales():
    """Scaling the row by 2**k (scales stay normal E4M3 and above the floor)
    multiplies every scale by 2**k and leaves every E2M1 code unchanged."""
    rng = np.random.default_rng(33)
    n = O.round_to_bf16(rng.standard_normal(512) * 4.0)
    base, sb = O.kv_row_nvfp4(n, np.zeros(64))
    for k in (-3, -1, 2, 5):
        row, sk = O.kv_row_nvfp4(n * 2.0**k, np.zeros(64))
        assert np.array_equal(row[:256], base[:256]), k
        assert np.array_equal(sk, sb * 2.0**k), k


def test_nvfp4_k_pe_is_unscaled_e4m3():
    kpe = O.round_to_bf16(np.linspace(-500, 500, 64))
    row, _ = O.kv_row_nvfp4(np.ones(512), kpe)
    ref = torch.from_numpy(kpe.astype(np.float32)).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(row[288:], ref.view(torch.uint8).numpy())


# ---------------------------------------------------------------- qkv_a projection


def test_qkv_a_projection_brute_force():
    rng = np.random.default_rng(41)
    B, N, K = 3, 5, 37
    x = _bf16(rng.standard_normal((B, K)))
    w = _bf16(rng.standard_normal((N, K)) * 0.1)
    y, exact, cond = O.qkv_a_projection(x, w)
    xf, wf = O.bf16_bits_to_f64(x), O.bf16_bits_to_f64(w)
    for b in range(B):
        for n in range(N):
            s = a = 0.0
            for k in range(K):
                s += xf[b, k] * wf[n, k]
                a += abs(xf[b, k] * wf[n, k])
            assert abs(exact[b, n] - s) <= 1e-12 * a
            assert abs(cond[b, n] - a) <= 1e-12 * a
            assert y[b, n] == _bf16([s])[0]


def test_qkv_a_projection_one_hot_and_orientation():
    """x = e_k picks column k of W for every output row: y[b, n] = W[n, k]
    (W is [N, K], rows are outputs); a transposed operand would fail."""
    N, K = 6, 10
    w = _bf16(np.arange(N * K, dtype=np.float64).reshape(N, K) / 64.0)
    for k in (0, 3, 9):
        x = np.zeros((1, K))
        x[0, k] = 1.0
        y, _, _ = O.qkv_a_projection(_bf16(x), w)
        assert np.array_equal(y[0], w[:, k])


def test_qkv_a_projection_rounds_once():
    """Terms whose exact sum is 1 + 2**-9 (below the BF16 midpoint 1 + 2**-8)
    give 1.0; 1 + 3 * 2**-9 (above it) gives 1 + 2**-7."""
    w = _bf16([[1.0, 2.0**-9, 0.0], [1.0, 2.0**-9, 2.0**-8]])
    y, exact, _ = O.qkv_a_projection(_bf16([[1.0, 1.0, 1.0]]), w)
    assert exact[0, 0] == 1 + 2.0**-9 and y[0, 0] == _bf16([1.0])[0]
    assert exact[0, 1] == 1 + 3 * 2.0**-9 and y[0, 1] == _bf16([1 + 2.0**-7])[0]
