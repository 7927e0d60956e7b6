"""FP64 CPU oracle for one decode step of the MLA query path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

What it computes follows the vLLM API page "mla.query" (module
``vllm/models/kimi_k3/nvidia/specialized_decode/cutedsl/mla/query.py``), class
``MlaQuery``:

* ``kernel`` section (q_a RMSNorm, Q_B projection, W_UK absorption): the q_a row
  is RMS-normalised and multiplied by its gamma, rounded once to BF16 (that row
  is also the ``q_c`` output, see ``store_qc``); every Q_B row is a 1536-long dot
  product rounded once to BF16; rows 0..127 of a head ("nope") feed the
  absorption through ``W_UK[head, p, c]``, rows 128..191 ("rope") are emitted
  unchanged as ``q_pe``.
* ``insert`` / ``kv_fp8`` sections: the 512-wide kv_c row is RMS-normalised,
  multiplied by gamma_kv and rounded to BF16; each value and each raw k_pe value
  is divided by ``k_scale`` and stored as an FP8 E4M3 byte at
  ``cache[slot // page_size, slot % page_size]``; a negative slot skips the row.
* ``insert_ds`` section and ``pow2_ceil`` function: the ``fp8_ds_mla`` row keeps
  one power-of-two scale per 128-column tile,
  ``exp2(ceil(log2(max(amax / 448, 1e-4))))``, and stores k_pe as raw BF16.
* ``insert_nvfp4`` section: the ``nvfp4_ds_mla`` row keeps one E4M3 scale
  ``max(amax / 6, 2**-9)`` per 16-value block, stores the values as E2M1 of
  ``x * (1 / scale)`` and k_pe as unscaled E4M3.

Every quantity is kept in float64; values are rounded only where the page
rounds them (the ``BFloat16(...)`` casts, the FP32 quotient and the FP8 casts).
Where the page is silent (the q_a norm helper is not printed, the FP8 cast's
overflow rule, the byte offsets of the ds scales and k_pe) the plainest reading
is taken; each reading is stated at the function that takes it.

Parity pins: every function here is pinned by CPU tests in
``tests/test_oracle_pins.py`` against hand-worked values of the number formats,
brute force, invariants and an independent library conversion.
"""

from __future__ import annotations

import numpy as np

# Geometry fixed by the method (page "mla.query", class MlaQuery: q_a rows of
# 1536, 192 Q_B rows per head of which 128 "nope" and 64 "rope", a 512-wide
# latent space, a 64-wide k_pe).
Q_LORA = 1536
QK_NOPE = 128
QK_ROPE = 64
QK_HEAD = QK_NOPE + QK_ROPE  # 192
KV_LORA = 512
DS_TILE = 128
# Row sizes of the two cache layouts: 512 E4M3 + 64 E4M3 k_pe; and
# 512 E4M3 + 4 FP32 tile scales + 64 BF16 k_pe.
ROW_BYTES_E4M3 = KV_LORA + QK_ROPE  # 576
DS_SCALES = KV_LORA  # byte offset of the four FP32 scales
DS_ROPE = KV_LORA + 4 * (KV_LORA // DS_TILE)  # 528: byte offset of BF16 k_pe
ROW_BYTES_DS = DS_ROPE + 2 * QK_ROPE  # 656

E4M3_MAX = 448.0

# ``nvfp4_ds_mla`` row: 512 E2M1 values packed two to a byte, one E4M3 scale
# per 16-value block, then the 64 k_pe values as E4M3.  The offsets are not
# printed on the page; reading taken: the three parts packed in that order.
NVFP4_BLOCK = 16
NVFP4_SCALES = KV_LORA // 2  # 256: byte offset of the 32 block scales
NVFP4_ROPE = NVFP4_SCALES + KV_LORA // NVFP4_BLOCK  # 288: byte offset of E4M3 k_pe
ROW_BYTES_NVFP4 = NVFP4_ROPE + QK_ROPE  # 352

# The fused row q_a | kv_c | k_pe that the path reads, and the hidden width
# of the down-projection producing it.
QKV_ROW = Q_LORA + KV_LORA + QK_ROPE  # 2112
HIDDEN = 7168
E2M1_MAX = 6.0
NVFP4_SCALE_FLOOR = 2.0**-9  # the smallest positive E4M3 value

# Relative width of the rounding tie zone of the normalised q_a row: a bound
# on the FP32 evaluation error of x * rr * gamma over every way the row is
# computed.  The sum of squares has positive terms, so a sum whose longest
# path from a term to the result passes d roundings is within d * 2**-24 of
# its value.  The longest such path: a 48-term FMA chain per lane (6 chunks of
# 8 values), 2 shuffle additions over a lane quad, 7 additions over the 8
# warps: d = 57.  Then the division by 1536 and the eps addition (2 more),
# halved by the square root, plus the reciprocal square root and the two
# products: (57 + 2) / 2 + 3 = 32.5 roundings of 2**-24.  33 * 2**-24 covers
# it (second-order terms are below 2**-40).
XQ_TIE_REL = 33 * 2.0**-24

LAYOUT_E4M3 = 0
LAYOUT_DS_MLA = 1
LAYOUT_NVFP4_DS_MLA = 2
ROW_BYTES = {LAYOUT_E4M3: ROW_BYTES_E4M3, LAYOUT_DS_MLA: ROW_BYTES_DS,
             LAYOUT_NVFP4_DS_MLA: ROW_BYTES_NVFP4}


# ---------------------------------------------------------------------------
# Number formats (written from the format definitions, not from any library).
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values.

    bfloat16 is the upper half of an IEEE binary32, so widening is exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # NaN patterns widen to NaN
        return b.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16: 8 significant bits, exponent range of binary32 (normal minimum
    2**-126, subnormal quantum 2**-133).  A value with ``x = m * 2**e`` and
    ``0.5 <= |m| < 1`` has quantum ``2**(e - 8)`` when normal.  The result is
    returned as float64 (exactly representable in bfloat16).  Values beyond the
    largest finite bfloat16 after rounding become infinities."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q_exp = np.maximum(e - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(x, -q_exp)), q_exp)
    bf16_max = (2.0 - 2.0**-7) * 2.0**127
    return np.where(np.abs(r) > bf16_max, np.copysign(np.inf, x), r)


def bf16_quantum(x) -> np.ndarray:
    """Spacing of the bfloat16 values around each float64 value (2**(e-8),
    2**-133 below the normal range)."""
    _, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def bf16_midpoint_distance(x) -> np.ndarray:
    """Distance from each value to the nearest midpoint between two adjacent
    bfloat16 values (0 at a tie of round-to-nearest)."""
    x = np.asarray(x, dtype=np.float64)
    q = bf16_quantum(x)
    frac = np.abs(x) / q - np.floor(np.abs(x) / q)
    return np.abs(frac - 0.5) * q


def bf16_other_rounding(x) -> np.ndarray:
    """The bfloat16 neighbour of each value that round-to-nearest does not
    pick (the other side of the value; equal to x when x is representable)."""
    x = np.asarray(x, dtype=np.float64)
    q = bf16_quantum(x)
    lo = np.floor(x / q) * q
    hi = np.ceil(x / q) * q
    r = round_to_bf16(x)
    return np.where(r == hi, lo, hi)


def f64_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (uint16), round to nearest even."""
    r = round_to_bf16(x).astype(np.float32)  # exact: r fits in binary32
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_to_f32(x) -> np.ndarray:
    """float64 -> nearest binary32 (ties to even), returned as float64.

    A library conversion (numpy's cast is IEEE round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def e4m3_satfinite(v) -> np.ndarray:
    """float64 -> OCP FP8 E4M3 byte, round to nearest even, saturating.

    E4M3 (the "fn" variant): sign, 4 exponent bits with bias 7, 3 mantissa bits;
    normal values (1 + m/8) * 2**(E - 7) for E = 1..15 except E=15, m=7, which
    is NaN, so the largest finite magnitude is 448; subnormals (m/8) * 2**-6.
    Reading taken: the cast saturates to +-448 instead of producing NaN (the
    page states FP8 bytes are never 0xFF), and the sign of a zero is kept."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3_satfinite: non-finite input")
    _, e = np.frexp(v)
    q_exp = np.maximum(e - 4, -9)  # 4 significant bits; subnormal quantum 2**-9
    r = np.ldexp(np.rint(np.ldexp(v, -q_exp)), q_exp)
    r = np.clip(r, -E4M3_MAX, E4M3_MAX)
    sign = np.signbit(r).astype(np.uint8) << np.uint8(7)
    a = np.abs(r)
    normal = a >= 2.0**-6
    m2, e2 = np.frexp(np.where(normal, a, 1.0))  # a = m2 * 2**e2, m2 in [0.5, 1)
    exp_field = np.where(normal, e2 - 1 + 7, 0)
    mant_normal = np.rint((m2 * 2.0 - 1.0) * 8.0)
    mant_sub = np.rint(a / 2.0**-9)
    mant = np.where(normal, mant_normal, mant_sub)
    code = (exp_field.astype(np.int64) << 3) | mant.astype(np.int64)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_to_f64(codes) -> np.ndarray:
    """OCP FP8 E4M3 byte -> float64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(E == 0, m / 8.0 * 2.0**-6, (1.0 + m / 8.0) * np.ldexp(1.0, E - 7))
    val = np.where((E == 15) & (m == 7), np.nan, val)
    return s * val


def e2m1_satfinite(v) -> np.ndarray:
    """float64 -> OCP FP4 E2M1 code (uint8, low 4 bits), round to nearest even,
    saturating.

    E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit; normal values
    (1 + m/2) * 2**(E - 1) for E = 1..3 (1, 1.5, 2, 3, 4, 6), subnormals
    (m/2) for E = 0 (0, 0.5); no infinities or NaN, so the largest magnitude
    is 6.  Reading taken: the cast saturates to +-6 and keeps the sign of a
    zero, as the E4M3 cast does."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e2m1_satfinite: non-finite input")
    _, e = np.frexp(v)
    q_exp = np.maximum(e - 2, -1)  # 2 significant bits; subnormal quantum 2**-1
    r = np.ldexp(np.rint(np.ldexp(v, -q_exp)), q_exp)
    r = np.clip(r, -E2M1_MAX, E2M1_MAX)
    sign = np.signbit(r).astype(np.uint8) << np.uint8(3)
    a = np.abs(r)
    normal = a >= 1.0
    m2, e2 = np.frexp(np.where(normal, a, 1.0))  # a = m2 * 2**e2, m2 in [0.5, 1)
    exp_field = np.where(normal, e2 - 1 + 1, 0)
    mant = np.where(normal, np.rint((m2 * 2.0 - 1.0) * 2.0), np.rint(a / 0.5))
    code = (exp_field.astype(np.int64) << 1) | mant.astype(np.int64)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e2m1_to_f64(codes) -> np.ndarray:
    """OCP FP4 E2M1 code (low 4 bits) -> float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    s = np.where(c & 0x8, -1.0, 1.0)
    E = (c >> 1) & 0x3
    m = c & 0x1
    return s * np.where(E == 0, m * 0.5, (1.0 + m / 2.0) * np.ldexp(1.0, E - 1))


def pow2_ceil(v) -> np.ndarray:
    """exp2(ceil(log2(v))) of positive normal binary32 values (function
    ``pow2_ceil`` on the page "mla.query"), computed from its definition:
    with ``v = m * 2**e`` and ``0.5 <= m < 1`` the result is ``v`` itself when
    ``m == 0.5`` (v is a power of two) and ``2**e`` otherwise."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(~(v > 0)):
        raise ValueError("pow2_ceil: needs positive values")
    m, e = np.frexp(v)
    return np.where(m == 0.5, v, np.ldexp(1.0, e))


def f32_bits(v) -> np.ndarray:
    """binary32 bit pattern (uint32) of float64 values exactly representable."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32)


# ---------------------------------------------------------------------------
# The steps of the path.
# ---------------------------------------------------------------------------


def rmsnorm(x, gamma, eps):
    """RMS normalisation of each row of ``x`` (float64 [..., n]) times ``gamma``.

    ``rr = 1 / sqrt(sum(x**2) / n + eps)``, output ``x * rr * gamma``, all in
    float64 and not rounded here.  Page "mla.query", ``kernel`` (q_a, n=1536)
    and ``insert`` (kv_c, n=512).  Reading taken for q_a, whose norm helper is
    not printed: the same form as the printed kv_c norm (mean of squares plus
    eps, reciprocal square root, then x * rr * gamma)."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    ss = np.sum(x * x, axis=-1, keepdims=True)
    rr = 1.0 / np.sqrt(ss / n + float(eps))
    return x * rr * np.asarray(gamma, dtype=np.float64)


def q_projection(xq, w_qb, heads):
    """Q_B projection: ``q[b, h, p] = sum_k xq[b, k] * W_QB[h*192 + p, k]``.

    ``xq`` float64 [B, 1536] (BF16 values), ``w_qb`` float64 [H*192, 1536].
    Returns (exact float64 sums [B, H, 192], sums of |terms| [B, H, 192]).
    Page "mla.query", ``kernel``: the Q_B slice of a head starts at row
    ``head * 192``; row p < 128 is nope, p >= 128 rope."""
    B = xq.shape[0]
    q = xq @ w_qb.T
    cond = np.abs(xq) @ np.abs(w_qb).T
    return q.reshape(B, heads, QK_HEAD), cond.reshape(B, heads, QK_HEAD)


def absorb(q_nope, w_uk):
    """W_UK absorption: ``out[b, h, c] = sum_p q_nope[b, h, p] * W_UK[h, p, c]``.

    ``q_nope`` float64 [B, H, 128] (BF16-rounded Q_B values), ``w_uk`` float64
    [H, 128, 512].  Returns (exact sums [B, H, 512], sums of |terms|).
    Page "mla.query", ``kernel``: the absorption reads the BF16-rounded q rows
    and ``uk[p, latent_col]`` from ``w_uk[head, p, column]``."""
    lat = np.einsum("bhp,hpc->bhc", q_nope, w_uk)
    cond = np.einsum("bhp,hpc->bhc", np.abs(q_nope), np.abs(w_uk))
    return lat, cond


def kv_row_e4m3(normed_bf16, k_pe, k_scale):
    """Per-tensor FP8 row (576 bytes): page "mla.query", ``insert`` and
    ``kv_fp8``.  Each BF16 normed value, then each raw k_pe value, is divided by
    ``k_scale`` (the quotient rounded to binary32, as a binary32 division does)
    and cast to E4M3 with saturation.  Reading taken: division, not
    multiplication by the reciprocal (the page keeps both; the division is the
    form ``concat_and_cache_mla`` uses)."""
    ks = float(np.float32(k_scale))
    row = np.empty(ROW_BYTES_E4M3, dtype=np.uint8)
    row[:KV_LORA] = e4m3_satfinite(round_to_f32(normed_bf16 / ks))
    row[KV_LORA:] = e4m3_satfinite(round_to_f32(k_pe / ks))
    return row


def query_fp8(bf16_bits, q_scale_inv) -> np.ndarray:
    """Per-tensor FP8 query element (page "mla.query", method ``kernel``, the
    FP8 query epilogue of the per-tensor cache): the BF16-rounded output value
    times ``q_scale_inv``, the product rounded to binary32 (a binary32
    multiplication; the float64 product of a BF16 and a binary32 value is
    exact), then cast to E4M3 with saturation."""
    qsi = float(np.float32(q_scale_inv))
    return e4m3_satfinite(round_to_f32(bf16_bits_to_f64(bf16_bits) * qsi))


def ds_tile_scale(amax):
    """Scale of one 128-column tile of the ``fp8_ds_mla`` row: the binary32
    quotient ``amax / 448``, floored at binary32 1e-4, then ``pow2_ceil``.
    Page "mla.query", ``insert_ds`` docstring and ``pow2_ceil``."""
    r = round_to_f32(np.asarray(amax, dtype=np.float64) / E4M3_MAX)
    floor = float(np.float32(1e-4))
    return pow2_ceil(np.maximum(r, floor))


def kv_row_ds(normed_bf16, k_pe_bits):
    """``fp8_ds_mla`` row (656 bytes): page "mla.query", ``insert_ds``.

    Bytes 0..511: E4M3 of ``n * (1 / s_t)`` for tile t = column // 128 (exact:
    s_t is a power of two); bytes 512..527: the four scales as binary32,
    little-endian; bytes 528..655: k_pe copied as raw BF16, little-endian.
    Readings taken: the scale and k_pe offsets (not printed) are the packed
    order above, which gives the 656-byte row; amax is taken over the
    BF16-rounded normed values, as the page does."""
    row = np.empty(ROW_BYTES_DS, dtype=np.uint8)
    n = np.asarray(normed_bf16, dtype=np.float64)
    scales = np.empty(KV_LORA // DS_TILE, dtype=np.float64)
    for t in range(KV_LORA // DS_TILE):
        seg = n[t * DS_TILE:(t + 1) * DS_TILE]
        s = float(ds_tile_scale(np.max(np.abs(seg))))
        scales[t] = s
        row[t * DS_TILE:(t + 1) * DS_TILE] = e4m3_satfinite(seg / s)
    row[DS_SCALES:DS_ROPE] = f32_bits(scales).astype("<u4").view(np.uint8)
    row[DS_ROPE:] = np.asarray(k_pe_bits, dtype="<u2").view(np.uint8)
    return row, scales


def nvfp4_block_scale(amax):
    """E4M3 scale of one 16-value block of the ``nvfp4_ds_mla`` row (page
    "mla.query", ``insert_nvfp4``): ``sf = max(amax / 6, 2**-9)`` with the
    binary32 quotient, cast to E4M3.  Returns (E4M3 code, its value, the
    binary32 reciprocal of that value).  Reading taken: the values are scaled
    by the reciprocal of the stored (E4M3-rounded) scale, so that code times
    scale is what a reader of the row decodes."""
    sf = np.maximum(round_to_f32(np.asarray(amax, dtype=np.float64) / E2M1_MAX),
                    NVFP4_SCALE_FLOOR)
    code = e4m3_satfinite(sf)
    value = e4m3_to_f64(code)
    return code, value, round_to_f32(1.0 / value)


def nvfp4_scale_byte(block):
    """Byte offset, within the row, of the scale of 16-value block ``block``
    (0..31): the page stores the scales four-way interleaved, block s at
    ``NVFP4_SCALES + 8 * (s % 4) + s // 4``."""
    return NVFP4_SCALES + 8 * (block % 4) + block // 4


def kv_row_nvfp4(normed_bf16, k_pe):
    """``nvfp4_ds_mla`` row (352 bytes): page "mla.query", ``insert_nvfp4``.

    Each 16-value block of the BF16 normed latent row gets an E4M3 scale
    (nvfp4_block_scale over the block's amax) and its values are stored as
    E2M1 of the binary32 product ``n * (1 / sf)``; k_pe is stored as E4M3 of
    its BF16 value, with no scale.  Bytes 0..255: E2M1 codes, value 2k in the
    low half of byte k and value 2k + 1 in the high half (reading taken: the
    page's packing helper is not printed; this is the order of the FP4 formats
    that hold two values per byte).  Bytes 256..287: the 32 scales, placed by
    nvfp4_scale_byte.  Bytes 288..351: k_pe."""
    n = np.asarray(normed_bf16, dtype=np.float64)
    row = np.empty(ROW_BYTES_NVFP4, dtype=np.uint8)
    codes = np.empty(KV_LORA, dtype=np.uint8)
    scales = np.empty(KV_LORA // NVFP4_BLOCK, dtype=np.float64)
    for s in range(KV_LORA // NVFP4_BLOCK):
        seg = n[s * NVFP4_BLOCK:(s + 1) * NVFP4_BLOCK]
        code, value, inv = nvfp4_block_scale(np.max(np.abs(seg)))
        scales[s] = value
        row[nvfp4_scale_byte(s)] = code
        codes[s * NVFP4_BLOCK:(s + 1) * NVFP4_BLOCK] = e2m1_satfinite(round_to_f32(seg * inv))
    row[:NVFP4_SCALES] = codes[0::2] | (codes[1::2] << np.uint8(4))
    row[NVFP4_ROPE:] = e4m3_satfinite(np.asarray(k_pe, dtype=np.float64))
    return row, scales


def qkv_a_projection(x_bits, w_bits):
    """The down-projection that produces the fused qkv row the path reads:
    ``y[b, n] = bf16(sum_k x[b, k] * W[n, k])`` (page "ws_gemm", class
    ``WsGemm``: ``y[M, N] = x[M, K] @ W[N, K]^T`` with BF16 operands, FP32
    accumulation and BF16 outputs).  With W = the stacked q_a / kv_a
    projections [2112, 7168], row b of y is the ``qkv`` row of page
    "mla.query" (``kernel``): q_a at columns 0..1535, kv_c at 1536..2047,
    k_pe at 2048..2111.

    ``x_bits`` uint16 BF16 [B, K], ``w_bits`` uint16 BF16 [N, K].  Returns
    (BF16 bits of y [B, N], exact float64 sums, sums of |terms|)."""
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_bits)
    exact = x @ w.T
    cond = np.abs(x) @ np.abs(w).T
    return f64_to_bf16_bits(exact), exact, cond


def slot_to_page(slot, page_size):
    """Paged-cache address of a slot: ``(slot // page_size, slot % page_size)``
    (page "mla.query", ``insert``).  Only called for slot >= 0."""
    return int(slot) // int(page_size), int(slot) % int(page_size)


def decode_step(inp, xq_alt=None):
    """One decode step of the whole path.

    ``inp`` is a dict with BF16 bit arrays ``w_qb [H*192, 1536]``,
    ``w_uk [H, 128, 512]``, ``gamma_q [1536]``, ``gamma_kv [512]``,
    ``q_a [B, 1536]``, ``kv_c [B, 512]``, ``k_pe [B, 64]``; ``slots`` int64 [B];
    ``cache`` uint8 [pages, page_size, row_bytes] (not modified); ``layout``
    (0 per-tensor E4M3, 1 fp8_ds_mla, 2 nvfp4_ds_mla); float ``k_scale`` and
    ``eps``.

    Returns a dict: BF16 bits ``q_c [B, 1536]``, ``q_pe [B, H, 64]``,
    ``q_latent [B, H, 512]`` (with a ``q_scale_inv`` entry in ``inp``, also
    the FP8 query outputs ``q_latent_fp8`` and ``q_pe_fp8``, see query_fp8);
    the updated ``cache``; float64 exact
    pre-rounding values and |term| sums for tolerance floors; ``bad_slots``
    (slots at or beyond the cache capacity, skipped).

    ``xq_alt`` (bool [B, 1536], optional) selects, for the marked elements of
    the normalised q_a row, the other correct BF16 rounding: an element whose
    exact value lies at a rounding midpoint to within the FP32 evaluation
    error has two correct roundings (FP32 arithmetic, as the page computes it,
    may land on either side).  Marked elements must lie within XQ_TIE_REL of
    their value from a midpoint; the rest of the step follows from the chosen
    rounding."""
    H = inp["w_uk"].shape[0]
    eps = float(np.float32(inp["eps"]))
    w_qb = bf16_bits_to_f64(inp["w_qb"])
    w_uk = bf16_bits_to_f64(inp["w_uk"])
    g_q = bf16_bits_to_f64(inp["gamma_q"])
    g_kv = bf16_bits_to_f64(inp["gamma_kv"])
    q_a = bf16_bits_to_f64(inp["q_a"])
    kv_c = bf16_bits_to_f64(inp["kv_c"])
    k_pe_bits = np.asarray(inp["k_pe"], dtype=np.uint16)
    k_pe = bf16_bits_to_f64(k_pe_bits)

    # q_a RMSNorm, one BF16 rounding; the rounded row is q_c and the GEMM input.
    xq_exact = rmsnorm(q_a, g_q, eps)
    xq = round_to_bf16(xq_exact)
    if xq_alt is not None:
        xq_alt = np.asarray(xq_alt, dtype=bool)
        near = bf16_midpoint_distance(xq_exact) <= XQ_TIE_REL * np.abs(xq_exact)
        if np.any(xq_alt & ~near):
            raise ValueError("xq_alt marks an element outside the rounding tie zone")
        xq = np.where(xq_alt, bf16_other_rounding(xq_exact), xq)
    # Q_B projection, one BF16 rounding per output.
    q_exact, q_cond = q_projection(xq, w_qb, H)
    q = round_to_bf16(q_exact)
    # rope part is emitted as is; nope part is absorbed through W_UK.
    q_pe = q[:, :, QK_NOPE:]
    lat_exact, lat_cond = absorb(q[:, :, :QK_NOPE], w_uk)
    q_latent = round_to_bf16(lat_exact)

    # KV: RMSNorm of kv_c (BF16), then the cache row of the chosen layout.
    normed = round_to_bf16(rmsnorm(kv_c, g_kv, eps))
    cache = np.array(inp["cache"], dtype=np.uint8, copy=True)
    pages, page_size, row_bytes = cache.shape
    layout = int(inp["layout"])
    if layout not in ROW_BYTES:
        raise ValueError(f"unknown cache layout {layout}")
    want = ROW_BYTES[layout]
    if row_bytes != want:
        raise ValueError(f"cache rows are {row_bytes} B, layout needs {want}")
    bad = []
    ds_scales = {}
    for b, slot in enumerate(np.asarray(inp["slots"], dtype=np.int64)):
        if slot < 0:
            continue
        page, off = slot_to_page(slot, page_size)
        if page >= pages:
            bad.append(b)
            continue
        if layout == LAYOUT_DS_MLA:
            row, sc = kv_row_ds(normed[b], k_pe_bits[b])
            ds_scales[b] = sc
        elif layout == LAYOUT_NVFP4_DS_MLA:
            row, sc = kv_row_nvfp4(normed[b], k_pe[b])
            ds_scales[b] = sc
        else:
            row = kv_row_e4m3(normed[b], k_pe[b], inp["k_scale"])
        cache[page, off, :] = row

    out = {
        "q_c": f64_to_bf16_bits(xq),
        "q_pe": f64_to_bf16_bits(q_pe),
        "q_latent": f64_to_bf16_bits(q_latent),
        "cache": cache,
        "q_exact": q_exact,
        "q_cond": q_cond,
        "lat_exact": lat_exact,
        "lat_cond": lat_cond,
        "xq_exact": xq_exact,
        "kv_normed": normed,
        "ds_scales": ds_scales,
        "bad_slots": bad,
    }
    # FP8 query outputs (a ``q_scale_inv`` entry in ``inp`` asks for them)
    if "q_scale_inv" in inp:
        out["q_latent_fp8"] = query_fp8(out["q_latent"], inp["q_scale_inv"])
        out["q_pe_fp8"] = query_fp8(out["q_pe"], inp["q_scale_inv"])
    return out
