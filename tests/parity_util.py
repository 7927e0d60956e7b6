"""Comparison of the CUDA path's outputs with the FP64 oracle's.

Tolerances (the acceptance bar of the MLA query path), with r the oracle's
BF16-rounded value, g the GPU's, and S = sum_i |a_i * b_i| the magnitude of the
terms of the dot product that produced the output (K terms):
  * BF16 outputs (q_c, q_pe, q_latent): at least 99.9% of elements within one
    BF16 ulp, i.e. |g - r| <= 2**-7 * |r| + K * 2**-24 * S.  The second term is
    the worst-case error bound of a K-term FP32 summation (Higham's gamma_K
    times S); without it, outputs whose dot product cancels to almost zero fail
    on rounding error alone (observed: q_pe = -1.39e-5 from terms summing to
    ~20 in magnitude).
  * Everywhere: |g - r| <= 1e-2 * max(|r|, S).  Relative error of a cancelling
    dot product is judged against the size of its terms: the absorption reads
    BF16-rounded q values, and one q value rounded to the other side of a tie
    (legitimate for any FP32 accumulation order) moves an output by up to one
    BF16 ulp of that single term, 6.2e-2 of 2**-8 * S in one observed case.
  * FP8 cache bytes: at least 99.9% identical; the rest within one E4M3 code
    (codes compared as signed ordinals, so +0 and -0 are equal).
  * fp8_ds_mla power-of-two scales, k_pe bytes, slot/page placement and every
    cache byte outside the written rows: bit-exact.
  * nvfp4_ds_mla rows: E4M3 block scales and E4M3 k_pe bit-exact; E2M1 codes
    at least 99.9% identical, the rest within one code.

Rounding ties.  The path rounds FP32 intermediates to BF16 where the page
does (the normalised q_a row, the Q_B outputs).  When an exact value lies at a
rounding midpoint to within the FP32 evaluation error, both neighbours are
correct results, and the choice moves everything downstream of it:
  * q_c: every element must equal the oracle's rounding, or lie in the tie
    zone (within 2**-20 of its value from a midpoint) and take the other
    rounding; the oracle then computes the rest of the step for the rounding
    the GPU took (``reference_for``).  Observed on GB300: q_c element -0.95117186
    (1.5e-8 from the midpoint) rounded the other way moved ~6% of that token's
    q_latent outputs by more than one ulp.
  * q_latent: Q_B outputs whose exact value lies within 2**-22 * S of a
    midpoint may round either way; each such q value widens the tolerance of
    the outputs it feeds by one BF16 quantum of q times |W_UK[h, p, c]|.
"""

from __future__ import annotations

import numpy as np

from oracle import mla_oracle as O

ULP_REL = 2.0**-7
MAX_REL = 1e-2
FRAC_WITHIN_ULP = 0.999
FRAC_FP8_EXACT = 0.999


Q_TIE_REL_S = 2.0**-22


def reference_for(inp, gpu_q_c=None):
    """The oracle's step for the inputs; if the GPU's q_c takes the other
    correct rounding of tie-zone elements, the oracle's step for that rounding."""
    ref = O.decode_step(inp)
    if gpu_q_c is None:
        return ref
    mism = np.asarray(gpu_q_c) != ref["q_c"]
    if not mism.any():
        return ref
    near = O.bf16_midpoint_distance(ref["xq_exact"]) <= O.XQ_TIE_REL * np.abs(ref["xq_exact"])
    bad = mism & ~near
    assert not bad.any(), f"q_c differs outside the rounding tie zone at {np.argwhere(bad)[:5]}"
    alt = O.decode_step(inp, xq_alt=mism)
    assert np.array_equal(alt["q_c"], gpu_q_c), "q_c is neither rounding of a tie-zone element"
    return alt


def latent_slack(ref, inp):
    """Tolerance added to q_latent for Q_B outputs whose rounding may go
    either way (see the module docstring)."""
    q_exact = ref["q_exact"][:, :, :128]
    cond = ref["q_cond"][:, :, :128]
    amb = O.bf16_midpoint_distance(q_exact) <= Q_TIE_REL_S * cond
    step = np.where(amb, O.bf16_quantum(q_exact), 0.0)
    w_uk = np.abs(O.bf16_bits_to_f64(inp["w_uk"]))
    return np.einsum("bhp,hpc->bhc", step, w_uk)


def check_bf16(name, got_bits, ref_bits, cond=None, k_terms=0, report=None, slack=None):
    g = O.bf16_bits_to_f64(got_bits)
    r = O.bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite GPU output"
    err = np.abs(g - r)
    if cond is None:
        cond = np.zeros_like(r)
    if slack is None:
        slack = 0.0
    tol = ULP_REL * np.abs(r) + k_terms * 2.0**-24 * cond + slack
    within = err <= tol
    denom = np.maximum(np.abs(r), cond)
    denom = np.where(denom == 0, 1.0, denom)
    rel = np.maximum(err - slack, 0.0) / denom
    frac = float(np.mean(within)) if within.size else 1.0
    if report is not None:
        report[name] = dict(
            within_tol=frac,
            within_plain_ulp=float(np.mean(err <= ULP_REL * np.abs(r))) if r.size else 1.0,
            bit_exact=float(np.mean(got_bits == ref_bits)) if r.size else 1.0,
            max_rel=float(rel.max(initial=0.0)),
        )
    assert frac >= FRAC_WITHIN_ULP, f"{name}: only {frac:.5f} within 1 BF16 ulp"
    assert rel.max(initial=0.0) <= MAX_REL, f"{name}: max rel {rel.max():.3e}"


def e4m3_ordinal(codes):
    c = codes.astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def e2m1_ordinal(codes):
    c = codes.astype(np.int64)
    mag = c & 0x7
    return np.where(c & 0x8, -mag, mag)


def check_cache(got, ref, before, slots, page_size, layout, report=None):
    """Compare the whole cache: written rows by tolerance, everything else exact."""
    assert got.shape == ref.shape
    pages = got.shape[0]
    written = np.zeros(got.shape[:2], dtype=bool)
    for s in np.asarray(slots, dtype=np.int64):
        if s >= 0 and s // page_size < pages:
            written[s // page_size, s % page_size] = True
    assert np.array_equal(got[~written], before[~written]), "bytes outside written rows changed"
    assert np.array_equal(ref[~written], before[~written])
    if not written.any():
        return
    g, r = got[written], ref[written]
    if layout == O.LAYOUT_NVFP4_DS_MLA:
        assert np.array_equal(g[:, O.NVFP4_SCALES:], r[:, O.NVFP4_SCALES:]), \
            "nvfp4 block scales / k_pe differ"
        gv, rv = g[:, :O.NVFP4_SCALES], r[:, :O.NVFP4_SCALES]
        gc = np.concatenate([gv & 0xF, gv >> 4], axis=1)
        rc = np.concatenate([rv & 0xF, rv >> 4], axis=1)
        frac = float(np.mean(gc == rc))
        dist = np.abs(e2m1_ordinal(gc) - e2m1_ordinal(rc))
        if report is not None:
            report["cache_fp4_exact"] = frac
            report["cache_fp4_max_code_dist"] = int(dist.max(initial=0))
        assert frac >= FRAC_FP8_EXACT, f"only {frac:.5f} of E2M1 codes identical"
        assert dist.max(initial=0) <= 1, f"E2M1 codes up to {dist.max()} apart"
        return
    if layout == O.LAYOUT_DS_MLA:
        assert np.array_equal(g[:, O.DS_SCALES:], r[:, O.DS_SCALES:]), "ds scales / k_pe differ"
        g, r = g[:, :O.DS_SCALES], r[:, :O.DS_SCALES]
    same = g == r
    frac = float(np.mean(same))
    dist = np.abs(e4m3_ordinal(g) - e4m3_ordinal(r))
    if report is not None:
        report["cache_fp8_exact"] = frac
        report["cache_fp8_max_code_dist"] = int(dist.max(initial=0))
    assert frac >= FRAC_FP8_EXACT, f"only {frac:.5f} of FP8 bytes identical"
    assert dist.max(initial=0) <= 1, f"FP8 bytes up to {dist.max()} codes apart"


def check_step(gpu: dict, ref: dict, inp: dict, report=None, q_c=True):
    if q_c:
        check_bf16("q_c", gpu["q_c"], ref["q_c"], report=report)
    check_bf16("q_pe", gpu["q_pe"], ref["q_pe"], ref["q_cond"][:, :, 128:], k_terms=1536,
               report=report)
    check_bf16("q_latent", gpu["q_latent"], ref["q_latent"], ref["lat_cond"], k_terms=128,
               report=report, slack=latent_slack(ref, inp))
    check_cache(gpu["cache"], ref["cache"], inp["cache"], inp["slots"], inp["cache"].shape[1],
                int(inp["layout"]), report=report)


def check_against_oracle(gpu: dict, inp: dict, report=None, q_c=True, dump_name=None):
    """Oracle reference (tie-aware) and every check; on failure, saves the GPU
    outputs under $MLA_PARITY_DUMP (if set) for offline analysis."""
    import os

    ref = reference_for(inp, gpu.get("q_c") if q_c else None)
    try:
        check_step(gpu, ref, inp, report=report, q_c=q_c)
    except AssertionError:
        d = os.environ.get("MLA_PARITY_DUMP")
        if d and dump_name:
            os.makedirs(d, exist_ok=True)
            np.savez_compressed(os.path.join(d, f"{dump_name}.npz"),
                                **{k: v for k, v in gpu.items() if k != "cache"})
        raise
    return ref
