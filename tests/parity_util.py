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
"""

from __future__ import annotations

import numpy as np

from oracle import mla_oracle as O

ULP_REL = 2.0**-7
MAX_REL = 1e-2
FRAC_WITHIN_ULP = 0.999
FRAC_FP8_EXACT = 0.999


def check_bf16(name, got_bits, ref_bits, cond=None, k_terms=0, report=None):
    g = O.bf16_bits_to_f64(got_bits)
    r = O.bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite GPU output"
    err = np.abs(g - r)
    if cond is None:
        cond = np.zeros_like(r)
    tol = ULP_REL * np.abs(r) + k_terms * 2.0**-24 * cond
    within = err <= tol
    denom = np.maximum(np.abs(r), cond)
    denom = np.where(denom == 0, 1.0, denom)
    rel = err / denom
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
               report=report)
    check_cache(gpu["cache"], ref["cache"], inp["cache"], inp["slots"], inp["cache"].shape[1],
                int(inp["layout"]), report=report)
