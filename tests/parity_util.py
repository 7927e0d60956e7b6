"""Comparison of the CUDA path's outputs with the FP64 oracle's.

Tolerances (the acceptance bar of the MLA query path):
  * BF16 outputs (q_c, q_pe, q_latent): at least 99.9% of elements within one
    BF16 ulp, measured as a relative error of 2**-7 against the oracle's
    BF16-rounded value, and relative error at most 1e-2 everywhere, where the
    denominator is max(|ref|, 2**-8 * sum|terms|) so that outputs whose dot
    product cancels to near zero are judged against the size of their terms.
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


def check_bf16(name, got_bits, ref_bits, cond=None, report=None):
    g = O.bf16_bits_to_f64(got_bits)
    r = O.bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite GPU output"
    err = np.abs(g - r)
    within = err <= ULP_REL * np.abs(r)
    denom = np.abs(r)
    if cond is not None:
        denom = np.maximum(denom, 2.0**-8 * cond)
    denom = np.where(denom == 0, 1.0, denom)
    rel = err / denom
    frac = float(np.mean(within)) if within.size else 1.0
    exact = float(np.mean(got_bits == ref_bits)) if within.size else 1.0
    if report is not None:
        report[name] = dict(within_ulp=frac, bit_exact=exact, max_rel=float(rel.max(initial=0.0)))
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
    check_bf16("q_pe", gpu["q_pe"], ref["q_pe"], ref["q_cond"][:, :, 128:], report=report)
    check_bf16("q_latent", gpu["q_latent"], ref["q_latent"], ref["lat_cond"], report=report)
    check_cache(gpu["cache"], ref["cache"], inp["cache"], inp["slots"], inp["cache"].shape[1],
                int(inp["layout"]), report=report)
