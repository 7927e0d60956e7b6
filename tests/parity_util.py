"""Comparison of the CUDA path's outputs with the FP64 oracle's.

The acceptance bar of the MLA query path, with r the oracle's BF16-rounded
value, g the GPU's, and S = sum_i |a_i * b_i| the magnitude of the terms of the
dot product that produced the output:
  * BF16 outputs (q_c, q_pe, q_latent): at least 99.9% of elements within one
    BF16 ulp, i.e. |g - r| <= 2**-7 * |r| (nothing added to it), and
  * everywhere: |g - r| <= 1e-2 * max(|r|, 2**-8 * S).  The floor keeps the
    relative error of a dot product that cancels to almost zero from being
    judged against that near-zero value alone.
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
  * q_c is an output, so the choice is seen: every element must equal the
    oracle's rounding, or lie in the tie zone (oracle.XQ_TIE_REL, a bound on
    the FP32 evaluation error of the kernels' normalisation) and take the
    other rounding; the oracle then computes the rest of the step for the
    rounding the GPU took (``reference_for``).  Every such element is counted
    in the report and in the session summary.
  * the nope Q_B values are not outputs.  Those whose exact value lies within
    Q_TIE_REL_S * S of a midpoint may round either way; each widens, in the
    1e-2 check only, the tolerance of the q_latent outputs it feeds by one BF16
    quantum of q times |W_UK[h, p, c]| (``latent_slack``).  The 1-ulp check
    takes no slack.
"""

from __future__ import annotations

import numpy as np

from oracle import mla_oracle as O

ULP_REL = 2.0**-7
MAX_REL = 1e-2
FLOOR_REL_S = 2.0**-8
FRAC_WITHIN_ULP = 0.999
FRAC_FP8_EXACT = 0.999

# Width of the ambiguous zone of a Q_B value, relative to S = sum |xq * w|.
# The kernels' FP32 sums of 1536 products round at most about 50 times along
# any path from a product to the result (the longest: 48 tcgen05 k16 steps
# accumulating one K half in TMEM, then the halves added), each time by at
# most 2**-24 of a partial sum.  The products have random signs, so partial
# sums stay near |q| ~ sqrt(1536) * |term|, about 1/40 of S, and the
# accumulated error (a random walk over those roundings) is about
# sqrt(50) * 2**-24 * S / 40 ~ 2**-26 * S.  2**-22 * S is 16 times that.
Q_TIE_REL_S = 2.0**-22

# Counts over the whole test session (printed by tests/conftest.py).
SESSION = {"steps_checked": 0, "q_c_ties_taken": 0, "steps_with_q_c_tie": 0,
           "q_ambiguous": 0, "q_latent_elems": 0, "q_latent_plain_fails": 0,
           "q_pe_plain_fails": 0, "q_c_plain_fails": 0, "worst_plain_frac": 1.0}


def reference_for(inp, gpu_q_c=None, report=None):
    """The oracle's step for the inputs; if the GPU's q_c takes the other
    correct rounding of tie-zone elements, the oracle's step for that rounding.
    The number of elements it took from the GPU goes to report["q_c_ties_taken"]."""
    ref = O.decode_step(inp)
    taken = 0
    if gpu_q_c is not None:
        mism = np.asarray(gpu_q_c) != ref["q_c"]
        if mism.any():
            near = O.bf16_midpoint_distance(ref["xq_exact"]) <= O.XQ_TIE_REL * np.abs(ref["xq_exact"])
            bad = mism & ~near
            assert not bad.any(), f"q_c differs outside the rounding tie zone at {np.argwhere(bad)[:5]}"
            alt = O.decode_step(inp, xq_alt=mism)
            assert np.array_equal(alt["q_c"], gpu_q_c), "q_c is neither rounding of a tie-zone element"
            ref = alt
            taken = int(mism.sum())
    if report is not None:
        report["q_c_ties_taken"] = taken
    SESSION["q_c_ties_taken"] += taken
    SESSION["steps_with_q_c_tie"] += int(taken > 0)
    return ref


def ambiguous_q(ref):
    """Nope Q_B values whose rounding may go either way (bool [B, H, 128])."""
    q_exact = ref["q_exact"][:, :, :128]
    cond = ref["q_cond"][:, :, :128]
    return O.bf16_midpoint_distance(q_exact) <= Q_TIE_REL_S * cond


def latent_slack(ref, inp):
    """Tolerance added to q_latent in the 1e-2 check for Q_B values whose
    rounding may go either way (see the module docstring)."""
    q_exact = ref["q_exact"][:, :, :128]
    step = np.where(ambiguous_q(ref), O.bf16_quantum(q_exact), 0.0)
    w_uk = np.abs(O.bf16_bits_to_f64(inp["w_uk"]))
    return np.einsum("bhp,hpc->bhc", step, w_uk)


def check_bf16(name, got_bits, ref_bits, cond=None, report=None, slack=None):
    """The BF16 bar on one output: >= 99.9% within 2**-7 |r|, and everywhere
    |g - r| <= 1e-2 max(|r|, 2**-8 S) (``slack`` subtracted first: only the
    ambiguous-rounding allowance of q_latent)."""
    g = O.bf16_bits_to_f64(got_bits)
    r = O.bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite GPU output"
    err = np.abs(g - r)
    if cond is None:
        cond = np.zeros_like(r)
    if slack is None:
        slack = np.zeros_like(r)
    within = err <= ULP_REL * np.abs(r)
    denom = np.maximum(np.abs(r), FLOOR_REL_S * cond)
    excess = np.maximum(err - slack, 0.0)
    # an exact zero reference with no terms (denominator 0) must be met exactly
    rel = np.where(denom > 0, excess / np.where(denom > 0, denom, 1.0),
                   np.where(excess > 0, np.inf, 0.0))
    frac = float(np.mean(within)) if within.size else 1.0
    if report is not None:
        report[name] = dict(
            within_plain_ulp=frac,
            plain_fails=int(np.sum(~within)),
            bit_exact=float(np.mean(got_bits == ref_bits)) if r.size else 1.0,
            max_rel=float(rel.max(initial=0.0)),
            slack_used=int(np.sum((err > ULP_REL * np.abs(r)) & (slack > 0))),
        )
    key = f"{name}_plain_fails"
    if key in SESSION:
        SESSION[key] += int(np.sum(~within))
    SESSION["worst_plain_frac"] = min(SESSION["worst_plain_frac"], frac)
    assert frac >= FRAC_WITHIN_ULP, f"{name}: only {frac:.5f} within 1 BF16 ulp ({int(np.sum(~within))} of {within.size})"
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
    check_bf16("q_pe", gpu["q_pe"], ref["q_pe"], ref["q_cond"][:, :, 128:], report=report)
    amb = ambiguous_q(ref)
    SESSION["q_ambiguous"] += int(amb.sum())
    SESSION["q_latent_elems"] += int(ref["q_latent"].size)
    if report is not None:
        report["q_ambiguous"] = int(amb.sum())
    check_bf16("q_latent", gpu["q_latent"], ref["q_latent"], ref["lat_cond"], report=report,
               slack=latent_slack(ref, inp))
    check_cache(gpu["cache"], ref["cache"], inp["cache"], inp["slots"], inp["cache"].shape[1],
                int(inp["layout"]), report=report)
    SESSION["steps_checked"] += 1


def check_fp8_query(name, got_codes, ref_bits, q_scale_inv, report=None, slack=None):
    """FP8 query outputs against the oracle's own codes (query_fp8 of the
    oracle's BF16 output ``ref_bits``): at least 99.9% identical, and every
    code within one E4M3 code (signed ordinals) of the codes the oracle allows.
    Those are its own code, or for q_latent elements fed by a nope Q_B value
    of ambiguous rounding (``slack``, as in the BF16 check) any code of a BF16
    value in [r - slack, r + slack]: one flipped q value of magnitude ~1.5
    moves q_latent by ~1e-3, two E4M3 quanta near 0.01."""
    got_codes = np.asarray(got_codes, dtype=np.uint8)
    ref_codes = O.query_fp8(ref_bits, q_scale_inv)
    assert got_codes.shape == ref_codes.shape, (name, got_codes.shape, ref_codes.shape)
    same = got_codes == ref_codes
    frac = float(np.mean(same)) if same.size else 1.0
    g = e4m3_ordinal(got_codes)
    lo = hi = e4m3_ordinal(ref_codes)
    if slack is not None:
        r = O.bf16_bits_to_f64(ref_bits)
        a = e4m3_ordinal(O.query_fp8(O.f64_to_bf16_bits(r - slack), q_scale_inv))
        b = e4m3_ordinal(O.query_fp8(O.f64_to_bf16_bits(r + slack), q_scale_inv))
        lo, hi = np.minimum(np.minimum(a, b), lo), np.maximum(np.maximum(a, b), hi)
    dist = np.maximum(0, np.maximum(lo - g, g - hi))
    if report is not None:
        report[name] = dict(exact=frac, max_code_dist=int(dist.max(initial=0)),
                            max_code_dist_own=int(np.abs(g - e4m3_ordinal(ref_codes)).max(initial=0)))
    assert frac >= FRAC_FP8_EXACT, f"{name}: only {frac:.5f} of E4M3 codes identical"
    assert dist.max(initial=0) <= 1, f"{name}: E4M3 codes up to {dist.max()} apart"


def check_against_oracle(gpu: dict, inp: dict, report=None, q_c=True, dump_name=None):
    """Oracle reference (tie-aware) and every check; on failure, saves the GPU
    outputs under $MLA_PARITY_DUMP (if set) for offline analysis."""
    import os

    if report is None:
        report = {}
    ref = reference_for(inp, gpu.get("q_c") if q_c else None, report=report)
    try:
        check_step(gpu, ref, inp, report=report, q_c=q_c)
    except AssertionError:
        d = os.environ.get("MLA_PARITY_DUMP")
        if d and dump_name:
            os.makedirs(d, exist_ok=True)
            np.savez_compressed(os.path.join(d, f"{dump_name}.npz"),
                                **{k: v for k, v in gpu.items() if k != "cache"})
        raise
    finally:
        print("parity", dump_name or "", report)
        log = os.environ.get("MLA_PARITY_LOG")
        if log:
            import json

            with open(log, "a") as f:
                f.write(json.dumps({"case": dump_name or os.environ.get("PYTEST_CURRENT_TEST", ""),
                                    **report}) + "\n")
    return ref
