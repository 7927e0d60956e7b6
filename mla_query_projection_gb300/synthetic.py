"""Seeded synthetic inputs for the decode-step MLA query path.

This module draws random numbers and packs them; it holds none of the path's
arithmetic.  Both the CUDA-side tests/bench and the CPU oracle consume what it
returns (plain numpy arrays of raw bits), so neither side generates its own data.

Workload recipe (the shapes and value distributions of the MLA query workloads):
  W_QB ~ N(0, 0.02), W_UK ~ N(0, 0.05), gamma_q / gamma_kv ~ 1 + N(0, 0.1),
  q_a, kv_c, k_pe ~ N(0, 1), all drawn in float32 and rounded to bfloat16 by
  torch's float32 -> bfloat16 cast; eps = 1e-6; k_scale = 0.05; page size 64;
  slot_mapping = the first B entries of a random permutation of all slots
  (distinct slots); the cache is pre-filled with random bytes.
  Options: ``row_scale`` multiplies each q_a and each kv_c row by its own factor
  drawn log-uniform in [0.1, 10]; ``outliers`` multiplies a Bernoulli(p) subset
  of kv_c values by 1e3; ``hidden`` also draws the down-projection that makes
  the fused q_a | kv_c | k_pe row: hidden rows [B, 7168] ~ N(0, 1) and its
  weight W_QKV_A [2112, 7168] ~ N(0, 0.012) (0.012 ~ 1/sqrt(7168), so the
  projected row has about unit variance, like the drawn activations).
Draw order is fixed: W_QB, W_UK, gamma_q, gamma_kv, q_a, kv_c, k_pe, slots,
outlier mask, row scales, cache pre-fill, then (``hidden``) W_QKV_A and the
hidden rows.
"""

from __future__ import annotations

import numpy as np

LAYOUT_E4M3 = 0
LAYOUT_DS_MLA = 1
LAYOUT_NVFP4_DS_MLA = 2
ROW_BYTES = {LAYOUT_E4M3: 576, LAYOUT_DS_MLA: 656, LAYOUT_NVFP4_DS_MLA: 352}
PAGE_SIZE = 64

# The named workloads: (batch, heads, layout, pages, options).
WORKLOADS = {
    "tiny_b1_h16_e4m3": dict(batch=1, heads=16, layout=LAYOUT_E4M3, pages=8, seed=0),
    "latency_b1_h64_e4m3": dict(batch=1, heads=64, layout=LAYOUT_E4M3, pages=1024, seed=1),
    "small_b8_h128_e4m3": dict(
        batch=8, heads=128, layout=LAYOUT_E4M3, pages=2048, seed=2, row_scale=True
    ),
    "tensorcore_b64_h128_ds": dict(
        batch=64, heads=128, layout=LAYOUT_DS_MLA, pages=4096, seed=3, outliers=0.01
    ),
    # the step from the hidden row: down-projection 7168 -> 2112, then the path
    "hidden_b1_h64_e4m3": dict(
        batch=1, heads=64, layout=LAYOUT_E4M3, pages=1024, seed=5, hidden=True
    ),
}
QKV_ROW = 2112
HIDDEN = 7168


def sweep_workload(batch: int, heads: int, layout: int, seed: int = 4) -> dict:
    """One point of the B x H x layout sweep (4096 pages, kv_c outliers 1%)."""
    return dict(batch=batch, heads=heads, layout=layout, pages=4096, seed=seed, outliers=0.01)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 draws -> bfloat16 bit patterns via torch's cast (a library call)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def make_weights(heads: int, rng: np.random.Generator) -> dict:
    w_qb = to_bf16_bits(rng.standard_normal((heads * 192, 1536), dtype=np.float32) * 0.02)
    w_uk = to_bf16_bits(rng.standard_normal((heads, 128, 512), dtype=np.float32) * 0.05)
    gamma_q = to_bf16_bits(1.0 + rng.standard_normal(1536, dtype=np.float32) * 0.1)
    gamma_kv = to_bf16_bits(1.0 + rng.standard_normal(512, dtype=np.float32) * 0.1)
    return dict(w_qb=w_qb, w_uk=w_uk, gamma_q=gamma_q, gamma_kv=gamma_kv)


def make_inputs(
    batch: int,
    heads: int,
    layout: int,
    pages: int,
    seed: int,
    row_scale: bool = False,
    outliers: float = 0.0,
    page_size: int = PAGE_SIZE,
    prefill: bool = True,
    hidden: bool = False,
) -> dict:
    """All inputs of one decode step, as numpy arrays of raw bits.

    Returns keys w_qb, w_uk, gamma_q, gamma_kv, q_a, kv_c, k_pe (uint16 BF16
    bits), slots (int64), cache (uint8 [pages, page_size, row_bytes]), layout,
    k_scale, eps, heads, batch."""
    rng = np.random.default_rng(seed)
    out = make_weights(heads, rng)
    q_a = rng.standard_normal((batch, 1536), dtype=np.float32)
    kv_c = rng.standard_normal((batch, 512), dtype=np.float32)
    k_pe = rng.standard_normal((batch, 64), dtype=np.float32)
    capacity = pages * page_size
    if batch > capacity:
        raise ValueError("batch exceeds the number of cache slots")
    slots = rng.permutation(capacity)[:batch].astype(np.int64)
    if outliers > 0.0:
        mask = rng.random((batch, 512)) < outliers
        kv_c = np.where(mask, kv_c * np.float32(1e3), kv_c).astype(np.float32)
    if row_scale:
        lo, hi = np.log(0.1), np.log(10.0)
        sq = np.exp(rng.uniform(lo, hi, size=(batch, 1))).astype(np.float32)
        skv = np.exp(rng.uniform(lo, hi, size=(batch, 1))).astype(np.float32)
        q_a = q_a * sq
        kv_c = kv_c * skv
    row_bytes = ROW_BYTES[layout]
    if prefill:
        cache = rng.integers(0, 256, size=(pages, page_size, row_bytes), dtype=np.uint8)
    else:
        cache = np.zeros((pages, page_size, row_bytes), dtype=np.uint8)
    out.update(
        q_a=to_bf16_bits(q_a),
        kv_c=to_bf16_bits(kv_c),
        k_pe=to_bf16_bits(k_pe),
        slots=slots,
        cache=cache,
        layout=layout,
        k_scale=0.05,
        eps=1e-6,
        heads=heads,
        batch=batch,
    )
    if hidden:
        out.update(qkv_a_weights(rng), hidden=hidden_rows(batch, rng))
    return out


def qkv_a_weights(rng: np.random.Generator, n: int = QKV_ROW, k: int = HIDDEN) -> dict:
    """W_QKV_A [n, k] ~ N(0, 0.012), BF16 bits."""
    w = rng.standard_normal((n, k), dtype=np.float32) * np.float32(0.012)
    return dict(w_qkv_a=to_bf16_bits(w))


def hidden_rows(batch: int, rng: np.random.Generator, k: int = HIDDEN) -> np.ndarray:
    """Hidden rows [batch, k] ~ N(0, 1), BF16 bits."""
    return to_bf16_bits(rng.standard_normal((batch, k), dtype=np.float32))


def workload_inputs(name: str, **override) -> dict:
    """Inputs of a named workload (see ``WORKLOADS``)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(override)
    return make_inputs(**cfg)
