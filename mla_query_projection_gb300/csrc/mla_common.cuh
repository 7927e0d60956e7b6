// mla_common.cuh - device pieces shared by the MLA query kernels: launch
// geometry constants, named barriers, timeline stamps of trace builds and the
// paged FP8 KV insert (page "mla.query", methods insert, kv_fp8, insert_ds).
#pragma once

#include "../../include/mla_query.h"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;  // 256
constexpr int kThreads = kConsumers + 32;        // + one producer warp
constexpr int kPitch = kRowBytes + 64;           // 3136 B: conflict-free MMA loads
constexpr long long kWaitLimit = 2000000000LL;   // ~1 s of SM clock

// Named barriers (0 is __syncthreads).
constexpr int kBarNorm = 1;       // warps 0-5: q_a RMSNorm
constexpr int kBarInsert = 2;     // warps 6-7: KV insert
constexpr int kBarConsumers = 3;  // warps 0-7

__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Timeline stamps (MLA_TRACE builds): slot 0 start, 1 producer ring filled,
// 2 consumer prologue done, 3 first W_UK wait start, 4 its end, 5 end of the
// nope phase, 6 last stage consumed, 7 end, 8..27 the time consumer thread 0
// saw stage s's data, 28..47 the time the producer issued stage s, 48..63 the
// time consumer thread 0 finished stage s (s < 16).
// Trace builds: add a cycle count to a per-CTA slot (one thread per CTA).
__device__ __forceinline__ void trace_add(const DecodeArgs& a, int slot, long long v) {
#ifdef MLA_TRACE
  if (a.trace != nullptr && slot < kTraceSlots)
    a.trace[(int64_t)(blockIdx.y * gridDim.x + blockIdx.x) * kTraceSlots + slot] += (uint64_t)v;
#else
  (void)a;
  (void)slot;
  (void)v;
#endif
}

// Trace builds: the time now (0 otherwise), to be stored later by trace_put.
__device__ __forceinline__ uint64_t trace_now() {
#ifdef MLA_TRACE
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
#else
  return 0;
#endif
}
__device__ __forceinline__ void trace_put(const DecodeArgs& a, int slot, uint64_t t) {
#ifdef MLA_TRACE
  if (a.trace != nullptr && slot < kTraceSlots)
    a.trace[(int64_t)(blockIdx.y * gridDim.x + blockIdx.x) * kTraceSlots + slot] = t;
#else
  (void)a;
  (void)slot;
  (void)t;
#endif
}

__device__ __forceinline__ void trace_stamp(const DecodeArgs& a, int slot) {
#ifdef MLA_TRACE
  if (a.trace != nullptr && slot < kTraceSlots) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    a.trace[(int64_t)(blockIdx.y * gridDim.x + blockIdx.x) * kTraceSlots + slot] = t;
  }
#else
  (void)a;
  (void)slot;
#endif
}

// Bounds checks of a checks build (compiled with -DMLA_CHECKS, standing in
// for a memory checker): MLA_IN_BOUNDS(a, cond, site) is cond, and a false
// cond raises MLA_DEVERR_CHECK with bit 8 + site in the error word; the
// caller then skips the access.  In other builds it is `true` and cond is
// not evaluated.  Sites: 0 paired copy source, 1 paired ring slot, 2 paired
// q_pe store, 3 paired q_latent store, 4 paired exchange offset, 5 wide tile
// source, 6 wide ring slot or TMEM column, 7 wide output store, 8 wide
// exchange or q tile offset, 9 normalised-row tile store, 10 small-batch copy
// source, 11 small-batch ring slot, 12 small-batch exchange offset, 13
// small-batch output store, 14 partials buffer, 15 partials output store,
// 16 KV row, 17 hand-off q buffer.
#ifdef MLA_CHECKS
__device__ __noinline__ void check_failed(const DecodeArgs& a, int site) {
  atomicOr(a.err, MLA_DEVERR_CHECK | (1u << (8 + site)));
}
#define MLA_IN_BOUNDS(a, cond, site) ((cond) ? true : (::mla::check_failed((a), (site)), false))
#else
#define MLA_IN_BOUNDS(a, cond, site) true
#endif

// One query output element (q_latent or q_pe) at index idx of its tensor:
// BF16 bits, or with the per-tensor FP8 query (a.q_scale_inv set) the E4M3
// code of bf16(v) * qsi, the product rounded to binary32 (qsi = *q_scale_inv,
// loaded once by the caller with load_qsi).
__device__ __forceinline__ float load_qsi(const DecodeArgs& a) {
  return a.q_scale_inv != nullptr ? *a.q_scale_inv : 1.0f;
}
__device__ __forceinline__ uint8_t q_fp8(float v, float qsi) {
  return (uint8_t)(e4m3x2(__fmul_rn(bf_round(v), qsi), 0.0f) & 0xFFu);
}
__device__ __forceinline__ void put_q(const DecodeArgs& a, uint16_t* base, int64_t idx, float v,
                                      float qsi) {
  if (a.q_scale_inv == nullptr)
    base[idx] = f2bf_bits(v);
  else
    reinterpret_cast<uint8_t*>(base)[idx] = q_fp8(v, qsi);
}
// The first n of the N values v[] go to base[i0 + t * step], t = 0..n-1, in the
// output type; the type is chosen once for the whole run.
template <int N>
__device__ __forceinline__ void put_q_run(const DecodeArgs& a, uint16_t* base, int64_t i0,
                                          int64_t step, const float (&v)[N], int n, float qsi) {
  if (a.q_scale_inv == nullptr) {
    uint16_t* d = base + i0;
#pragma unroll
    for (int t = 0; t < N; ++t, d += step)
      if (t < n) *d = f2bf_bits(v[t]);
  } else {
    uint8_t* d = reinterpret_cast<uint8_t*>(base) + i0;
#pragma unroll
    for (int t = 0; t < N; ++t, d += step)
      if (t < n) *d = q_fp8(v[t], qsi);
  }
}

// The cache bytes of latent columns 8 lt..8 lt + 7 of a token's row (its
// normalised BF16 values n) and, for lt < 8, of its k_pe values 8 lt..8 lt + 7,
// in the row's layout (page "mla.query", methods insert, kv_fp8, insert_ds,
// insert_nvfp4).  The fp8_ds_mla tile amax and the nvfp4 block amax are
// reduced across the lanes that share them (16 and 2 consecutive lanes), so
// the whole warp calls this together, with lt % 32 equal to the lane.
__device__ __forceinline__ void kv_store_group(const DecodeArgs& a, uint8_t* row,
                                               const float (&n)[8], uint4 pe, int lt, bool ds,
                                               bool nv, float ks) {
  const int lane = lt & 31;
  if (nv) {
    // one 16-value block per thread pair: E4M3 scale of max(amax / 6, 2^-9),
    // values as E2M1 of n * (1 / scale) with the stored (rounded) scale
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(n[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    const float sf = fmaxf(__fdiv_rn(amax, 6.0f), 0x1p-9f);
    const uint32_t code = e4m3x2(sf, 0.0f) & 0xFFu;
    const float inv = __fdiv_rn(1.0f, e4m3_value(code));
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(n[i], inv);
    *reinterpret_cast<uint32_t*>(row + 4 * lt) = e2m1x8(y);
    if ((lt & 1) == 0) {
      const int s = lt >> 1;
      row[kNvScales + 8 * (s & 3) + (s >> 2)] = (uint8_t)code;
    }
    if (lt < 8) {
      const uint32_t w2[4] = {pe.x, pe.y, pe.z, pe.w};
      uint2 o2;
      o2.x = (uint32_t)e4m3x2(bf16lo(w2[0]), bf16hi(w2[0])) |
             ((uint32_t)e4m3x2(bf16lo(w2[1]), bf16hi(w2[1])) << 16);
      o2.y = (uint32_t)e4m3x2(bf16lo(w2[2]), bf16hi(w2[2])) |
             ((uint32_t)e4m3x2(bf16lo(w2[3]), bf16hi(w2[3])) << 16);
      *reinterpret_cast<uint2*>(row + kNvRope + 8 * lt) = o2;
    }
    return;
  }
  uint2 out;
  if (!ds) {
    out.x = (uint32_t)e4m3x2(__fdiv_rn(n[0], ks), __fdiv_rn(n[1], ks)) |
            ((uint32_t)e4m3x2(__fdiv_rn(n[2], ks), __fdiv_rn(n[3], ks)) << 16);
    out.y = (uint32_t)e4m3x2(__fdiv_rn(n[4], ks), __fdiv_rn(n[5], ks)) |
            ((uint32_t)e4m3x2(__fdiv_rn(n[6], ks), __fdiv_rn(n[7], ks)) << 16);
  } else {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(n[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float scale = pow2_ceil_f32(fmaxf(__fdiv_rn(amax, 448.0f), 1e-4f));
    const float inv = __fdiv_rn(1.0f, scale);  // exact: a power of two
    out.x = (uint32_t)e4m3x2(n[0] * inv, n[1] * inv) |
            ((uint32_t)e4m3x2(n[2] * inv, n[3] * inv) << 16);
    out.y = (uint32_t)e4m3x2(n[4] * inv, n[5] * inv) |
            ((uint32_t)e4m3x2(n[6] * inv, n[7] * inv) << 16);
    if ((lane & 15) == 0) *reinterpret_cast<float*>(row + kDsScales + 4 * (lt >> 4)) = scale;
  }
  *reinterpret_cast<uint2*>(row + 8 * lt) = out;
  if (lt < 8) {
    if (ds) {
      *reinterpret_cast<uint4*>(row + kDsRope + 16 * lt) = pe;
    } else {
      const uint32_t w2[4] = {pe.x, pe.y, pe.z, pe.w};
      uint2 o2;
      o2.x = (uint32_t)e4m3x2(__fdiv_rn(bf16lo(w2[0]), ks), __fdiv_rn(bf16hi(w2[0]), ks)) |
             ((uint32_t)e4m3x2(__fdiv_rn(bf16lo(w2[1]), ks), __fdiv_rn(bf16hi(w2[1]), ks)) << 16);
      o2.y = (uint32_t)e4m3x2(__fdiv_rn(bf16lo(w2[2]), ks), __fdiv_rn(bf16hi(w2[2]), ks)) |
             ((uint32_t)e4m3x2(__fdiv_rn(bf16lo(w2[3]), ks), __fdiv_rn(bf16hi(w2[3]), ks)) << 16);
      *reinterpret_cast<uint2*>(row + kKvLora + 8 * lt) = o2;
    }
  }
}

// Sum of squares of 8 BF16 values in one FMA chain.
__device__ __forceinline__ float kv_group_ss(uint4 v, float (&x)[8]) {
  const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16lo(xw[i]);
    x[2 * i + 1] = bf16hi(xw[i]);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
  return ss;
}

// The cache row of a slot, or null (a negative slot skips the row; a slot
// beyond the cache skips it and sets MLA_DEVERR_BAD_SLOT).
__device__ __forceinline__ uint8_t* kv_row(const DecodeArgs& a, int64_t slot, bool flag) {
  if (slot < 0) return nullptr;
  const int64_t page = slot / a.page_size, off = slot % a.page_size;
  if (page >= a.num_pages) {
    if (flag) atomicOr(a.err, MLA_DEVERR_BAD_SLOT);
    return nullptr;
  }
  const bool ds = a.layout == MLA_KV_FP8_DS_MLA, nv = a.layout == MLA_KV_NVFP4_DS_MLA;
  if (!MLA_IN_BOUNDS(a, page >= 0 && off >= 0 && off < a.page_size, 16)) return nullptr;
  return a.cache + (page * a.page_size + off) * (ds ? kRowDs : nv ? kRowNvfp4 : kRowE4m3);
}

// Normalised BF16 values of 8 columns: bf16((x * rr) * gamma).
__device__ __forceinline__ void kv_group_norm(const float (&x)[8], uint4 gv, float rr,
                                              float (&n)[8]) {
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    n[2 * i] = bf_round(__fmul_rn(__fmul_rn(x[2 * i], rr), bf16lo(gw[i])));
    n[2 * i + 1] = bf_round(__fmul_rn(__fmul_rn(x[2 * i + 1], rr), bf16hi(gw[i])));
  }
}

// Paged KV insert of token b (page "mla.query", methods insert, kv_fp8,
// insert_ds, insert_nvfp4), run by 64 threads (lt = 0..63, two whole warps).
// Thread lt owns latent columns 8*lt..8*lt+7; threads 0..7 also own k_pe
// values 8*lt..8*lt+7.  red2 holds the two warps' partial sums.
// The inputs of thread lt's share of token b's KV insert, loaded ahead of
// the arithmetic (kv_insert_loaded), so a kernel can issue them together
// with its other loads.
struct KvLoads {
  int64_t slot;
  uint4 v, gv, pe;
};
__device__ __forceinline__ KvLoads kv_insert_load(const DecodeArgs& a, int b, int lt) {
  KvLoads l;
  l.slot = a.slots[b];
  l.v = *reinterpret_cast<const uint4*>(a.kv_c + (int64_t)b * a.kv_c_stride + 8 * lt);
  l.gv = *reinterpret_cast<const uint4*>(a.gamma_kv + 8 * lt);
  l.pe = make_uint4(0, 0, 0, 0);
  if (lt < 8) l.pe = *reinterpret_cast<const uint4*>(a.k_pe + (int64_t)b * a.k_pe_stride + 8 * lt);
  return l;
}

__device__ void kv_insert_loaded(const DecodeArgs& a, int lt, float* red2, const KvLoads& l) {
  const int lane = lt & 31, w = lt >> 5;
  const int64_t slot = l.slot;
  const uint4 v = l.v, gv = l.gv, pe = l.pe;
  const bool ds = a.layout == MLA_KV_FP8_DS_MLA;
  const bool nv = a.layout == MLA_KV_NVFP4_DS_MLA;
  const float ks = (ds || nv) ? 1.0f : *a.k_scale;
  float x[8];
  float ss = warp_sum(kv_group_ss(v, x));
  if (lane == 0) red2[w] = ss;
  named_barrier(kBarInsert, 64);
  const float total = red2[0] + red2[1];
  named_barrier(kBarInsert, 64);  // red2 may be reused by the next token
  uint8_t* row = kv_row(a, slot, lt == 0);
  if (row == nullptr) return;
  const float rr = __frsqrt_rn(__fadd_rn(__fmul_rn(total, 1.0f / 512.0f), a.eps));
  float n[8];
  kv_group_norm(x, gv, rr, n);
  kv_store_group(a, row, n, pe, lt, ds, nv, ks);
}

__device__ void kv_insert(const DecodeArgs& a, int b, int lt, float* red2) {
  kv_insert_loaded(a, lt, red2, kv_insert_load(a, b, lt));
}

// The same insert run by one warp: lane l takes the columns of threads l and
// l + 32 of the 64-thread insert, and the sums are formed in the same order
// (each group's FMA chain, each group reduced across the warp, group 0 plus
// group 1), so the bytes written are the same.
// The inputs of one lane's share of the one-warp insert (kv_insert_warp),
// loaded ahead of its arithmetic (kv_insert_warp_loaded).
struct KvWarpLoads {
  int64_t slot;
  uint4 v[2], gv[2], pe;
};
__device__ __forceinline__ KvWarpLoads kv_insert_warp_load(const DecodeArgs& a, int b, int lane) {
  KvWarpLoads l;
  l.slot = a.slots[b];
  const uint16_t* kv = a.kv_c + (int64_t)b * a.kv_c_stride;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    l.v[g] = *reinterpret_cast<const uint4*>(kv + 8 * (lane + 32 * g));
    l.gv[g] = *reinterpret_cast<const uint4*>(a.gamma_kv + 8 * (lane + 32 * g));
  }
  l.pe = make_uint4(0, 0, 0, 0);
  if (lane < 8) l.pe = *reinterpret_cast<const uint4*>(a.k_pe + (int64_t)b * a.k_pe_stride + 8 * lane);
  return l;
}

__device__ void kv_insert_warp_loaded(const DecodeArgs& a, int lane, const KvWarpLoads& l) {
  const int64_t slot = l.slot;
  const uint4 v[2] = {l.v[0], l.v[1]}, gv[2] = {l.gv[0], l.gv[1]};
  const uint4 pe = l.pe;
  const bool ds = a.layout == MLA_KV_FP8_DS_MLA;
  const bool nv = a.layout == MLA_KV_NVFP4_DS_MLA;
  const float ks = (ds || nv) ? 1.0f : *a.k_scale;
  float x[2][8];
  const float s0 = warp_sum(kv_group_ss(v[0], x[0]));
  const float s1 = warp_sum(kv_group_ss(v[1], x[1]));
  uint8_t* row = kv_row(a, slot, lane == 0);
  if (row == nullptr) return;
  const float rr = __frsqrt_rn(__fadd_rn(__fmul_rn(s0 + s1, 1.0f / 512.0f), a.eps));
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    float n[8];
    kv_group_norm(x[g], gv[g], rr, n);
    kv_store_group(a, row, n, g == 0 ? pe : make_uint4(0, 0, 0, 0), lane + 32 * g, ds, nv, ks);
  }
}

__device__ void kv_insert_warp(const DecodeArgs& a, int b, int lane) {
  kv_insert_warp_loaded(a, lane, kv_insert_warp_load(a, b, lane));
}

}  // namespace
}  // namespace mla
