// mla_fused.cu - the fused decode-step kernel of the MLA query path.
//
// One persistent launch (one CTA per SM, `groups` token groups along grid.y)
// computes, for the tokens of its group (page "mla.query", class MlaQuery,
// methods kernel / tiled / insert / insert_ds / store_qc):
//   q_a RMSNorm -> xq (q_c), Q_B rows -> q (BF16), rope rows -> q_pe,
//   nope rows through W_UK -> q_latent, and the paged FP8 KV insert.
//
// GB300 design (not the page's cluster design):
//  * Weight streaming.  Each CTA owns a byte-balanced share of three lists:
//    the H*128 nope rows of W_QB, then a combined list per head of the eight
//    64-column W_UK tiles and the 64 rope rows.  A producer warp streams them
//    into a ring of stages: rows by 1-D bulk TMA (3 KiB each, padded smem
//    pitch), W_UK tiles by 2-D tensor TMA with 128 B swizzle; full/empty
//    mbarriers pace it, so a slot is refilled as soon as the eight consumer
//    warps release it.  Weights do not depend on the previous kernel, so the
//    producer starts before the programmatic-dependent-launch wait.
//  * Nope hand-off.  All CTAs stream their nope rows first and publish the
//    BF16 q values to a small global scratch; a per-(group, head) counter
//    reaches 128 when a head is complete (one release per head and writer).
//    Every CTA streams its rope rows next and its W_UK tiles last, so by then
//    the counters are normally full; each warp waits (bounded: a timeout
//    raises MLA_DEVERR_TIMEOUT instead of hanging) and loads the head's q
//    once per head.  The last CTA re-arms the counters.
//  * Arithmetic (16-row stages of 49 KiB: fewer, larger stages stream faster).
//    FMA flavour (1-2 tokens): FP32 FMAs, one warp per row, x in registers.
//    MMA flavour (8 or 16 tokens per CTA): BF16 mma.sync m16n8k16 with the weight rows as the M side
//    (tokens are N), K split over the eight consumer warps and reduced in a
//    fixed order through smem; the absorption takes the swizzled W_UK tile as
//    the M side through ldmatrix.trans.
#include <cuda_bf16.h>

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

enum StageKind { kNopeRows = 0, kRopeRows = 1, kUkTiles = 2 };

struct Stage {
  int kind;
  int first;  // nope index n (h*128+p), rope index r (h*64+p-128) or unit u (h*8+cb)
  int count;
};

template <bool MMA>
struct Geo {
  static constexpr int kStageRows = 16;
  static constexpr int kStageBytes = ((kStageRows * kPitch + 1023) / 1024) * 1024;
  static constexpr int kUkPerStage = kStageBytes / kUkUnitBytes;  // 3
  static_assert(kNope % kStageRows == 0 && kRope % kStageRows == 0, "stages within a head");
  static_assert(kUkPerStage >= 3, "three W_UK units per stage");
};

__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The stage list of one token group: H*8 stages of 16 nope rows, then H*3
// stages of W_UK units (units 0-2, 3-5 and 6-7 of each head), then H*4
// stages of 16 rope rows.  Stages never straddle heads.  CTA i takes stages
// i, i+P, i+2P, ...: every CTA streams nope rows first; by the time a CTA
// reaches the absorption of head h, the nope rows of h were taken at least
// a round earlier, and the rope rows it streams afterwards keep its copy
// queue busy while it waits.
__device__ __forceinline__ int total_stages(int H) { return 15 * H; }

__device__ __forceinline__ Stage decode_stage(int idx, int H) {
  Stage s;
  const int n_nope = 8 * H, n_uk = 3 * H;
  if (idx < n_nope) {
    s.kind = kNopeRows;
    s.first = 16 * idx;
    s.count = 16;
  } else if (idx < n_nope + n_uk) {
    const int u = idx - n_nope, h = u / 3, k = u % 3;
    s.kind = kUkTiles;
    s.first = h * kUkUnitsPerHead + 3 * k;
    s.count = k == 2 ? 2 : 3;
  } else {
    s.kind = kRopeRows;
    s.first = 16 * (idx - n_nope - n_uk);
    s.count = 16;
  }
  return s;
}

__device__ __forceinline__ int stage_row(const Stage& s, int j) {
  if (s.kind == kNopeRows) {
    const int n = s.first + j;
    return (n / kNope) * kHeadRows + (n % kNope);
  }
  const int r = s.first + j;
  return (r / kRope) * kHeadRows + kNope + (r % kRope);
}

// Issue the copies of stage `s` into `buf` (all 32 lanes of the producer warp).
__device__ __forceinline__ void issue_stage(const Stage& s, uint8_t* buf, uint64_t* bar,
                                            const DecodeArgs& a, const CUtensorMap* uk_map,
                                            int lane) {
  if (s.kind == kUkTiles) {
    if (lane == 0 && a.w_uk_packed != nullptr) {
      // consecutive units of one head are contiguous in the packed copy
      mbar_arrive_expect_tx(bar, (uint32_t)(s.count * kUkUnitBytes));
      bulk_g2s(buf, a.w_uk_packed + (int64_t)s.first * kUkUnitBytes,
               (uint32_t)(s.count * kUkUnitBytes), bar);
    } else if (lane == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)(s.count * kUkUnitBytes));
      for (int j = 0; j < s.count; ++j) {
        const int u = s.first + j;
        tma_g2s_2d(buf + j * kUkUnitBytes, uk_map, (u % kUkUnitsPerHead) * kUkCols,
                   (u / kUkUnitsPerHead) * kNope, bar);
      }
    }
  } else {
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(s.count * kRowBytes));
    __syncwarp();
    if (lane < s.count) {
      const int row = stage_row(s, lane);
      bulk_g2s(buf + lane * kPitch, a.w_qb + (int64_t)row * kQLora, kRowBytes, bar);
    }
  }
}

// Paged FP8 KV insert of token b (page "mla.query", methods insert, kv_fp8,
// insert_ds), run by the 64 threads of warps 6-7 (lt = 0..63) while warps 0-5
// normalise q_a.  Thread lt owns latent columns 8*lt..8*lt+7; threads 0..7
// also own k_pe values 8*lt..8*lt+7.  red2 holds the two warps' partial sums.
__device__ void kv_insert(const DecodeArgs& a, int b, int lt, float* red2) {
  const int lane = lt & 31, w = lt >> 5;
  const int64_t slot = a.slots[b];
  const uint4 v = *reinterpret_cast<const uint4*>(a.kv_c + (int64_t)b * a.kv_c_stride + 8 * lt);
  const uint4 gv = *reinterpret_cast<const uint4*>(a.gamma_kv + 8 * lt);
  uint4 pe = make_uint4(0, 0, 0, 0);
  if (lt < 8) pe = *reinterpret_cast<const uint4*>(a.k_pe + (int64_t)b * a.k_pe_stride + 8 * lt);
  const bool ds = a.layout == MLA_KV_FP8_DS_MLA;
  const float ks = ds ? 1.0f : *a.k_scale;
  float x[8];
  const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16lo(xw[i]);
    x[2 * i + 1] = bf16hi(xw[i]);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
  ss = warp_sum(ss);
  if (lane == 0) red2[w] = ss;
  named_barrier(kBarInsert, 64);
  const float total = red2[0] + red2[1];
  named_barrier(kBarInsert, 64);  // red2 may be reused by the next token
  if (slot < 0) return;
  const int64_t page = slot / a.page_size, off = slot % a.page_size;
  if (page >= a.num_pages) {
    if (lt == 0) atomicOr(a.err, MLA_DEVERR_BAD_SLOT);
    return;
  }
  uint8_t* row = a.cache + (page * a.page_size + off) * (ds ? kRowDs : kRowE4m3);
  const float rr = __frsqrt_rn(__fadd_rn(__fmul_rn(total, 1.0f / 512.0f), a.eps));
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  float n[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    n[2 * i] = bf_round(__fmul_rn(__fmul_rn(x[2 * i], rr), bf16lo(gw[i])));
    n[2 * i + 1] = bf_round(__fmul_rn(__fmul_rn(x[2 * i + 1], rr), bf16hi(gw[i])));
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

// Timeline stamps (MLA_TRACE builds): slot 0 start, 1 producer ring filled,
// 2 consumer prologue done, 3 first W_UK wait start, 4 its end, 5 end of the
// nope phase, 6 last stage consumed, 7 end, 8..27 the time consumer thread 0
// saw stage s's data, 28..47 the time the producer issued stage s, 48..63 the
// time consumer thread 0 finished stage s (s < 16).
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

// Bounded wait of one lane until `ready` reaches `target`; false on timeout.
__device__ __forceinline__ bool wait_ready(const uint32_t* ready, uint32_t target) {
  if (ld_acquire_gpu(ready) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(ready) < target) {
    if (clock64() - t0 > kWaitLimit) return false;
    __nanosleep(64);
  }
  return true;
}

// Nope rows a warp (FMA: its own rows, two per stage) or the CTA (MMA: a
// whole stage, via thread 0) stored but has not yet published: a list of
// head indices in shared memory, each entry `rows` rows of that head.  One
// lane publishes the whole list with a single fence when the CTA leaves its
// nope stages, or when the list is full.
constexpr int kPendMax = 16;

__device__ __forceinline__ void flush_pending(int* list, int& n, int rows, uint32_t* ready_g) {
  if (n == 0) return;
  __threadfence();
  for (int e = 0; e < n; ++e) red_release_gpu_add(ready_g + list[e], (uint32_t)rows);
  n = 0;
}

// End of a CTA's nope stages: publish every pending row.  In the MMA
// flavour thread 0 publishes for the CTA, so the consumer warps first meet
// at `sync_bar` (used once per call): every warp's q stores precede it.
template <bool MMA>
__device__ __forceinline__ void leave_nope(int* pend, int& npend, int& last_h, uint64_t* sync_bar,
                                           int lane, int tid, uint32_t* ready_g, bool& timed_out) {
  if constexpr (MMA) {
    __syncwarp();
    if (lane == 0) mbar_arrive(sync_bar);
    if (!mbar_wait_bounded(sync_bar, 0u, kWaitLimit)) timed_out = true;
    if (tid == 0 && last_h >= 0) {
      pend[npend++] = last_h;
      last_h = -1;
    }
    flush_pending(pend, npend, 16, ready_g);
  } else {
    (void)last_h;
    (void)sync_bar;
    (void)lane;
    (void)tid;
    (void)timed_out;
    flush_pending(pend, npend, 2, ready_g);
  }
}

template <int NT, bool MMA>
struct Smem {
  using G = Geo<MMA>;
  static constexpr int kStages = MMA ? 3 : 4;
  static constexpr int kRing = kStages * G::kStageBytes;
  static constexpr int kXq = NT * kPitch;
  // FMA: per-warp staged q of one head [warp][NT][128] FP32; MMA: split-K
  // partial sums [2 buffers][warp][16 rows][NT] FP32.
  static constexpr int kScratch =
      MMA ? 2 * kConsumerWarps * 16 * NT * 4 : kConsumerWarps * NT * kNope * 4;
  static constexpr int oXq = kRing;
  static constexpr int oScratch = oXq + kXq;
  static constexpr int oSs = oScratch + kScratch;  // [NT][8] + [8] floats
  static constexpr int oFull = oSs + (NT * 8 + 8) * 4;
  static constexpr int oEmpty = oFull + kStages * 8;
  static constexpr int oRbar = oEmpty + kStages * 8;  // 2 reduction barriers (MMA)
  static constexpr int oDesc = oRbar + 16;            // stage index per ring slot
  static constexpr int oPend = oDesc + kStages * 4;    // [warp][kPendMax] pending heads
  static constexpr int oFlag = oPend + kConsumerWarps * kPendMax * 4;
  static constexpr int kBytes = oFlag + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1 KiB
};

template <int NT, bool MMA>
__global__ void __launch_bounds__(kThreads, 1)
    mla_fused_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap uk_map) {
  using S = Smem<NT, MMA>;
  using G = Geo<MMA>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint8_t* xq = smem + S::oXq;
  float* ss_part = reinterpret_cast<float*>(smem + S::oSs);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::oFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::oEmpty);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + S::oRbar);
  volatile int* desc = reinterpret_cast<volatile int*>(smem + S::oDesc);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + S::oFlag);  // [1]: last CTA

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = gridDim.x, i = blockIdx.x, grp = blockIdx.y;
  const int H = a.heads;
  const int total = total_stages(H);
  const int tok0 = grp * NT;
  uint16_t* qn_g = a.qn + (int64_t)grp * NT * H * kNope;
  uint32_t* ready_g = a.ready + grp * H;

  if (tid == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
      desc[s] = -1;
    }
    mbar_init(&rbar[0], kConsumerWarps);
    mbar_init(&rbar[1], kConsumerWarps);
    flag[1] = 0;
    mbar_fence_init();
    prefetch_tensormap(&uk_map);
    trace_stamp(a, 0);
  }
  __syncthreads();

  bool timed_out = false;

  if (warp == kConsumerWarps) {
    // ================= producer warp =================================
    // Stage k of this CTA is stage k*P + i of the list.  Weights do not
    // depend on the previous kernel and the producer touches no scratch, so
    // it starts streaming without waiting for it.
    int k = 0;
    while (true) {
      const int slot = k % S::kStages;
      if (k >= S::kStages) {
        const uint32_t par = (uint32_t)(((k / S::kStages) - 1) & 1);
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(&empty[slot], par, kWaitLimit) ? 1 : 0;
        // On a timeout keep going (results are flagged invalid): every wait in
        // this kernel is bounded, so it still ends.
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) timed_out = true;
      }
      const int idx = k * P + i;
      if (idx >= total) {
        // end marker: the consumers stop at this slot
        if (lane == 0) {
          desc[slot] = -1;
          mbar_arrive(&full[slot]);
        }
        break;
      }
      if (lane == 0) {
        desc[slot] = idx;
        if (k < 20) trace_stamp(a, 28 + k);
        if (k == S::kStages) trace_stamp(a, 1);
      }
      issue_stage(decode_stage(idx, H), ring + slot * G::kStageBytes, &full[slot], a, &uk_map,
                  lane);
      ++k;
    }
    // Every issued stage is consumed; after a timeout this bounded wait also
    // covers copies that may still be landing before the CTA exits.  (Stage
    // k - kStages shared its slot with the end marker and is already done.)
    if (lane == 0) {
      for (int s = max(0, k - S::kStages + 1); s < k; ++s)
        (void)mbar_wait_bounded(&full[s % S::kStages], (uint32_t)((s / S::kStages) & 1),
                                kWaitLimit);
    }
  } else {
    // ================= consumer warps 0-7 ============================
    pdl_wait();
    if (tid == 0) pdl_launch_dependents();

    // ---- q_a RMSNorm -> xq (warps 0-5); KV insert (warps 6-7) -------
    if (warp < 6) {
      uint4 xv[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (tok0 + t < a.batch)
          xv[t] = *reinterpret_cast<const uint4*>(a.q_a + (int64_t)(tok0 + t) * a.q_a_stride +
                                                  8 * tid);
        else
          xv[t] = make_uint4(0, 0, 0, 0);
      }
      const uint4 gv = *reinterpret_cast<const uint4*>(a.gamma_q + 8 * tid);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint32_t ww[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ss = fmaf(bf16lo(ww[k]), bf16lo(ww[k]), ss);
          ss = fmaf(bf16hi(ww[k]), bf16hi(ww[k]), ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) ss_part[t * 8 + warp] = ss;
      }
      named_barrier(kBarNorm, 192);
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float* sp = ss_part + t * 8;
        const float total = ((((sp[0] + sp[1]) + sp[2]) + sp[3]) + sp[4]) + sp[5];
        const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, 1536.0f), a.eps));
        const uint32_t ww[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
        uint4 o;
        o.x = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[0]), rr), bf16lo(gw[0])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[0]), rr), bf16hi(gw[0])));
        o.y = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[1]), rr), bf16lo(gw[1])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[1]), rr), bf16hi(gw[1])));
        o.z = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[2]), rr), bf16lo(gw[2])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[2]), rr), bf16hi(gw[2])));
        o.w = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[3]), rr), bf16lo(gw[3])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[3]), rr), bf16hi(gw[3])));
        if (tok0 + t >= a.batch) o = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(xq + t * kPitch + 16 * tid) = o;
        // q_c rows (page "mla.query", method store_qc): CTA 0 of the group.
        if (i == 0 && a.q_c != nullptr && tok0 + t < a.batch)
          *reinterpret_cast<uint4*>(a.q_c + (int64_t)(tok0 + t) * kQLora + 8 * tid) = o;
      }
    } else {
      // token t of the group is inserted by CTA t % P
      for (int t = i; t < NT; t += P)
        if (tok0 + t < a.batch) kv_insert(a, tok0 + t, tid - 192, ss_part + NT * 8);
    }
    named_barrier(kBarConsumers, kConsumers);
    if (tid == 0) trace_stamp(a, 2);

    // FMA flavour: this lane's x values in registers (k = 256 c + 8 lane + e).
    float xr[MMA ? 1 : NT][MMA ? 1 : 48];
    if constexpr (!MMA) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int c = 0; c < 6; ++c) {
          const uint4 v =
              *reinterpret_cast<const uint4*>(xq + t * kPitch + 2 * (256 * c + 8 * lane));
          const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            xr[t][8 * c + 2 * k] = bf16lo(ww[k]);
            xr[t][8 * c + 2 * k + 1] = bf16hi(ww[k]);
          }
        }
    }

    // Pending nope publications (see flush_pending): kept by lane 0 of each
    // warp (FMA) or by thread 0 (MMA).
    int* pend = reinterpret_cast<int*>(smem + S::oPend) + warp * kPendMax;
    int npend = 0;
    constexpr int kPendRows = MMA ? 16 : 2;
    int last_h = -1;      // MMA: head of the last nope stage, listed after the next barrier
    bool in_nope = true;  // still in this CTA's nope stages
    int rsteps = 0;       // MMA row stages done: buffer and phase of the reduction

    // Head whose nope q this warp holds (FMA: staged in smem; MMA: as B
    // fragments in registers) after its hand-off wait, or -1.
    int cached_h = -1;
    uint32_t bf[MMA ? NT / 8 : 1][kNope / 16][2];

    for (int s = 0; s <= total; ++s) {
      const int slot = s % S::kStages;
      uint8_t* buf = ring + slot * G::kStageBytes;
      if (!mbar_wait_bounded(&full[slot], (uint32_t)((s / S::kStages) & 1), kWaitLimit))
        timed_out = true;  // the call is flagged invalid; every wait stays bounded
      const int idx = desc[slot];
      if (idx < 0 || idx >= total) break;  // end marker
      const Stage st = decode_stage(idx, H);
      if (tid == 0) {
        if (s < 20) trace_stamp(a, 8 + s);
        if (s > 0 && s <= 16) trace_stamp(a, 47 + s);
        if (st.kind != kNopeRows && in_nope) trace_stamp(a, 5);
      }
      if (in_nope && st.kind != kNopeRows) {
        in_nope = false;
        leave_nope<MMA>(pend, npend, last_h, &rbar[1], lane, tid, ready_g, timed_out);
      }

      if (st.kind == kUkTiles) {
        // ---- absorption of one head's nope q through W_UK tiles -------
        const int h = st.first / kUkUnitsPerHead;
        const int cb0 = st.first % kUkUnitsPerHead;
        const bool fresh = h != cached_h;  // warp-uniform
        if (fresh) {
          int rdy = 1;
          if (tid == 0) trace_stamp(a, 3);
          if (lane == 0) rdy = wait_ready(ready_g + h, (uint32_t)kNope) ? 1 : 0;
          if (tid == 0) trace_stamp(a, 4);
          rdy = __shfl_sync(0xFFFFFFFFu, rdy, 0);
          __syncwarp();  // orders the lanes' q loads below after lane 0's acquire
          if (!rdy) timed_out = true;
          cached_h = h;
        }
        const uint16_t* qsrc = qn_g + (int64_t)h * kNope;  // token t at + t*H*128
        if constexpr (MMA) {
          const int g = lane >> 2, q = lane & 3;
          if (fresh) {
            // B fragments (q^T, 8 tokens per n-tile) straight from L2.
#pragma unroll
            for (int nt = 0; nt < NT / 8; ++nt)
#pragma unroll
              for (int ks = 0; ks < kNope / 16; ++ks) {
                const uint16_t* qr = qsrc + (int64_t)(8 * nt + g) * H * kNope + 16 * ks + 2 * q;
                bf[nt][ks][0] = ld_cg_u32(qr);
                bf[nt][ks][1] = ld_cg_u32(qr + 8);
              }
          }
          for (int pair = warp; pair < 4 * st.count; pair += kConsumerWarps) {
            const int u = pair >> 2, mt = pair & 3;
            const uint32_t tile = smem_u32(buf + u * kUkUnitBytes);
            float acc[NT / 8][4];
#pragma unroll
            for (int nt = 0; nt < NT / 8; ++nt)
              acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kNope / 16; ++ks) {
              const int m = lane >> 3;
              const int p = 16 * ks + (lane & 7) + 8 * (m >> 1);
              const int chunk = 2 * mt + (m & 1);
              uint32_t af[4];
              ldmatrix_x4_trans(af, tile + p * 128 + ((chunk ^ (p & 7)) << 4));
#pragma unroll
              for (int nt = 0; nt < NT / 8; ++nt)
                mma_bf16_16816(acc[nt], af[0], af[1], af[2], af[3], bf[nt][ks][0], bf[nt][ks][1]);
            }
            const int cbase = (cb0 + u) * kUkCols + 16 * mt + g;
#pragma unroll
            for (int nt = 0; nt < NT / 8; ++nt) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int t = 8 * nt + 2 * q + (e & 1);
                const int c = cbase + 8 * (e >> 1);
                if (tok0 + t < a.batch)
                  a.q_latent[((int64_t)(tok0 + t) * H + h) * kKvLora + c] = f2bf_bits(acc[nt][e]);
              }
            }
          }
        } else {
          // W_UK units of 64 columns; in each, warp w owns columns 8w..8w+7.
          // Lane: column pair cp = lane & 3, rows p = pg + 8 k (pg = lane >> 2).
          float* qs = reinterpret_cast<float*>(smem + S::oScratch) + warp * NT * kNope;
          if (fresh) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const uint2 v = ld_cg_u32x2(qsrc + (int64_t)t * H * kNope + 4 * lane);
              qs[t * kNope + 4 * lane] = bf16lo(v.x);
              qs[t * kNope + 4 * lane + 1] = bf16hi(v.x);
              qs[t * kNope + 4 * lane + 2] = bf16lo(v.y);
              qs[t * kNope + 4 * lane + 3] = bf16hi(v.y);
            }
            __syncwarp();
          }
          const int cp = lane & 3, pg = lane >> 2;
          for (int u = 0; u < st.count; ++u) {
            const uint8_t* tile = buf + u * kUkUnitBytes;
            float acc[NT][2];
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
            for (int k = 0; k < kNope / 8; ++k) {
              const int p = pg + 8 * k;
              const uint32_t wv = *reinterpret_cast<const uint32_t*>(
                  tile + p * 128 + ((warp ^ (p & 7)) << 4) + 4 * cp);
              const float w0 = bf16lo(wv), w1 = bf16hi(wv);
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                acc[t][0] = fmaf(qs[t * kNope + p], w0, acc[t][0]);
                acc[t][1] = fmaf(qs[t * kNope + p], w1, acc[t][1]);
              }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float v = acc[t][e];
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
                acc[t][e] = v;
              }
            if (pg == 0) {
              const int c = (cb0 + u) * kUkCols + 8 * warp + 2 * cp;
#pragma unroll
              for (int t = 0; t < NT; ++t)
                if (tok0 + t < a.batch)
                  *reinterpret_cast<uint32_t*>(a.q_latent +
                                               ((int64_t)(tok0 + t) * H + h) * kKvLora + c) =
                      pack_bf16x2(acc[t][0], acc[t][1]);
            }
          }
        }
      } else if constexpr (MMA) {
        // ---- Q_B rows, tensor cores, K split over the warps ----------
        // partial sums, double-buffered: one barrier per stage suffices
        float* red = reinterpret_cast<float*>(smem + S::oScratch) + (rsteps & 1) * (kConsumerWarps * 16 * NT);
        const int g = lane >> 2, q = lane & 3;
        float acc[NT / 8][4];
#pragma unroll
        for (int nt = 0; nt < NT / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
        for (int c = 0; c < 6; ++c) {
          const int kb = 2 * (192 * warp + 32 * c + 8 * q);
          const uint4 alo = *reinterpret_cast<const uint4*>(buf + g * kPitch + kb);
          const uint4 ahi = *reinterpret_cast<const uint4*>(buf + (g + 8) * kPitch + kb);
#pragma unroll
          for (int nt = 0; nt < NT / 8; ++nt) {
            const uint4 bx = *reinterpret_cast<const uint4*>(xq + (8 * nt + g) * kPitch + kb);
            mma_bf16_16816(acc[nt], alo.x, ahi.x, alo.y, ahi.y, bx.x, bx.y);
            mma_bf16_16816(acc[nt], alo.z, ahi.z, alo.w, ahi.w, bx.z, bx.w);
          }
        }
        // the weight slot is no longer read: release it to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        float* rw = red + warp * 16 * NT;
#pragma unroll
        for (int nt = 0; nt < NT / 8; ++nt) {
          rw[g * NT + 8 * nt + 2 * q] = acc[nt][0];
          rw[g * NT + 8 * nt + 2 * q + 1] = acc[nt][1];
          rw[(g + 8) * NT + 8 * nt + 2 * q] = acc[nt][2];
          rw[(g + 8) * NT + 8 * nt + 2 * q + 1] = acc[nt][3];
        }
        // partial sums of all warps written (bounded mbarrier wait); also
        // orders every warp's q stores of the previous stage before it
        __syncwarp();
        if (lane == 0) mbar_arrive(&rbar[0]);
        if (!mbar_wait_bounded(&rbar[0], (uint32_t)(rsteps & 1), kWaitLimit)) timed_out = true;
        if (tid == 0 && last_h >= 0) {
          pend[npend++] = last_h;
          last_h = -1;
          if (npend == kPendMax) flush_pending(pend, npend, kPendRows, ready_g);
        }
        for (int e = tid; e < 16 * NT; e += kConsumers) {
          const int j = e / NT, t = e % NT;
          float v = 0.f;
#pragma unroll
          for (int ww = 0; ww < kConsumerWarps; ++ww) v += red[ww * 16 * NT + e];
          const uint16_t bits = f2bf_bits(v);
          if (st.kind == kNopeRows) {
            const int n = st.first + j;
            qn_g[((int64_t)t * H + n / kNope) * kNope + n % kNope] = bits;
          } else if (tok0 + t < a.batch) {
            const int r = st.first + j;
            a.q_pe[((int64_t)(tok0 + t) * H + r / kRope) * kRope + r % kRope] = bits;
          }
        }
        ++rsteps;
        if (st.kind == kNopeRows && tid == 0) last_h = st.first / kNope;
        continue;  // slot already released
      } else {
        // ---- Q_B rows, FP32 FMA: warp w owns rows w and w + 8 -----------
        float v[2][NT];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int j = warp + kConsumerWarps * rr;
          if (j < st.count) {
            const uint8_t* rowp = buf + j * kPitch;
            float acc[NT][2];
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
            for (int c = 0; c < 6; ++c) {
              const uint4 wv = *reinterpret_cast<const uint4*>(rowp + 2 * (256 * c + 8 * lane));
              const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float w0 = bf16lo(ww[k]), w1 = bf16hi(ww[k]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                  acc[t][0] = fmaf(w0, xr[t][8 * c + 2 * k], acc[t][0]);
                  acc[t][1] = fmaf(w1, xr[t][8 * c + 2 * k + 1], acc[t][1]);
                }
              }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) v[rr][t] = acc[t][0] + acc[t][1];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // the slot is no longer read
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int j = warp + kConsumerWarps * rr;
          if (j >= st.count) break;
#pragma unroll
          for (int t = 0; t < NT; ++t) v[rr][t] = warp_sum(v[rr][t]);
          if (lane == 0) {
            if (st.kind == kNopeRows) {
              const int n = st.first + j;
              const int h = n / kNope;
#pragma unroll
              for (int t = 0; t < NT; ++t)
                qn_g[((int64_t)t * H + h) * kNope + n % kNope] = f2bf_bits(v[rr][t]);
              if (rr == 1) {  // both rows of this warp stored (one head per stage)
                pend[npend++] = h;
                if (npend == kPendMax) flush_pending(pend, npend, kPendRows, ready_g);
              }
            } else {
              const int r = st.first + j;
#pragma unroll
              for (int t = 0; t < NT; ++t)
                if (tok0 + t < a.batch)
                  a.q_pe[((int64_t)(tok0 + t) * H + r / kRope) * kRope + r % kRope] =
                      f2bf_bits(v[rr][t]);
            }
          }
        }
        continue;  // slot already released
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (in_nope) leave_nope<MMA>(pend, npend, last_h, &rbar[1], lane, tid, ready_g, timed_out);
    if (tid == 0) trace_stamp(a, 6);
  }

  // ---- end of call: flags, and the last CTA re-arms the counters ------
  if (timed_out) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t total = gridDim.x * gridDim.y;
    const uint32_t prev = atomicAdd(a.finished, 1u);
    flag[1] = (prev == total - 1) ? 1 : 0;
  }
  if (tid == 0) trace_stamp(a, 7);
  __syncthreads();
  if (flag[1]) {
    for (int e = tid; e < a.groups * H; e += kThreads) a.ready[e] = 0u;
    __syncthreads();
    if (tid == 0) {
      *a.finished = 0u;
      __threadfence();
    }
  }
}

// ===========================================================================
// Absorbing kernel (1-2 tokens): no hand-off between CTAs.
//
// A "task" is 16 consecutive nope rows of one head (48 KiB of W_QB) together
// with the same 16 rows of that head's W_UK (16 KiB, contiguous in the
// caller's [H][128][512] layout).  The CTA computes the 16 BF16 q values, then
// their contribution to all 512 latent columns, and stores that FP32 partial
// sum.  A per-head counter finds the last of a head's 8 tasks; that CTA's
// finisher warp adds the 8 partials in task order and writes q_latent.  Rope
// rows stream after a CTA's tasks and go straight to q_pe.  Each CTA owns a
// contiguous run of tasks and of rope rows, balanced in bytes on the host.
// ===========================================================================

constexpr int kTaskRows = 16;
constexpr int kTasksPerHead = kNope / kTaskRows;              // 8
constexpr int kTaskUkBytes = kTaskRows * kKvLora * 2;         // 16 KiB
constexpr int kTaskQbBytes = kTaskRows * kPitch;              // 50176
constexpr int kTaskStage = kTaskQbBytes + kTaskUkBytes;       // 66560
constexpr int kAbsStages = 3;
constexpr int kAbsThreads = kConsumers + 64;                  // + producer + finisher
constexpr int kSigRing = 4;                                   // consumer -> finisher signals

template <int NT>
struct AbsSmem {
  static constexpr int kRing = kAbsStages * kTaskStage;
  static constexpr int oXq = kRing;
  static constexpr int oQ16 = oXq + NT * kPitch;                 // [2][NT][16] FP32
  static constexpr int oSs = oQ16 + 2 * NT * kTaskRows * 4;      // [NT][8] + [8]
  static constexpr int oFull = oSs + (NT * 8 + 8) * 4;
  static constexpr int oEmpty = oFull + kAbsStages * 8;
  static constexpr int oQbar = oEmpty + kAbsStages * 8;
  static constexpr int oSig = oQbar + 8;
  static constexpr int oFree = oSig + kSigRing * 8;
  static constexpr int kBytes = oFree + kSigRing * 8;
  static constexpr int kAlloc = kBytes + 128;
};

// This CTA's stages: tasks [t0, t1), then rope rows [r0, r1) in chunks of 16.
struct AbsSeq {
  int t0, t1, r0, r1;
  __device__ int tasks() const { return t1 - t0; }
  __device__ int stages() const { return (t1 - t0) + (r1 - r0 + kTaskRows - 1) / kTaskRows; }
};

__device__ __forceinline__ int rope_row(int r) {  // rope index -> W_QB row
  return (r / kRope) * kHeadRows + kNope + (r % kRope);
}

template <int NT>
__global__ void __launch_bounds__(kAbsThreads, 1)
    mla_absorb_kernel(const DecodeArgs a, const __grid_constant__ AbsSplit split) {
  using S = AbsSmem<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint8_t* ring = smem;
  uint8_t* xq = smem + S::oXq;
  float* q16 = reinterpret_cast<float*>(smem + S::oQ16);
  float* ss_part = reinterpret_cast<float*>(smem + S::oSs);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::oFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::oEmpty);
  uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + S::oQbar);
  uint64_t* sig = reinterpret_cast<uint64_t*>(smem + S::oSig);
  uint64_t* sfree = reinterpret_cast<uint64_t*>(smem + S::oFree);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x, P = gridDim.x;
  const int H = a.heads;
  const AbsSeq seq{split.task[i], split.task[i + 1], split.rope[i], split.rope[i + 1]};
  const int nst = seq.stages();

  if (tid == 0) {
    for (int s = 0; s < kAbsStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(qbar, kConsumerWarps);
    for (int s = 0; s < kSigRing; ++s) {
      mbar_init(&sig[s], kConsumerWarps);
      mbar_init(&sfree[s], 1);
    }
    mbar_fence_init();
    trace_stamp(a, 0);
  }
  __syncthreads();
  bool timed_out = false;

  if (warp == kConsumerWarps) {
    // ================= producer: weights only, no PDL wait ============
    for (int k = 0; k < nst; ++k) {
      const int slot = k % kAbsStages;
      uint8_t* buf = ring + slot * kTaskStage;
      if (k >= kAbsStages) {
        int ok = 1;
        if (lane == 0)
          ok = mbar_wait_bounded(&empty[slot], (uint32_t)(((k / kAbsStages) - 1) & 1), kWaitLimit)
                   ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) timed_out = true;
      }
      if (lane == 0 && k < 20) trace_stamp(a, 28 + k);
      if (k < seq.tasks()) {
        const int tk = seq.t0 + k, h = tk / kTasksPerHead, p0 = (tk % kTasksPerHead) * kTaskRows;
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], kTaskRows * kRowBytes + kTaskUkBytes);
        __syncwarp();
        if (lane < kTaskRows)
          bulk_g2s(buf + lane * kPitch, a.w_qb + ((int64_t)h * kHeadRows + p0 + lane) * kQLora,
                   kRowBytes, &full[slot]);
        else if (lane == kTaskRows)
          bulk_g2s(buf + kTaskQbBytes, a.w_uk + ((int64_t)h * kNope + p0) * kKvLora,
                   kTaskUkBytes, &full[slot]);
      } else {
        const int r = seq.r0 + (k - seq.tasks()) * kTaskRows;
        const int n = min(kTaskRows, seq.r1 - r);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * kRowBytes));
        __syncwarp();
        if (lane < n)
          bulk_g2s(buf + lane * kPitch, a.w_qb + (int64_t)rope_row(r + lane) * kQLora, kRowBytes,
                   &full[slot]);
      }
    }
    if (lane == 0)
      for (int k = max(0, nst - kAbsStages); k < nst; ++k)
        (void)mbar_wait_bounded(&full[k % kAbsStages], (uint32_t)((k / kAbsStages) & 1),
                                kWaitLimit);
  } else if (warp == kConsumerWarps + 1) {
    // ================= finisher: publish partials, close heads ========
    // Takes every task whose partials are stored (up to the signal ring):
    // one fence makes them visible GPU-wide, then one lane per task bumps
    // that head's counter (one round trip for the batch).  A task that
    // completes its head adds the head's 8 partials in task order.
    pdl_wait();
    const int ntasks = seq.tasks();
    for (int n = 0; n < ntasks;) {
      int m = 0;
      if (lane == 0) {
        if (!mbar_wait_bounded(&sig[n % kSigRing], (uint32_t)((n / kSigRing) & 1), kWaitLimit))
          timed_out = true;
        trace_stamp(a, 51);
        m = 1;
        while (m < kSigRing && n + m < ntasks &&
               mbar_try_wait(&sig[(n + m) % kSigRing], (uint32_t)(((n + m) / kSigRing) & 1)))
          ++m;
        __threadfence();  // the consumers' partial stores precede `sig`
        trace_stamp(a, 52);
      }
      m = __shfl_sync(0xFFFFFFFFu, m, 0);
      int last = 0;
      if (lane < m) {
        const int h = (seq.t0 + n + lane) / kTasksPerHead;
        last = atomicAdd(a.ready + h, 1u) == kTasksPerHead - 1;
      }
      __syncwarp();
      if (lane == 0)
        for (int j = 0; j < m; ++j) mbar_arrive(&sfree[(n + j) % kSigRing]);
      unsigned lastmask = __ballot_sync(0xFFFFFFFFu, last);
      if (lane == 0) trace_stamp(a, 48);
      if (lastmask) __threadfence();  // acquire: the other tasks' partials are visible
      if (lastmask && lane == 0) trace_stamp(a, 53);
      while (lastmask) {
        const int j = __ffs(lastmask) - 1;
        lastmask &= lastmask - 1;
        const int h = (seq.t0 + n + j) / kTasksPerHead;
        const float* part = a.partial + (int64_t)h * kTasksPerHead * NT * kKvLora;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          for (int c4 = lane; c4 < kKvLora / 4; c4 += 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int pb = 0; pb < kTasksPerHead; ++pb) {
              const float4 v = ld_cg_f32x4(part + ((int64_t)pb * NT + t) * kKvLora + 4 * c4);
              acc.x += v.x;
              acc.y += v.y;
              acc.z += v.z;
              acc.w += v.w;
            }
            if (t < a.batch) {
              uint2 o;
              o.x = pack_bf16x2(acc.x, acc.y);
              o.y = pack_bf16x2(acc.z, acc.w);
              *reinterpret_cast<uint2*>(a.q_latent + ((int64_t)t * H + h) * kKvLora + 4 * c4) = o;
            }
          }
        }
        if (lane == 0) a.ready[h] = 0u;  // re-armed for the next call
        if (lane == 0) trace_stamp(a, 49);
      }
      n += m;
    }
    if (lane == 0) trace_stamp(a, 50);
  } else {
    // ================= consumer warps 0-7 ============================
    pdl_wait();
    if (tid == 0) pdl_launch_dependents();
    // q_a RMSNorm -> xq (warps 0-5); KV insert of token i (warps 6-7)
    if (warp < 6) {
      uint4 xv[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t)
        xv[t] = t < a.batch ? *reinterpret_cast<const uint4*>(a.q_a + (int64_t)t * a.q_a_stride +
                                                               8 * tid)
                            : make_uint4(0, 0, 0, 0);
      const uint4 gv = *reinterpret_cast<const uint4*>(a.gamma_q + 8 * tid);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint32_t ww[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ss = fmaf(bf16lo(ww[k]), bf16lo(ww[k]), ss);
          ss = fmaf(bf16hi(ww[k]), bf16hi(ww[k]), ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) ss_part[t * 8 + warp] = ss;
      }
      named_barrier(kBarNorm, 192);
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float* sp = ss_part + t * 8;
        const float total = ((((sp[0] + sp[1]) + sp[2]) + sp[3]) + sp[4]) + sp[5];
        const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, 1536.0f), a.eps));
        const uint32_t ww[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
        uint4 o;
        o.x = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[0]), rr), bf16lo(gw[0])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[0]), rr), bf16hi(gw[0])));
        o.y = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[1]), rr), bf16lo(gw[1])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[1]), rr), bf16hi(gw[1])));
        o.z = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[2]), rr), bf16lo(gw[2])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[2]), rr), bf16hi(gw[2])));
        o.w = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(ww[3]), rr), bf16lo(gw[3])),
                          __fmul_rn(__fmul_rn(bf16hi(ww[3]), rr), bf16hi(gw[3])));
        if (t >= a.batch) o = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(xq + t * kPitch + 16 * tid) = o;
        if (i == 0 && a.q_c != nullptr && t < a.batch)
          *reinterpret_cast<uint4*>(a.q_c + (int64_t)t * kQLora + 8 * tid) = o;
      }
    } else {
      for (int t = i; t < NT; t += P)
        if (t < a.batch) kv_insert(a, t, tid - 192, ss_part + NT * 8);
    }
    named_barrier(kBarConsumers, kConsumers);
    if (tid == 0) trace_stamp(a, 2);

    float xr[NT][48];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(xq + t * kPitch + 2 * (256 * c + 8 * lane));
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xr[t][8 * c + 2 * k] = bf16lo(ww[k]);
          xr[t][8 * c + 2 * k + 1] = bf16hi(ww[k]);
        }
      }

    for (int k = 0; k < nst; ++k) {
      const int slot = k % kAbsStages;
      const uint8_t* buf = ring + slot * kTaskStage;
      if (!mbar_wait_bounded(&full[slot], (uint32_t)((k / kAbsStages) & 1), kWaitLimit))
        timed_out = true;
      if (tid == 0 && k < 20) trace_stamp(a, 8 + k);
      const bool task = k < seq.tasks();
      // rows w and w + 8 of the stage: FP32 dot products with xq
      const int nrows = task ? kTaskRows : min(kTaskRows, seq.r1 - (seq.r0 + (k - seq.tasks()) * kTaskRows));
      float v[2][NT];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int j = warp + kConsumerWarps * rr;
#pragma unroll
        for (int t = 0; t < NT; ++t) v[rr][t] = 0.f;
        if (j < nrows) {
          const uint8_t* rowp = buf + j * kPitch;
          float acc[NT][2];
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
          for (int c = 0; c < 6; ++c) {
            const uint4 wv = *reinterpret_cast<const uint4*>(rowp + 2 * (256 * c + 8 * lane));
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const float w0 = bf16lo(ww[kk]), w1 = bf16hi(ww[kk]);
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                acc[t][0] = fmaf(w0, xr[t][8 * c + 2 * kk], acc[t][0]);
                acc[t][1] = fmaf(w1, xr[t][8 * c + 2 * kk + 1], acc[t][1]);
              }
            }
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) v[rr][t] = warp_sum(acc[t][0] + acc[t][1]);
        }
      }
      if (!task) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (lane == 0) {
          const int r0 = seq.r0 + (k - seq.tasks()) * kTaskRows;
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int j = warp + kConsumerWarps * rr;
            if (j < nrows) {
              const int r = r0 + j;
#pragma unroll
              for (int t = 0; t < NT; ++t)
                if (t < a.batch)
                  a.q_pe[((int64_t)t * H + r / kRope) * kRope + r % kRope] = f2bf_bits(v[rr][t]);
            }
          }
        }
        continue;
      }
      // ---- task: share the 16 BF16-rounded q values, absorb them --------
      const int n = k, tk = seq.t0 + k;
      float* qb = q16 + (n & 1) * NT * kTaskRows;
      if (lane == 0) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
          for (int t = 0; t < NT; ++t) qb[t * kTaskRows + warp + kConsumerWarps * rr] = bf_round(v[rr][t]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qbar);
      if (!mbar_wait_bounded(qbar, (uint32_t)(n & 1), kWaitLimit)) timed_out = true;
      // this lane: latent columns c, c + 1 with c = 64 w + 2 lane
      const int c = 64 * warp + 2 * lane;
      const uint8_t* uk = buf + kTaskQbBytes;
      float acc[NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.f;
#pragma unroll
      for (int p = 0; p < kTaskRows; ++p) {
        const uint32_t wv = *reinterpret_cast<const uint32_t*>(uk + p * (kKvLora * 2) + 2 * c);
        const float w0 = bf16lo(wv), w1 = bf16hi(wv);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          acc[t][0] = fmaf(qb[t * kTaskRows + p], w0, acc[t][0]);
          acc[t][1] = fmaf(qb[t * kTaskRows + p], w1, acc[t][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // W_QB and W_UK of the slot are read
      float* part = a.partial + ((int64_t)tk * NT) * kKvLora;
#pragma unroll
      for (int t = 0; t < NT; ++t)
        *reinterpret_cast<float2*>(part + (int64_t)t * kKvLora + c) = make_float2(acc[t][0], acc[t][1]);
      // signal the finisher (its ring slot must have been consumed)
      __syncwarp();
      if (lane == 0) {
        if (n >= kSigRing &&
            !mbar_wait_bounded(&sfree[n % kSigRing], (uint32_t)(((n / kSigRing) - 1) & 1), kWaitLimit))
          timed_out = true;
        mbar_arrive(&sig[n % kSigRing]);
      }
    }
    if (tid == 0) trace_stamp(a, 6);
  }

  if (timed_out) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  __syncthreads();
  if (tid == 0) trace_stamp(a, 7);
}

template <int NT, bool MMA>
cudaError_t launch_one(const DecodeArgs& a, const CUtensorMap* map, int num_sms,
                       cudaStream_t stream) {
  using S = Smem<NT, MMA>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms / a.groups), (unsigned)a.groups, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = S::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_fused_kernel<NT, MMA>, a, *map);
}

template <int NT, bool MMA>
cudaError_t prepare_one() {
  using S = Smem<NT, MMA>;
  static_assert(S::kAlloc <= 232448, "shared memory budget");
  return cudaFuncSetAttribute(mla_fused_kernel<NT, MMA>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
}

}  // namespace

int tokens_per_cta(int batch, bool mma) {
  if (!mma) return batch <= 1 ? 1 : 2;
  return batch <= 8 ? 8 : 16;
}

size_t scratch_qn_elems(int heads) { return (size_t)(MLA_MAX_BATCH + 16) * heads * kNope; }
size_t scratch_ready_elems(int heads) { return (size_t)(MLA_MAX_BATCH / 8 + 2) * heads; }

__global__ void repack_w_uk_kernel(const uint16_t* __restrict__ w_uk, uint8_t* __restrict__ dst,
                                   int heads) {
  const int64_t n = (int64_t)heads * kUkUnitsPerHead * kNope * 8;  // 16-byte chunks
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(e % 8);
    const int p = (int)((e / 8) % kNope);
    const int cb = (int)((e / (8 * kNope)) % kUkUnitsPerHead);
    const int h = (int)(e / (8 * kNope * kUkUnitsPerHead));
    const uint4 v = *reinterpret_cast<const uint4*>(
        w_uk + ((int64_t)h * kNope + p) * kKvLora + cb * kUkCols + 8 * j);
    *reinterpret_cast<uint4*>(dst + ((int64_t)(h * kUkUnitsPerHead + cb) * kNope + p) * 128 +
                              16 * (j ^ (p & 7))) = v;
  }
}

cudaError_t repack_w_uk(const uint16_t* w_uk, uint8_t* dst, int heads, cudaStream_t stream) {
  repack_w_uk_kernel<<<256, 256, 0, stream>>>(w_uk, dst, heads);
  return cudaGetLastError();
}

void make_abs_split(int heads, int ctas, AbsSplit* sp) {
  // tasks: even split; rope rows: fill each CTA up to an even share of bytes
  const int64_t tasks = (int64_t)heads * kTasksPerHead, rope = (int64_t)heads * kRope;
  const int64_t tb = kTaskRows * kRowBytes + kTaskUkBytes, rb = kRowBytes;
  const int64_t total = tasks * tb + rope * rb;
  int prev = 0;
  for (int i = 0; i <= ctas; ++i) {
    const int64_t t = tasks * i / ctas;
    sp->task[i] = (uint16_t)t;
    int64_t r = (total * i / ctas - t * tb + rb / 2) / rb;
    if (r < prev) r = prev;
    if (r > rope) r = rope;
    if (i == ctas) r = rope;
    sp->rope[i] = (uint16_t)r;
    prev = (int)r;
  }
}

template <int NT>
cudaError_t launch_abs(const DecodeArgs& a, const AbsSplit& sp, int ctas, cudaStream_t stream) {
  using S = AbsSmem<NT>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kAbsThreads, 1, 1);
  cfg.dynamicSmemBytes = S::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_absorb_kernel<NT>, a, sp);
}

template <int NT>
cudaError_t prepare_abs() {
  using S = AbsSmem<NT>;
  static_assert(S::kAlloc <= 232448, "shared memory budget");
  return cudaFuncSetAttribute(mla_absorb_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              S::kAlloc);
}

cudaError_t prepare_fused_kernels() {
  cudaError_t e;
  if ((e = prepare_abs<1>()) != cudaSuccess) return e;
  if ((e = prepare_abs<2>()) != cudaSuccess) return e;
  if ((e = prepare_one<1, false>()) != cudaSuccess) return e;
  if ((e = prepare_one<2, false>()) != cudaSuccess) return e;
  if ((e = prepare_one<8, true>()) != cudaSuccess) return e;
  if ((e = prepare_one<16, true>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_absorb(const DecodeArgs& a, const AbsSplit& sp, int nt, int ctas,
                          cudaStream_t stream) {
  if (nt == 1) return launch_abs<1>(a, sp, ctas, stream);
  if (nt == 2) return launch_abs<2>(a, sp, ctas, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fused(const DecodeArgs& a, const CUtensorMap* map, int nt, bool mma,
                         int num_sms, cudaStream_t stream) {
  if (!mma) {
    if (nt == 1) return launch_one<1, false>(a, map, num_sms, stream);
    if (nt == 2) return launch_one<2, false>(a, map, num_sms, stream);
  } else {
    if (nt == 8) return launch_one<8, true>(a, map, num_sms, stream);
    if (nt == 16) return launch_one<16, true>(a, map, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mla
