// mla_small.cu - the decode step for up to eight tokens on FP32 FMAs.
//
// What it computes is the step of page "mla.query", class MlaQuery (method
// kernel, the small-batch path, and insert / insert_ds / insert_nvfp4 /
// store_qc): q_a RMSNorm -> xq (q_c), Q_B rows -> q (BF16, FP32 accumulate),
// rope rows -> q_pe, nope rows through W_UK -> q_latent, and the KV insert.
//
// GB300 design.  With one or two tokens a weight element feeds one or two
// FMAs, so the projection is no dense contraction: plain FP32 FMAs keep up
// with the stream, and the kernel is shaped around the stream instead.  It
// is built for 1, 2, 4 and 8 tokens (the last two so that the dispatch
// between FP32 FMAs and tensor cores rests on measurements at every batch
// up to 8).
//  * Clusters of C CTAs (2, 4 or 8) own whole heads (at most two per
//    cluster); rank r takes nope rows [r 128/C, (r+1) 128/C) of each head and
//    the same rows of W_UK, and rope rows fill every CTA to an even byte
//    share.  A stage is 16 consecutive Q_B rows (48 KiB) plus, for nope
//    rows, their 16 W_UK rows (16 KiB), one 1-D bulk copy per row issued by
//    separate lanes.  The static weights are copied before the programmatic-
//    dependent-launch wait, as the page's class docstring has them: a 3-stage
//    ring (192 KiB, one CTA per SM; two stages at 8 tokens) holds a small
//    head count's whole share (16 heads: at most 128 KiB a CTA) before the
//    wait ends.  (A ring of about 100 KiB measured slower, 10.3 against
//    9.3 us at 64 heads with 8-row stages.  It does not let the next step's
//    CTA share the SM on its own: 288 threads at 112 registers fill the
//    register file for one CTA; capped at 96 registers two CTAs did share
//    each SM, and the spills made it 10.7 us.)
//  * Warp w computes rows w and w + 8 of a stage, their chains interleaved:
//    each lane dots 48 of a row's 1536 values with the normalised xq (one
//    token: kept in registers as BF16 pairs; more tokens: each normalised
//    by one warp into shared memory), then the warp adds the lanes.  The 16
//    BF16-rounded nope q values go through shared memory to all 256 threads,
//    and thread t adds their products with W_UK columns 2t, 2t + 1 into its
//    FP32 absorption sums.  (Stages of 8 rows, one a warp, measured slower:
//    the shuffles and the barrier of a stage are paid per row; 9.32 against
//    8.45 us at 64 heads, 5.24 against 4.89 at 16.)
//  * After a head's last stage each thread sends the sums of columns another
//    rank owns (rank r owns columns [r 512/C, (r+1) 512/C)) into that CTA's
//    shared memory (st.async, counted on its mbarrier); each owner adds the
//    C partials in rank order (row order of the head) and writes q_latent.
//    No L2 round trip closes a head, which is where this kernel beats the
//    tensor-core partials kernel at small head counts.
// Every wait is bounded (MLA_DEVERR_TIMEOUT instead of a hang).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdio>

#include "../../include/mla_query.h"
#include "mla_common.cuh"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

// Q_B rows per stage: MLA_SMALL_ROWS_PER_WARP (1 or 2) per consumer warp.
#ifndef MLA_SMALL_ROWS_PER_WARP
#define MLA_SMALL_ROWS_PER_WARP 2
#endif
constexpr int kSmRowsPerWarp = MLA_SMALL_ROWS_PER_WARP;
constexpr int kSmRows = 8 * kSmRowsPerWarp;
static_assert(kSmRowsPerWarp == 1 || kSmRowsPerWarp == 2, "rows per warp");
static_assert(2 * kSmRows <= 32, "one producer lane per copy of a stage");
constexpr int kSmQbBytes = kSmRows * kRowBytes;    // 24 or 48 KiB
constexpr int kSmUkBytes = kSmRows * kKvLora * 2;  // 8 or 16 KiB
constexpr int kSmStage = kSmQbBytes + kSmUkBytes;  // 32 or 64 KiB
#ifndef MLA_SMALL_SLOTS
#define MLA_SMALL_SLOTS 3
#endif
constexpr int kSmSlots = MLA_SMALL_SLOTS;
#ifndef MLA_SMALL_PREFETCH
#define MLA_SMALL_PREFETCH 0
#endif
constexpr bool kSmPrefetch = MLA_SMALL_PREFETCH != 0;
constexpr int kSmThreads = kConsumers + 32;        // 8 consumer warps + the producer warp

template <int NT, int C>
struct SmallSmem {
  // ring slots: three, two at 8 tokens (their partials and xq rows take the
  // third slot's shared memory)
  static constexpr int kSlots = NT >= 8 ? 2 : kSmSlots;
  static constexpr int kCols = kKvLora / C;            // latent columns a rank owns
  static constexpr int kStagesPerHead = kNope / C / kSmRows;
  static constexpr int kRecvHead = C * kCols * NT * 4;  // [rank][column][token] FP32
  static constexpr int kRecvBytesIn = (C - 1) * kCols * NT * 4;  // what the peers send
  static constexpr int oRing = 0;
  static constexpr int oRecv = kSlots * kSmStage;       // [2 heads][kRecvHead]
  static constexpr int oQv = oRecv + 2 * kRecvHead;     // [2][kSmRows][NT] FP32
  static constexpr int oFull = oQv + 2 * kSmRows * NT * 4;
  static constexpr int oEmpty = oFull + kSlots * 8;
  static constexpr int oRbar = oEmpty + kSlots * 8;     // [2] received partials
  static constexpr int oQbar = oRbar + 16;              // [2] q values of a stage written
  // two or more tokens: their xq rows in shared memory [NT][1536] BF16 (one
  // token keeps its 48 values a lane in registers)
  static constexpr int kXsBytes = NT > 1 ? NT * kRowBytes : 0;
  static constexpr int oXs = oQbar + 16;
  static constexpr int kBytes = oXs + kXsBytes;
  static constexpr int kAlloc = kBytes + 128;
  static_assert(kStagesPerHead * kSmRows * C == kNope, "stages per head");
  static_assert(kAlloc <= 227 * 1024, "shared memory of one CTA");
};

// This CTA's stages: the nope stages of each head of its cluster, then its
// rope rows in stages of up to kSmRows.
template <int C>
struct SmallSeq {
  static constexpr int kPerHead = kNope / C / kSmRows;
  int h0, nh, rank, r0, r1;
  __device__ int nope() const { return kPerHead * nh; }
  __device__ int stages() const { return nope() + (r1 - r0 + kSmRows - 1) / kSmRows; }
  __device__ int head(int k) const { return h0 + k / kPerHead; }
  __device__ int p0(int k) const { return (kNope / C) * rank + kSmRows * (k % kPerHead); }
};

__device__ __forceinline__ int small_rope_row(int r) {  // rope index -> W_QB row
  return (r / kRope) * kHeadRows + kNope + (r % kRope);
}

// Stage k of a CTA into L2 (no shared memory, no completion): its Q_B rows
// and, for nope rows, their W_UK rows; rope rows may span two heads.
template <int C>
__device__ __forceinline__ void small_prefetch_stage(const DecodeArgs& a, const SmallSeq<C>& seq,
                                                     int k) {
  if (k < seq.nope()) {
    const int h = seq.head(k), p0 = seq.p0(k);
    bulk_prefetch_l2(a.w_qb + ((int64_t)h * kHeadRows + p0) * kQLora, kSmQbBytes);
    bulk_prefetch_l2(a.w_uk + ((int64_t)h * kNope + p0) * kKvLora, kSmUkBytes);
  } else {
    const int r = seq.r0 + (k - seq.nope()) * kSmRows;
    const int n = min(kSmRows, seq.r1 - r);
    const int n1 = min(n, kRope - r % kRope);
    bulk_prefetch_l2(a.w_qb + (int64_t)small_rope_row(r) * kQLora, (uint32_t)(n1 * kRowBytes));
    if (n > n1)
      bulk_prefetch_l2(a.w_qb + (int64_t)small_rope_row(r + n1) * kQLora,
                       (uint32_t)((n - n1) * kRowBytes));
  }
}

__device__ __forceinline__ void st_async_v2(uint32_t raddr, float x, float y, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
          raddr),
      "f"(x), "f"(y), "r"(rbar)
      : "memory");
}

// FP32 dot products of one 8-value chunk of a Q_B row with the same chunk of
// each token's xq (BF16 pairs): pair e of the chunk goes to accumulator e, so
// four independent FMA chains run side by side.
template <int NT>
__device__ __forceinline__ void dot_chunk(const uint4 w, const uint4 (&x)[NT], float (&s)[NT][4]) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const uint32_t xx[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[t][e] = fmaf(bf16lo(ww[e]), bf16lo(xx[e]), s[t][e]);
      s[t][e] = fmaf(bf16hi(ww[e]), bf16hi(xx[e]), s[t][e]);
    }
  }
}

// One CTA an SM (the ring takes most of the shared memory), so up to
// 65536 / 288 = 227 registers a thread would fit; for one or two tokens 112
// measured faster than 160 (8.45 against 8.60 us at 64 heads, one spill of
// 8 bytes at C = 8); four and eight tokens take 168 (their accumulators).
#ifndef MLA_SMALL_MAXNREG
#define MLA_SMALL_MAXNREG 112
#endif
template <int NT, int C>
__global__ void __maxnreg__(NT >= 4 ? 168 : MLA_SMALL_MAXNREG)
    mla_small_kernel(const DecodeArgs a, const __grid_constant__ SmallSplit split) {
  using S = SmallSmem<NT, C>;
  constexpr int SL = S::kSlots;
  const uint64_t t_entry = trace_now();  // slot 1 of a trace build
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint8_t* ring = smem + S::oRing;
  float* qv = reinterpret_cast<float*>(smem + S::oQv);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::oFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::oEmpty);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + S::oRbar);
  uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + S::oQbar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x;
  const int g = i / C, rank = i % C;  // cluster (C, 1, 1): rank = blockIdx.x % C
  const SmallSeq<C> seq{split.head[g], split.head[g + 1] - split.head[g], rank, split.rope[i],
                        split.rope[i + 1]};
  const int nst = seq.stages();
  bool timed_out = false;

  if (tid == 0) {
    for (int s = 0; s < SL; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&rbar[0], 1);
    mbar_init(&rbar[1], 1);
    mbar_init(&qbar[0], kConsumerWarps);
    mbar_init(&qbar[1], kConsumerWarps);
    // the peers' partials of head j land in recv[j]: armed before this CTA
    // arrives at the cluster barrier, so no byte can arrive before its count
    // is expected
    for (int j = 0; j < seq.nh; ++j) mbar_arrive_expect_tx(&rbar[j], S::kRecvBytesIn);
    mbar_fence_init();
    pdl_launch_dependents();
    trace_stamp(a, 0);
    trace_put(a, 1, t_entry);
  }
  __syncthreads();
  // The cluster barrier's first phase orders the peers' rbar before the
  // first remote store: every thread arrives now (relaxed: the mbarrier-init
  // fence publishes the barriers; a release arrive measured slower), the
  // consumers wait after the q_a prologue, the producer after its last copy.
  // The producer starts copying without waiting for the cluster.  (Other
  // start-ups measured: the producer initialising its own ring barriers and
  // issuing before the CTA meets, with or without holding its second stage
  // until the programmatic-dependent-launch wait: 8.83 and 8.48 against
  // 8.47 us at 64 heads, 6.14 and 5.88 against 5.72 at 32; more copies in
  // flight when the q_a row is loaded delay the prologue.)
  cluster_arrive_relaxed();

  if (warp == kConsumerWarps) {
    // ================= producer: weights only, no PDL wait ============
    // A stage's copies are issued by separate lanes in one instruction (Q_B
    // rows below lane kSmRows, their W_UK rows from there): copies one
    // thread issues complete one after another, copies of different threads
    // side by side.  A nope stage goes out as one copy per row, or, where the
    // CTA's whole share is at most two stages, one copy per two rows: then
    // both stages' copies are out at once (at 16 heads the second stage's
    // row copies left 1.15 us after the first's; 4.29 against 4.72 us a
    // step), while a longer stream keeps more copies in flight with one row
    // each (two rows a copy measured 9.70 against 8.30 us at 64 heads).
    if (lane == 0) trace_stamp(a, 4);  // the producer starts
    const uint64_t pol = l2_policy_evict_first();
    const int rpc = nst <= 2 ? 2 : 1;  // nope rows per copy
    if (kSmPrefetch && lane == 0)
      for (int k = SL; k < min(nst, 2 * SL); ++k) small_prefetch_stage<C>(a, seq, k);
    int issued = 0;
    for (int k = 0; k < nst; ++k) {
      const int slot = k % SL;
      uint8_t* buf = ring + slot * kSmStage;
      int ok = 1;
      if (k >= SL && lane == 0)
        ok = mbar_wait_bounded(&empty[slot], (uint32_t)(((k / SL) - 1) & 1), kWaitLimit);
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
        timed_out = true;  // the consumers stopped: issue nothing more
        break;
      }
      issued = k + 1;
      if (lane == 0 && k < 20) trace_stamp(a, 28 + k);  // stage k issued
      if (kSmPrefetch && lane == 0 && k >= SL && k + SL < nst)
        small_prefetch_stage<C>(a, seq, k + SL);
      if (k < seq.nope()) {
        const int h = seq.head(k), p0 = seq.p0(k);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], kSmStage);
        __syncwarp();
        if (!MLA_IN_BOUNDS(a, h >= 0 && h < a.heads && p0 >= 0 && p0 + kSmRows <= kNope, 10) ||
            !MLA_IN_BOUNDS(a, slot >= 0 && slot < SL, 11)) {
        } else if (lane < kSmRows / rpc)
          bulk_g2s_hint(buf + lane * rpc * kRowBytes,
                        a.w_qb + ((int64_t)h * kHeadRows + p0 + lane * rpc) * kQLora,
                        (uint32_t)(rpc * kRowBytes), &full[slot], pol);
        else if (lane >= kSmRows && lane < kSmRows + kSmRows / rpc)
          bulk_g2s_hint(buf + kSmQbBytes + (lane - kSmRows) * rpc * kKvLora * 2,
                        a.w_uk + ((int64_t)h * kNope + p0 + (lane - kSmRows) * rpc) * kKvLora,
                        (uint32_t)(rpc * kKvLora * 2), &full[slot], pol);
      } else {
        const int r = seq.r0 + (k - seq.nope()) * kSmRows;
        const int n = min(kSmRows, seq.r1 - r);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * kRowBytes));
        __syncwarp();
        if (lane < n && MLA_IN_BOUNDS(a, r + lane >= 0 && r + lane < a.heads * kRope, 10))
          bulk_g2s_hint(buf + lane * kRowBytes, a.w_qb + (int64_t)small_rope_row(r + lane) * kQLora,
                        kRowBytes, &full[slot], pol);
      }
    }
    // every copy issued lands before the CTA may leave
    if (lane == 0)
      for (int k = issued > SL ? issued - SL : 0; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % SL], (uint32_t)((k / SL) & 1), kWaitLimit);
    cluster_wait_acquire();
  } else {
    // ================= consumer warps 0-7 ============================
    // gamma_q is a weight: one token loads it before the wait (with more
    // tokens each normalising warp reads it from L2 as it goes)
    uint4 gq[NT == 1 ? 6 : 1];
    if constexpr (NT == 1) {
#pragma unroll
      for (int j = 0; j < 6; ++j)
        gq[j] = *reinterpret_cast<const uint4*>(a.gamma_q + 8 * (lane + 32 * j));
    }
    pdl_wait();
    if (tid == 0) trace_stamp(a, 3);
    // The KV row of token i (CTA i < B): its loads go out with the q_a row's,
    // its arithmetic after the normalisation; a CTA inserts at most one
    // token (B <= 8 < P).
    const bool kv_here = warp == kConsumerWarps - 1 && i < a.batch;
    KvWarpLoads kvl;
    if (kv_here) kvl = kv_insert_warp_load(a, i, lane);
    // q_a RMSNorm: lane l holds columns 8 (l + 32 j) .. + 7, j < 6, of a
    // token's xq as BF16 pairs.  One token: every warp normalises it and
    // keeps it in registers.  More tokens: warp w normalises tokens w,
    // w + 8, .. into shared memory.
    uint4 xq1[6];  // one token: its xq
    for (int t = NT == 1 ? 0 : warp; t < NT; t += NT == 1 ? 1 : kConsumerWarps) {
      uint4 x[6];
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 6; ++j) {
        x[j] = t < a.batch ? *reinterpret_cast<const uint4*>(a.q_a + (int64_t)t * a.q_a_stride +
                                                             8 * (lane + 32 * j))
                           : make_uint4(0, 0, 0, 0);
        const uint32_t vv[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ss = fmaf(bf16lo(vv[e]), bf16lo(vv[e]), ss);
          ss = fmaf(bf16hi(vv[e]), bf16hi(vv[e]), ss);
        }
      }
      ss = warp_sum(ss);
      const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, 1536.0f), a.eps));
#pragma unroll
      for (int j = 0; j < 6; ++j) {
        const uint4 gj = NT == 1 ? gq[NT == 1 ? j : 0]
                                 : *reinterpret_cast<const uint4*>(a.gamma_q + 8 * (lane + 32 * j));
        const uint32_t gw[4] = {gj.x, gj.y, gj.z, gj.w};
        const uint32_t vv[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = rms_scale_bf16x2(vv[e], rr, gw[e]);
        x[j] = make_uint4(o[0], o[1], o[2], o[3]);
        if constexpr (NT == 1)
          xq1[j] = x[j];
        else
          *reinterpret_cast<uint4*>(smem + S::oXs + t * kRowBytes + 16 * (lane + 32 * j)) = x[j];
        if (i == 0 && (NT > 1 || warp == 0) && a.q_c != nullptr && t < a.batch)
          *reinterpret_cast<uint4*>(a.q_c + (int64_t)t * kQLora + 8 * (lane + 32 * j)) = x[j];
      }
    }
    if (kv_here) kv_insert_warp_loaded(a, lane, kvl);
    if constexpr (NT > 1) named_barrier(4, kConsumers);  // xq rows written (before any wait)
    if (tid == 0) trace_stamp(a, 2);
    cluster_wait_acquire();  // every peer's rbar armed (long since, by now)
    const float qsi = load_qsi(a);

    // Thread tid's latent columns 2 tid, 2 tid + 1 belong to rank owner.
    const int owner = tid * C / kConsumers;
    const int lc = 2 * tid - owner * S::kCols;  // column within the owner's range
    float acc[NT][2];    // absorption sums of the current head
    float keep[2][NT][2];  // owned sums of heads 0 and 1 of the cluster
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      acc[t][0] = acc[t][1] = 0.f;
      keep[0][t][0] = keep[0][t][1] = keep[1][t][0] = keep[1][t][1] = 0.f;
    }

    for (int k = 0; k < nst; ++k) {
      const int slot = k % SL;
      const uint8_t* buf = ring + slot * kSmStage;
      // a stage that never arrives ends the loop; the other warps' barrier
      // waits below are then bounded by the same limit
      if (!mbar_wait_bounded(&full[slot], (uint32_t)((k / SL) & 1), kWaitLimit)) {
        timed_out = true;
        break;
      }
      if (tid == 0 && k < 20) trace_stamp(a, 8 + k);  // stage k's data seen
      const bool nope = k < seq.nope();
      const int r = seq.r0 + (k - seq.nope()) * kSmRows;  // first rope row (rope stages)
      const int rows = nope ? kSmRows : min(kSmRows, seq.r1 - r);
      // ---- Q_B rows warp + 8 i of the stage: 48 products per lane, then
      // the warp; the rows' chains interleave
      float s[kSmRowsPerWarp][NT];
      {
        float s4[kSmRowsPerWarp][NT][4];
#pragma unroll
        for (int i = 0; i < kSmRowsPerWarp; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) s4[i][t][0] = s4[i][t][1] = s4[i][t][2] = s4[i][t][3] = 0.f;
#pragma unroll
        for (int j = 0; j < 6; ++j) {
          uint4 xj[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t)
            xj[t] = NT == 1 ? xq1[j]
                            : *reinterpret_cast<const uint4*>(smem + S::oXs + t * kRowBytes +
                                                               16 * (lane + 32 * j));
#pragma unroll
          for (int i = 0; i < kSmRowsPerWarp; ++i)
            if (warp + 8 * i < rows)
              dot_chunk<NT>(reinterpret_cast<const uint4*>(buf + (warp + 8 * i) * kRowBytes)[lane + 32 * j],
                            xj, s4[i]);
        }
#pragma unroll
        for (int i = 0; i < kSmRowsPerWarp; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            s[i][t] = warp_sum((s4[i][t][0] + s4[i][t][1]) + (s4[i][t][2] + s4[i][t][3]));
      }
      if (!nope) {
        // ---- rope rows -> q_pe ------------------------------------------
#pragma unroll
        for (int i = 0; i < kSmRowsPerWarp; ++i) {
          if (warp + 8 * i >= rows) continue;
          const int rr_ = r + warp + 8 * i;
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (lane == t && t < a.batch &&
                MLA_IN_BOUNDS(a, rr_ >= 0 && rr_ < a.heads * kRope, 13))
              put_q(a, a.q_pe,
                    (int64_t)t * a.qp_ts + (int64_t)(rr_ / kRope) * a.qp_hs + rr_ % kRope,
                    s[i][t], qsi);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (tid == 0 && k < 14) trace_stamp(a, 48 + k);  // stage k done
        continue;
      }
      // ---- nope rows: BF16 q of the stage's rows to every thread --------
      // (nope stages are k = 0 .. nope() - 1: buffer k & 1, its use k >> 1)
      float* qk = qv + (k & 1) * kSmRows * NT;
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kSmRowsPerWarp; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) qk[(warp + 8 * i) * NT + t] = bf_round(s[i][t]);
        mbar_arrive(&qbar[k & 1]);
      }
      if (!mbar_wait_bounded(&qbar[k & 1], (uint32_t)((k >> 1) & 1), kWaitLimit))
        timed_out = true;
      // ---- absorption: W_UK rows p0.., columns 2 tid and 2 tid + 1 ------
      const uint32_t* uk = reinterpret_cast<const uint32_t*>(buf + kSmQbBytes);
#pragma unroll
      for (int p = 0; p < kSmRows; ++p) {
        const uint32_t w2 = uk[p * (kKvLora / 2) + tid];
        const float w0 = bf16lo(w2), w1 = bf16hi(w2);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float qq = qk[p * NT + t];
          acc[t][0] = fmaf(qq, w0, acc[t][0]);
          acc[t][1] = fmaf(qq, w1, acc[t][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // W_QB and W_UK of the slot are read
      if (tid == 0 && k < 14) trace_stamp(a, 48 + k);  // stage k done
      if (k % S::kStagesPerHead == S::kStagesPerHead - 1) {
        // the head's last stage here: columns of other ranks go to them
        const int j = k / S::kStagesPerHead;
        if (owner == rank) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (j == 0) {
              keep[0][t][0] = acc[t][0];
              keep[0][t][1] = acc[t][1];
            } else {
              keep[1][t][0] = acc[t][0];
              keep[1][t][1] = acc[t][1];
            }
          }
        } else if (MLA_IN_BOUNDS(a, j >= 0 && j < 2 && owner >= 0 && owner < C && lc >= 0 &&
                                          lc + 2 <= S::kCols, 12)) {
          // owner's recv[j][rank][lc .. lc + 1][token]
          const uint32_t peer = (uint32_t)owner;
          const uint32_t rb = mapa_shared(smem_u32(&rbar[j]), peer);
          const uint32_t dst = smem_u32(smem + S::oRecv + j * S::kRecvHead +
                                        ((rank * S::kCols + lc) * NT) * 4);
          if constexpr (NT == 1) {
            st_async_v2(mapa_shared(dst, peer), acc[0][0], acc[0][1], rb);
          } else {
            // element e of the 2 NT: column e / NT, token e % NT
#pragma unroll
            for (int q = 0; q < NT / 2; ++q) {
              float f[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) f[e] = acc[(4 * q + e) % NT][(4 * q + e) / NT];
              st_async_v4(mapa_shared(dst + 16 * q, peer), f[0], f[1], f[2], f[3], rb);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = 0.f;
      }
    }
    if (tid == 0) trace_stamp(a, 6);

    // ---- owned columns: the C partials in rank order -> q_latent --------
    // (columns 2 tid, 2 tid + 1 are the same in every CTA of the cluster;
    // only their owner holds every partial)
    for (int j = 0; j < seq.nh && owner == rank; ++j) {
      if (!mbar_wait_bounded(&rbar[j], 0u, kWaitLimit)) timed_out = true;
      const float* rv = reinterpret_cast<const float*>(smem + S::oRecv + j * S::kRecvHead);
      float v[NT][2];
#pragma unroll
      for (int t = 0; t < NT; ++t) v[t][0] = v[t][1] = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float k0 = j == 0 ? keep[0][t][0] : keep[1][t][0];
          const float k1 = j == 0 ? keep[0][t][1] : keep[1][t][1];
          const float p0 = c == rank ? k0 : rv[((c * S::kCols + lc) * NT) + t];
          const float p1 = c == rank ? k1 : rv[((c * S::kCols + lc + 1) * NT) + t];
          v[t][0] = c == 0 ? p0 : v[t][0] + p0;
          v[t][1] = c == 0 ? p1 : v[t][1] + p1;
        }
      }
      const int h = seq.h0 + j;
      if (!MLA_IN_BOUNDS(a, h >= 0 && h < a.heads && 2 * tid + 2 <= kKvLora, 13)) break;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t >= a.batch) continue;
        const int64_t idx = (int64_t)t * a.ql_ts + (int64_t)h * a.ql_hs + 2 * tid;
        if (a.q_scale_inv == nullptr)
          *reinterpret_cast<uint32_t*>(a.q_latent + idx) = pack_bf16x2(v[t][0], v[t][1]);
        else
          *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.q_latent) + idx) =
              (uint16_t)(q_fp8(v[t][0], qsi) | ((uint16_t)q_fp8(v[t][1], qsi) << 8));
      }
    }
  }

  if (timed_out) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  __syncthreads();
  cluster_sync_relaxed();
  if (tid == 0) trace_stamp(a, 7);
}

template <int NT, int C>
cudaLaunchConfig_t small_config(int ctas, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kSmThreads, 1, 1);
  cfg.dynamicSmemBytes = SmallSmem<NT, C>::kAlloc;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // spread the clusters over the SMs, one CTA of this kernel per SM
  attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
  attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicySpread;
  attr[2].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[2].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 3;
  return cfg;
}

template <int NT, int C>
cudaError_t prepare_small_one() {
  // (the limit covers the one-per-SM occupancy query below; a launch asks
  // for kAlloc)
  cudaError_t e = cudaFuncSetAttribute(
      mla_small_kernel<NT, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      SmallSmem<NT, C>::kAlloc > 120 * 1024 ? SmallSmem<NT, C>::kAlloc : 120 * 1024);
  if (e != cudaSuccess) return e;
  // the whole unified memory as shared memory (the ring and the partials
  // take up to about 220 KiB)
  e = cudaFuncSetAttribute(mla_small_kernel<NT, C>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
#ifdef MLA_DEBUG_SPLIT
  if (e == cudaSuccess) {
    int blocks = 0, clusters = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, mla_small_kernel<NT, C>, kSmThreads,
                                                  SmallSmem<NT, C>::kAlloc);
    cudaLaunchAttribute attr[3];
    cudaLaunchConfig_t cfg = small_config<NT, C>(C, nullptr, attr);
    cfg.numAttrs = 1;
    cudaOccupancyMaxActiveClusters(&clusters, mla_small_kernel<NT, C>, &cfg);
    cudaGetLastError();
    fprintf(stderr, "small kernel NT %d C %d: %d bytes, %d CTAs an SM, %d clusters\n", NT, C,
            SmallSmem<NT, C>::kAlloc, blocks, clusters);
  }
#endif
  return e;
}

// Clusters that fit with one CTA per SM: the occupancy of a CTA asking for
// more than half an SM's shared memory (a grid takes one CTA per SM).
template <int NT, int C>
int small_max_clusters_one() {
  cudaLaunchAttribute attr[3];
  cudaLaunchConfig_t cfg = small_config<NT, C>(C, nullptr, attr);
  cfg.numAttrs = 1;  // the cluster shape only
  if (cfg.dynamicSmemBytes < 120 * 1024) cfg.dynamicSmemBytes = 120 * 1024;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, mla_small_kernel<NT, C>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

template <int NT, int C>
cudaError_t launch_small_one(const DecodeArgs& a, const SmallSplit& sp, int ctas,
                             cudaStream_t stream) {
  cudaLaunchAttribute attr[3];
  cudaLaunchConfig_t cfg = small_config<NT, C>(ctas, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_small_kernel<NT, C>, a, sp);
}

template <int NT>
cudaError_t prepare_small_nt() {
  cudaError_t e;
  if ((e = prepare_small_one<NT, 2>()) != cudaSuccess) return e;
  if ((e = prepare_small_one<NT, 4>()) != cudaSuccess) return e;
  return prepare_small_one<NT, 8>();
}

template <int NT>
int small_max_clusters_nt(int cluster) {
  return cluster == 2 ? small_max_clusters_one<NT, 2>()
         : cluster == 4 ? small_max_clusters_one<NT, 4>()
         : cluster == 8 ? small_max_clusters_one<NT, 8>()
                        : 0;
}

template <int NT>
cudaError_t launch_small_nt(const DecodeArgs& a, const SmallSplit& sp, int ctas,
                            cudaStream_t stream) {
  switch (sp.cluster) {
    case 2: return launch_small_one<NT, 2>(a, sp, ctas, stream);
    case 4: return launch_small_one<NT, 4>(a, sp, ctas, stream);
    case 8: return launch_small_one<NT, 8>(a, sp, ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t prepare_small_kernels() {
  cudaError_t e;
  if ((e = prepare_small_nt<1>()) != cudaSuccess) return e;
  if ((e = prepare_small_nt<2>()) != cudaSuccess) return e;
  if ((e = prepare_small_nt<4>()) != cudaSuccess) return e;
  return prepare_small_nt<8>();
}

int small_kernel_max_clusters(int cluster, int nt) {
  switch (nt) {
    case 1: return small_max_clusters_nt<1>(cluster);
    case 2: return small_max_clusters_nt<2>(cluster);
    case 4: return small_max_clusters_nt<4>(cluster);
    case 8: return small_max_clusters_nt<8>(cluster);
    default: return 0;
  }
}

cudaError_t launch_small(const DecodeArgs& a, const SmallSplit& sp, int ctas, int nt,
                         cudaStream_t stream) {
  switch (nt) {
    case 1: return launch_small_nt<1>(a, sp, ctas, stream);
    case 2: return launch_small_nt<2>(a, sp, ctas, stream);
    case 4: return launch_small_nt<4>(a, sp, ctas, stream);
    case 8: return launch_small_nt<8>(a, sp, ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
