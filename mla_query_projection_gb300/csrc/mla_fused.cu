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
#include "mla_common.cuh"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {


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
  if (!MLA_IN_BOUNDS(a, grp >= 0 && (grp + 1) * NT <= MLA_MAX_BATCH + 16, 17)) return;
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
        o.x = rms_scale_bf16x2(ww[0], rr, gw[0]);
        o.y = rms_scale_bf16x2(ww[1], rr, gw[1]);
        o.z = rms_scale_bf16x2(ww[2], rr, gw[2]);
        o.w = rms_scale_bf16x2(ww[3], rr, gw[3]);
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
// Absorbing kernels: tasks, with no hand-off between CTAs.
//
// A "task" is 16 consecutive nope rows of one head (48 KiB of W_QB) together
// with the same 16 rows of that head's W_UK (16 KiB, contiguous in the
// caller's [H][128][512] layout).  The CTA computes the 16 BF16 q values, then
// their contribution to all 512 latent columns, and stores that FP32 partial
// sum.  A per-head counter finds the last of a head's 8 tasks; that CTA adds
// the 8 partials in task order and writes q_latent.  Rope rows stream after a
// CTA's tasks and go straight to q_pe.  Each CTA owns a contiguous run of
// tasks and of rope rows, balanced in bytes on the host.
// ===========================================================================

constexpr int kTaskQbBytes = kTaskRows * kPitch;              // 50176
constexpr int kAbsStages = 3;
constexpr int kAbsThreads = kConsumers + 32;                  // + producer warp
// The 16-token paired kernel has a KV insert warp besides: its consumers'
// longer prologue would otherwise carry the insert (measured at H = 64: 11.6
// against 11.0 us); the 8-token kernel's consumers are faster without it.
template <int NT>
constexpr int pair_threads() {
  return NT == 16 ? kAbsThreads + 32 : kAbsThreads;
}

// This CTA's stages: tasks [t0, t1), then rope rows [r0, r1) in chunks of 16.
struct AbsSeq {
  int t0, t1, r0, r1;
  __device__ int tasks() const { return t1 - t0; }
  __device__ int stages() const { return (t1 - t0) + (r1 - r0 + kTaskRows - 1) / kTaskRows; }
};

__device__ __forceinline__ int rope_row(int r) {  // rope index -> W_QB row
  return (r / kRope) * kHeadRows + kNope + (r % kRope);
}

// Prefetch stage k of a CTA's sequence into L2: a task's 16 W_QB rows and 16
// W_UK rows are two contiguous runs, a rope chunk at most two (it may cross
// into the next head).
__device__ __forceinline__ void abs_prefetch_stage(const DecodeArgs& a, const AbsSeq& seq, int k) {
  if (k < seq.tasks()) {
    const int tk = seq.t0 + k, h = tk / kTasksPerHead, p0 = (tk % kTasksPerHead) * kTaskRows;
    bulk_prefetch_l2(a.w_qb + ((int64_t)h * kHeadRows + p0) * kQLora, kTaskRows * kRowBytes);
    bulk_prefetch_l2(a.w_uk + ((int64_t)h * kNope + p0) * kKvLora, kTaskUkBytes);
  } else {
    const int r = seq.r0 + (k - seq.tasks()) * kTaskRows;
    const int n = min(kTaskRows, seq.r1 - r);
    const int n1 = min(n, kRope - r % kRope);
    bulk_prefetch_l2(a.w_qb + (int64_t)rope_row(r) * kQLora, (uint32_t)(n1 * kRowBytes));
    if (n > n1)
      bulk_prefetch_l2(a.w_qb + (int64_t)rope_row(r + n1) * kQLora, (uint32_t)((n - n1) * kRowBytes));
  }
}

// Latent columns 4 c4..4 c4 + 3 of head h, token t: the head's 8 FP32
// partials (laid out [task][token < NT][512]) added in task order and rounded
// once (BF16, or with a per-tensor query scale the E4M3 code of the BF16
// value).
template <int NT>
__device__ __forceinline__ void close_item(const DecodeArgs& a, int h, int t, int c4) {
  {
    const float* part = a.partial + ((int64_t)h * kTasksPerHead * NT + t) * kKvLora + 4 * c4;
    float4 v[kTasksPerHead];
#pragma unroll
    for (int pb = 0; pb < kTasksPerHead; ++pb)
      v[pb] = ld_cg_f32x4(part + (int64_t)pb * NT * kKvLora);
    float4 acc = v[0];
#pragma unroll
    for (int pb = 1; pb < kTasksPerHead; ++pb) {
      acc.x += v[pb].x;
      acc.y += v[pb].y;
      acc.z += v[pb].z;
      acc.w += v[pb].w;
    }
    const int64_t idx = (int64_t)t * a.ql_ts + (int64_t)h * a.ql_hs + 4 * c4;
    if (a.q_scale_inv == nullptr) {
      uint2 o;
      o.x = pack_bf16x2(acc.x, acc.y);
      o.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(a.q_latent + idx) = o;
    } else {
      const float qsi = *a.q_scale_inv;
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(a.q_latent) + idx) =
          (uint32_t)q_fp8(acc.x, qsi) | ((uint32_t)q_fp8(acc.y, qsi) << 8) |
          ((uint32_t)q_fp8(acc.z, qsi) << 16) | ((uint32_t)q_fp8(acc.w, qsi) << 24);
    }
  }
}

// ===========================================================================
// Absorbing kernel on tensor cores (up to 16 tokens per CTA).
//
// The tasks, rope chunks, host split and head closing above, with the
// arithmetic on mma.sync m16n8k16 (BF16 operands, FP32 accumulate):
//  * Q_B: a stage's 16 weight rows are the M side and the tokens the N side
//    (8 per n-tile); warp w takes the K slice [192 w, 192 w + 192), and the
//    eight split-K partial tiles are added in warp order after one barrier
//    (two partial buffers alternate, so one barrier per stage suffices).
//  * absorption: W_UK^T of the task (512 latent columns x 16 rows) is the M
//    side, read with ldmatrix.trans from rows padded to 1040 B; the task's 16
//    BF16-rounded q values of each token are the N side.  Warp w owns the
//    latent columns [64 w, 64 w + 64).
// The normalised q_a row never lives in shared memory: each lane builds the
// B fragments of its K slice straight from q_a and keeps them in registers.
// Both contractions use one k order for A and B: a lane's 8 consecutive K
// values (one 16-byte load of a weight row and of its xq) feed two mma
// k-steps, which only permutes the terms of each dot product.
// ===========================================================================

constexpr int kUkPitchM = kKvLora * 2 + 16;               // 1040 B: conflict-free ldmatrix
constexpr int kTaskUkBytesM = kTaskRows * kUkPitchM;      // 16640
constexpr int kTaskStageM = kTaskQbBytes + kTaskUkBytesM; // 66816
constexpr int kRedTok = 24;  // floats per (warp, token) row of split-K partials (16 used)

template <int NT>
struct AbsMmaSmem {
  static constexpr int kRing = kAbsStages * kTaskStageM;
  static constexpr int kRedBuf = kConsumerWarps * NT * kRedTok;   // floats per buffer
  static constexpr int oRed = kRing;                               // [2][warp][token][kRedTok]
  static constexpr int oSs = oRed + 2 * kRedBuf * 4;               // [warp][NT] + [8] floats
  static constexpr int oFull = oSs + (kConsumerWarps * NT + 8) * 4;
  static constexpr int oEmpty = oFull + kAbsStages * 8;
  static constexpr int oRbar = oEmpty + kAbsStages * 8;            // [2] split-K barriers
  static constexpr int oClose = oRbar + 16;                        // head this CTA closes, or -1
  static constexpr int kBytes = oClose + 16;
  static constexpr int kAlloc = kBytes + 128;
};

template <int NT>
__global__ void __launch_bounds__(kAbsThreads, 1)
    mla_absorb_mma_kernel(const DecodeArgs a, const __grid_constant__ AbsSplit split) {
  using S = AbsMmaSmem<NT>;
  constexpr int NTL = NT / 8;  // n-tiles
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint8_t* ring = smem;
  float* redp = reinterpret_cast<float*>(smem + S::oRed);
  float* ss_s = reinterpret_cast<float*>(smem + S::oSs);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::oFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::oEmpty);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + S::oRbar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x, P = gridDim.x;
  const AbsSeq seq{split.task[i], split.task[i + 1], split.rope[i], split.rope[i + 1]};
  const int nst = seq.stages();

  if (tid == 0) {
    for (int s = 0; s < kAbsStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&rbar[0], kConsumerWarps);
    mbar_init(&rbar[1], kConsumerWarps);
    mbar_fence_init();
    pdl_launch_dependents();  // the head-closing kernel may be scheduled now
    trace_stamp(a, 0);
  }
  __syncthreads();
  bool timed_out = false;

  if (warp == kConsumerWarps) {
    // ================= producer: weights only, no PDL wait ============
    // As in the FMA flavour; a task's W_UK rows land at a 1040-byte pitch.
    const uint64_t pol = l2_policy_evict_first();
    for (int k = 0; k < nst; ++k) {
      if (k == kAbsStages) {
        for (int kk = kAbsStages + lane; kk < nst; kk += 32) abs_prefetch_stage(a, seq, kk);
        __syncwarp();
      }
      const int slot = k % kAbsStages;
      uint8_t* buf = ring + slot * kTaskStageM;
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
        if (lane == 0)
          mbar_arrive_expect_tx(&full[slot], kTaskRows * kRowBytes + kTaskRows * kKvLora * 2);
        __syncwarp();
        if (lane < kTaskRows)
          bulk_g2s_hint(buf + lane * kPitch,
                        a.w_qb + ((int64_t)h * kHeadRows + p0 + lane) * kQLora, kRowBytes,
                        &full[slot], pol);
        else
          bulk_g2s_hint(buf + kTaskQbBytes + (lane - kTaskRows) * kUkPitchM,
                        a.w_uk + ((int64_t)h * kNope + p0 + lane - kTaskRows) * kKvLora,
                        kKvLora * 2, &full[slot], pol);
      } else {
        const int r = seq.r0 + (k - seq.tasks()) * kTaskRows;
        const int n = min(kTaskRows, seq.r1 - r);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * kRowBytes));
        __syncwarp();
        if (lane < n)
          bulk_g2s_hint(buf + lane * kPitch, a.w_qb + (int64_t)rope_row(r + lane) * kQLora,
                        kRowBytes, &full[slot], pol);
      }
    }
    if (lane == 0)
      for (int k = max(0, nst - kAbsStages); k < nst; ++k)
        (void)mbar_wait_bounded(&full[k % kAbsStages], (uint32_t)((k / kAbsStages) & 1),
                                kWaitLimit);
  } else {
    // ================= consumer warps 0-7 ============================
    const int g = lane >> 2, q = lane & 3;
    // gamma_q of this lane's K slice: a static weight, loaded before the wait
    uint4 gam[6];
#pragma unroll
    for (int c = 0; c < 6; ++c)
      gam[c] = *reinterpret_cast<const uint4*>(a.gamma_q + 192 * warp + 32 * c + 8 * q);
    pdl_wait();
    if (tid == 0) trace_stamp(a, 3);
    // q_a RMSNorm -> B fragments xb[nt][c] (token 8 nt + g, K 192 w + 32 c + 8 q + 0..7)
    uint4 xb[NTL][6];
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      const int tok = 8 * nt + g;
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        xb[nt][c] = tok < a.batch
                        ? *reinterpret_cast<const uint4*>(a.q_a + (int64_t)tok * a.q_a_stride +
                                                          192 * warp + 32 * c + 8 * q)
                        : make_uint4(0, 0, 0, 0);
        const uint32_t ww[4] = {xb[nt][c].x, xb[nt][c].y, xb[nt][c].z, xb[nt][c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ss = fmaf(bf16lo(ww[e]), bf16lo(ww[e]), ss);
          ss = fmaf(bf16hi(ww[e]), bf16hi(ww[e]), ss);
        }
      }
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
      if (q == 0) ss_s[warp * NT + tok] = ss;
    }
    named_barrier(kBarConsumers, kConsumers);
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      const int tok = 8 * nt + g;
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) total += ss_s[w * NT + tok];
      const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, 1536.0f), a.eps));
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const uint32_t ww[4] = {xb[nt][c].x, xb[nt][c].y, xb[nt][c].z, xb[nt][c].w};
        const uint32_t gw[4] = {gam[c].x, gam[c].y, gam[c].z, gam[c].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = rms_scale_bf16x2(ww[e], rr, gw[e]);
        xb[nt][c] = make_uint4(o[0], o[1], o[2], o[3]);
        if (i == 0 && a.q_c != nullptr && tok < a.batch)
          *reinterpret_cast<uint4*>(a.q_c + (int64_t)tok * kQLora + 192 * warp + 32 * c + 8 * q) =
              xb[nt][c];
      }
    }
    // KV insert of token i (and i + P, ...) by warps 6-7
    if (warp >= 6)
      for (int t = i; t < a.batch; t += P) kv_insert(a, t, tid - 192, ss_s + kConsumerWarps * NT);
    if (tid == 0) trace_stamp(a, 2);

#ifdef MLA_TRACE
    long long ph[6] = {0, 0, 0, 0, 0, 0};
    long long tc = clock64();
#define MLA_PHASE(j)                   \
  do {                                 \
    const long long t2_ = clock64();   \
    ph[j] += t2_ - tc;                 \
    tc = t2_;                          \
  } while (0)
#else
#define MLA_PHASE(j) \
  do {               \
  } while (0)
#endif
    for (int k = 0; k < nst; ++k) {
      const int slot = k % kAbsStages;
      const uint8_t* buf = ring + slot * kTaskStageM;
      if (!mbar_wait_bounded(&full[slot], (uint32_t)((k / kAbsStages) & 1), kWaitLimit))
        timed_out = true;
      MLA_PHASE(0);
      if (tid == 0 && k < 20) trace_stamp(a, 8 + k);
      const bool task = k < seq.tasks();
      // ---- Q_B rows of the stage over this warp's K slice ---------------
      // Four independent accumulator chains (the 12 k-steps would otherwise
      // wait on one another's results), added pairwise at the end.
      float acc[NTL][4];
      {
        uint4 alo[6], ahi[6];
#pragma unroll
        for (int c = 0; c < 6; ++c) {
          const int kb = 2 * (192 * warp + 32 * c + 8 * q);
          alo[c] = *reinterpret_cast<const uint4*>(buf + g * kPitch + kb);
          ahi[c] = *reinterpret_cast<const uint4*>(buf + (g + 8) * kPitch + kb);
        }
        float ch[NTL][4][4];
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) ch[nt][j][0] = ch[nt][j][1] = ch[nt][j][2] = ch[nt][j][3] = 0.f;
#pragma unroll
        for (int c = 0; c < 6; ++c)
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            mma_bf16_16816(ch[nt][2 * (c & 1)], alo[c].x, ahi[c].x, alo[c].y, ahi[c].y,
                           xb[nt][c].x, xb[nt][c].y);
            mma_bf16_16816(ch[nt][2 * (c & 1) + 1], alo[c].z, ahi[c].z, alo[c].w, ahi[c].w,
                           xb[nt][c].z, xb[nt][c].w);
          }
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[nt][e] = (ch[nt][0][e] + ch[nt][1][e]) + (ch[nt][2][e] + ch[nt][3][e]);
      }
      if (!task) {  // a rope stage holds no W_UK: the slot is free now
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      MLA_PHASE(1);
      // ---- split-K partials -> shared, one barrier ----------------------
      float* red = redp + (k & 1) * S::kRedBuf;
      {
        float* rw = red + warp * NT * kRedTok;
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) {
          const int t0 = 8 * nt + 2 * q;
          rw[t0 * kRedTok + g] = acc[nt][0];
          rw[(t0 + 1) * kRedTok + g] = acc[nt][1];
          rw[t0 * kRedTok + g + 8] = acc[nt][2];
          rw[(t0 + 1) * kRedTok + g + 8] = acc[nt][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rbar[k & 1]);
      if (!mbar_wait_bounded(&rbar[k & 1], (uint32_t)((k >> 1) & 1), kWaitLimit)) timed_out = true;
      MLA_PHASE(2);

      if (!task) {
        // ---- rope rows -> q_pe ------------------------------------------
        const int r0 = seq.r0 + (k - seq.tasks()) * kTaskRows;
        const int nrows = min(kTaskRows, seq.r1 - r0);
        for (int e = tid; e < kTaskRows * NT; e += kConsumers) {
          const int row = e & (kTaskRows - 1), tok = e >> 4;
          if (row < nrows && tok < a.batch) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * NT + tok) * kRedTok + row];
            const int r = r0 + row;
            put_q(a, a.q_pe, (int64_t)tok * a.qp_ts + (int64_t)(r / kRope) * a.qp_hs + r % kRope, v,
                  load_qsi(a));
          }
        }
        MLA_PHASE(5);
        continue;
      }
      // ---- task: BF16 q of the 16 rows (B fragments of q^T), absorption --
      uint32_t qb[NTL][2];
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt) {
        const int tok = 8 * nt + g;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float* rr = red + (w * NT + tok) * kRedTok;
          const float2 lo = *reinterpret_cast<const float2*>(rr + 2 * q);
          const float2 hi = *reinterpret_cast<const float2*>(rr + 2 * q + 8);
          s0 += lo.x;
          s1 += lo.y;
          s2 += hi.x;
          s3 += hi.y;
        }
        qb[nt][0] = pack_bf16x2(s0, s1);
        qb[nt][1] = pack_bf16x2(s2, s3);
      }
      const uint32_t uk = smem_u32(buf + kTaskQbBytes);
      float d[4][NTL][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int m = lane >> 3;
        const int p = (lane & 7) + 8 * (m >> 1);
        const int c = 64 * warp + 16 * mt + 8 * (m & 1);
        uint32_t af[4];
        ldmatrix_x4_trans(af, uk + p * kUkPitchM + 2 * c);
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) {
          d[mt][nt][0] = d[mt][nt][1] = d[mt][nt][2] = d[mt][nt][3] = 0.f;
          mma_bf16_16816(d[mt][nt], af[0], af[1], af[2], af[3], qb[nt][0], qb[nt][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // W_QB and W_UK of the slot are read
      MLA_PHASE(3);
      // FP32 partial absorption of this task: [task][token][512]
      const int n = k, tk = seq.t0 + k;
      (void)n;
      float* part = a.partial + (int64_t)tk * NT * kKvLora;
      const bool part_ok = MLA_IN_BOUNDS(a, tk >= 0 && tk < a.heads * kTasksPerHead, 14);
#pragma unroll
      for (int mt = 0; mt < 4 && part_ok; ++mt) {
        const int c = 64 * warp + 16 * mt + g;
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) {
          const int t0 = 8 * nt + 2 * q;
          if (t0 < a.batch) {
            part[(int64_t)t0 * kKvLora + c] = d[mt][nt][0];
            part[(int64_t)t0 * kKvLora + c + 8] = d[mt][nt][2];
          }
          if (t0 + 1 < a.batch) {
            part[(int64_t)(t0 + 1) * kKvLora + c] = d[mt][nt][1];
            part[(int64_t)(t0 + 1) * kKvLora + c + 8] = d[mt][nt][3];
          }
        }
      }
      // The CTA that stores a head's last partial closes the head: it adds
      // the 8 partials in task order (no second kernel).  A per-head counter
      // in the handle's scratch counts the stored tasks; the closer resets
      // it for the next call.
      __threadfence();
      named_barrier(kBarConsumers, kConsumers);
      int* close_s = reinterpret_cast<int*>(smem + S::oClose);
      if (tid == 0) {
        const int h = tk / kTasksPerHead;
        int ch = -1;
        if (atomicAdd(&a.ready[h], 1u) + 1 == (uint32_t)kTasksPerHead) {
          __threadfence();
          a.ready[h] = 0;
          ch = h;
        }
        *close_s = ch;
      }
      named_barrier(kBarConsumers, kConsumers);
      const int ch = *close_s;
      if (ch >= 0)
        for (int it = tid; it < a.batch * (kKvLora / 4); it += kConsumers)
          close_item<NT>(a, ch, it / (kKvLora / 4), it % (kKvLora / 4));
      MLA_PHASE(4);
    }
#ifdef MLA_TRACE
    if (lane == 0 && (warp == 0 || warp == 5))
      for (int j = 0; j < 6; ++j) trace_add(a, (warp == 0 ? 56 : 22) + j, ph[j]);
#endif
#undef MLA_PHASE
    if (tid == 0) trace_stamp(a, 6);
  }

  if (timed_out) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  __syncthreads();
  if (tid == 0) trace_stamp(a, 7);
}

// ===========================================================================
// Paired absorbing kernel (tensor cores, up to 16 tokens): clusters of two CTAs.
//
// Both CTAs of a pair take the same heads; rank r streams nope tasks
// 4r..4r+3 (rows 64r..64r+63) of each, with their W_UK rows, and accumulates
// the head's absorption over its four tasks in the mma accumulators.  After a
// head's last task, the warps whose latent columns the other CTA owns (rank 0
// owns columns 0..255, rank 1 columns 256..511) send their FP32 sums into the
// other CTA's shared memory (st.async, counted on its mbarrier).  After the
// rope stages each CTA adds the two halves of its columns - rows 0..63 first,
// then rows 64..127 - and writes q_latent.  No global scratch, no second
// kernel, no wait on any CTA outside the pair.
//
// NT = 8 tokens: a 3-stage ring, the owned sums stay in registers.
// NT = 16: a 2-stage ring (shared memory), the owned sums go to shared memory.
// ===========================================================================

constexpr int kPairPrefetch = 1;  // stages prefetched into L2 beyond the ring

template <int NT>
struct PairSmem {
  static constexpr int NTL = NT / 8;
  static constexpr int kStages = NT == 8 ? 3 : 2;
  static constexpr int kRecvBytes = 4 * 4 * NTL * 32 * 16;  // 4 warps x 4 m-tiles x n-tiles x 32 lanes x 16 B
  static constexpr bool kKeepInSmem = NT > 8;
  static constexpr int kRing = kStages * kTaskStageM;
  static constexpr int kRedBuf = kConsumerWarps * NT * kRedTok;     // floats per buffer
  static constexpr int oRed = kRing;                                 // [2][warp][token][kRedTok]
  static constexpr int oRecv = oRed + 2 * kRedBuf * 4;               // [2 heads][kRecvBytes]
  static constexpr int oKeep = oRecv + 2 * kRecvBytes;               // [2 heads][kRecvBytes] (NT > 8)
  static constexpr int oSs = oKeep + (kKeepInSmem ? 2 * kRecvBytes : 0);  // [warp][NT] + [8] floats
  static constexpr int oFull = oSs + (kConsumerWarps * NT + 8) * 4;
  static constexpr int oEmpty = oFull + kStages * 8;
  static constexpr int oRbar = oEmpty + kStages * 8;                 // [2] split-K barriers
  static constexpr int oRecvBar = oRbar + 16;                        // [2] received halves
  static constexpr int kBytes = oRecvBar + 16;
  static constexpr int kAlloc = kBytes + 128;
};

// This CTA's stages: 4 tasks per head of its pair, then rope rows [r0, r1).
struct PairSeq {
  int h0, nh, rank, r0, r1;
  __device__ int tasks() const { return 4 * nh; }
  __device__ int stages() const { return 4 * nh + (r1 - r0 + kTaskRows - 1) / kTaskRows; }
  __device__ int head(int k) const { return h0 + k / 4; }
  __device__ int p0(int k) const { return kTaskRows * (4 * rank + k % 4); }
};

__device__ __forceinline__ void pair_prefetch_stage(const DecodeArgs& a, const PairSeq& seq, int k) {
  if (k < seq.tasks()) {
    const int h = seq.head(k), p0 = seq.p0(k);
    bulk_prefetch_l2(a.w_qb + ((int64_t)h * kHeadRows + p0) * kQLora, kTaskRows * kRowBytes);
    bulk_prefetch_l2(a.w_uk + ((int64_t)h * kNope + p0) * kKvLora, kTaskUkBytes);
  } else {
    const int r = seq.r0 + (k - seq.tasks()) * kTaskRows;
    const int n = min(kTaskRows, seq.r1 - r);
    const int n1 = min(n, kRope - r % kRope);
    bulk_prefetch_l2(a.w_qb + (int64_t)rope_row(r) * kQLora, (uint32_t)(n1 * kRowBytes));
    if (n > n1)
      bulk_prefetch_l2(a.w_qb + (int64_t)rope_row(r + n1) * kQLora, (uint32_t)((n - n1) * kRowBytes));
  }
}

template <int NT>
__global__ void __launch_bounds__(pair_threads<NT>(), 1)
    mla_absorb_pair_kernel(const DecodeArgs a, const __grid_constant__ PairSplit split) {
  using S = PairSmem<NT>;
  constexpr int NTL = S::NTL;
  constexpr int ST = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  uint8_t* ring = smem;
  float* redp = reinterpret_cast<float*>(smem + S::oRed);
  float* ss_s = reinterpret_cast<float*>(smem + S::oSs);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::oFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::oEmpty);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + S::oRbar);
  uint64_t* recvbar = reinterpret_cast<uint64_t*>(smem + S::oRecvBar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x, P = gridDim.x;
  const int pair = i >> 1, rank = i & 1;  // cluster (2, 1, 1): rank = blockIdx.x % 2
  const PairSeq seq{split.head[pair], split.head[pair + 1] - split.head[pair], rank,
                    split.rope[i], split.rope[i + 1]};
  const int nst = seq.stages();
  bool timed_out = false;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&rbar[0], kConsumerWarps);
    mbar_init(&rbar[1], kConsumerWarps);
    mbar_init(&recvbar[0], 1);
    mbar_init(&recvbar[1], 1);
    // The other CTA's sums of head j land in recv[j]: armed before this CTA
    // arrives at the cluster barrier, so no byte can arrive before its count
    // is expected.
    for (int j = 0; j < seq.nh; ++j) mbar_arrive_expect_tx(&recvbar[j], S::kRecvBytes);
    mbar_fence_init();
    pdl_launch_dependents();
    trace_stamp(a, 0);
  }
  __syncthreads();
  // The cluster barrier's first phase orders the other CTA's recvbar before
  // the first remote store: every thread arrives now (relaxed: the
  // mbarrier-init fence publishes the barriers; a release arrive measured
  // slower, 8.07 against 7.94 us at 64 heads), the consumers wait after the
  // q_a prologue, the other warps at their end.  The producer starts
  // copying without waiting for the pair.  (The producer initialising its
  // own ring barriers and issuing before the CTA meets measured 8.18 us.)
  cluster_arrive_relaxed();

  if (warp == kConsumerWarps) {
    // ================= producer: weights only, no PDL wait ============
    // L2 prefetch runs kPairPrefetch stages ahead of the ring: HBM keeps
    // streaming while the ring is full, without a whole two-head share
    // (about 450 KiB per CTA) sitting in L2 at once (measured: a window of one
    // stage beats deeper ones at 128 heads, 14.9 us against 16.9 us for four).
    const uint64_t pol = l2_policy_evict_first();
    for (int k = 0; k < nst; ++k) {
      if (k == ST) {
        for (int kk = ST + lane; kk < min(nst, ST + kPairPrefetch); kk += 32)
          pair_prefetch_stage(a, seq, kk);
        __syncwarp();
      } else if (k > ST && lane == 0 && k - 1 + kPairPrefetch < nst) {
        pair_prefetch_stage(a, seq, k - 1 + kPairPrefetch);
      }
      const int slot = k % ST;
      uint8_t* buf = ring + slot * kTaskStageM;
      if (k >= ST) {
        int ok = 1;
        if (lane == 0)
          ok = mbar_wait_bounded(&empty[slot], (uint32_t)(((k / ST) - 1) & 1), kWaitLimit) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) timed_out = true;
      }
      if (lane == 0 && k < 20) trace_stamp(a, 28 + k);
      if (k < seq.tasks()) {
        const int h = seq.head(k), p0 = seq.p0(k);
        if (lane == 0)
          mbar_arrive_expect_tx(&full[slot], kTaskRows * kRowBytes + kTaskRows * kKvLora * 2);
        __syncwarp();
        if (!MLA_IN_BOUNDS(a, h >= 0 && h < a.heads && p0 >= 0 && p0 + kTaskRows <= kNope, 0) ||
            !MLA_IN_BOUNDS(a, slot >= 0 && slot < ST, 1)) {
        } else if (lane < kTaskRows)
          bulk_g2s_hint(buf + lane * kPitch,
                        a.w_qb + ((int64_t)h * kHeadRows + p0 + lane) * kQLora, kRowBytes,
                        &full[slot], pol);
        else
          bulk_g2s_hint(buf + kTaskQbBytes + (lane - kTaskRows) * kUkPitchM,
                        a.w_uk + ((int64_t)h * kNope + p0 + lane - kTaskRows) * kKvLora,
                        kKvLora * 2, &full[slot], pol);
      } else {
        const int r = seq.r0 + (k - seq.tasks()) * kTaskRows;
        const int n = min(kTaskRows, seq.r1 - r);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * kRowBytes));
        __syncwarp();
        if (lane < n &&
            MLA_IN_BOUNDS(a, r + lane >= 0 && r + lane < a.heads * kRope && slot < ST, 0))
          bulk_g2s_hint(buf + lane * kPitch, a.w_qb + (int64_t)rope_row(r + lane) * kQLora,
                        kRowBytes, &full[slot], pol);
      }
    }
    if (lane == 0)
      for (int k = max(0, nst - ST); k < nst; ++k)
        (void)mbar_wait_bounded(&full[k % ST], (uint32_t)((k / ST) & 1), kWaitLimit);
    cluster_wait_acquire();
  } else if (warp == kConsumerWarps + 1) {
    // ================= KV insert warp (16 tokens) ====================
    // The CTA's KV rows (kv_c and k_pe are inputs: after the PDL wait), off
    // the consumers' and the producer's paths.
    pdl_wait();
    for (int t = i; t < a.batch; t += P) kv_insert_warp(a, t, lane);
    cluster_wait_acquire();
  } else {
    // ================= consumer warps 0-7 ============================
    const int g = lane >> 2, q = lane & 3;
    uint4 gam[6];
#pragma unroll
    for (int c = 0; c < 6; ++c)
      gam[c] = *reinterpret_cast<const uint4*>(a.gamma_q + 192 * warp + 32 * c + 8 * q);
    pdl_wait();
    if (tid == 0) trace_stamp(a, 3);
    // q_a RMSNorm -> B fragments xb[nt][c] (token 8 nt + g, K 192 w + 32 c + 8 q + 0..7).
    // Every n-tile's loads go out before the first sum of squares (one load
    // round trip for 16 tokens: 10.51 against 10.58 us at B = 16, H = 64).
    // The 16-token flavour reads q_a through the read-only path (q_a is an
    // input of the step, complete once the wait has passed): 9.73 against
    // 10.54 us at B = 16, H = 64; the 8-token flavour keeps plain loads
    // (7.84 against 7.79 us at B = 1 with the read-only path).
    uint4 xb[NTL][6];
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      const int tok = 8 * nt + g;
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const uint4* src = reinterpret_cast<const uint4*>(a.q_a + (int64_t)tok * a.q_a_stride +
                                                          192 * warp + 32 * c + 8 * q);
        if constexpr (NT == 16)
          xb[nt][c] = tok < a.batch ? __ldg(src) : make_uint4(0, 0, 0, 0);
        else
          xb[nt][c] = tok < a.batch ? *src : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      const int tok = 8 * nt + g;
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const uint32_t ww[4] = {xb[nt][c].x, xb[nt][c].y, xb[nt][c].z, xb[nt][c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ss = fmaf(bf16lo(ww[e]), bf16lo(ww[e]), ss);
          ss = fmaf(bf16hi(ww[e]), bf16hi(ww[e]), ss);
        }
      }
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
      ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
      if (q == 0) ss_s[warp * NT + tok] = ss;
    }
    named_barrier(kBarConsumers, kConsumers);
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
      const int tok = 8 * nt + g;
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) total += ss_s[w * NT + tok];
      const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, 1536.0f), a.eps));
#pragma unroll
      for (int c = 0; c < 6; ++c) {
        const uint32_t ww[4] = {xb[nt][c].x, xb[nt][c].y, xb[nt][c].z, xb[nt][c].w};
        const uint32_t gw[4] = {gam[c].x, gam[c].y, gam[c].z, gam[c].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = rms_scale_bf16x2(ww[e], rr, gw[e]);
        xb[nt][c] = make_uint4(o[0], o[1], o[2], o[3]);
        if (i == 0 && a.q_c != nullptr && tok < a.batch)
          *reinterpret_cast<uint4*>(a.q_c + (int64_t)tok * kQLora + 192 * warp + 32 * c + 8 * q) =
              xb[nt][c];
      }
    }
    if (NT == 8 && warp >= 6)
      for (int t = i; t < a.batch; t += P) kv_insert(a, t, tid - 192, ss_s + kConsumerWarps * NT);
    if (tid == 0) trace_stamp(a, 2);
    cluster_wait_acquire();  // the other CTA's recvbar armed (long since, by now)

    // Columns 64 w .. 64 w + 63 belong to rank 0 for w < 4, to rank 1 else.
    // A warp's slot of a per-head buffer: [m-tile][n-tile][lane][16 B].
    const bool own = (warp < 4) == (rank == 0);
    const int slot_off = (warp & 3) * (4 * NTL * 32 * 16);
    float dacc[4][NTL][4];   // this head's absorption over the tasks so far
    float keep[2][4][4];     // NT = 8: owned sums of heads 0 and 1 of the pair
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        keep[0][mt][e] = keep[1][mt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) dacc[mt][nt][e] = 0.f;
      }

    for (int k = 0; k < nst; ++k) {
      const int slot = k % ST;
      const uint8_t* buf = ring + slot * kTaskStageM;
      if (!mbar_wait_bounded(&full[slot], (uint32_t)((k / ST) & 1), kWaitLimit)) timed_out = true;
      if (tid == 0 && k < 20) trace_stamp(a, 8 + k);
      const bool task = k < seq.tasks();
      // ---- Q_B rows of the stage over this warp's K slice ---------------
      float acc[NTL][4];
      {
        uint4 alo[6], ahi[6];
#pragma unroll
        for (int c = 0; c < 6; ++c) {
          const int kb = 2 * (192 * warp + 32 * c + 8 * q);
          alo[c] = *reinterpret_cast<const uint4*>(buf + g * kPitch + kb);
          ahi[c] = *reinterpret_cast<const uint4*>(buf + (g + 8) * kPitch + kb);
        }
        float ch[NTL][4][4];
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) ch[nt][j][0] = ch[nt][j][1] = ch[nt][j][2] = ch[nt][j][3] = 0.f;
#pragma unroll
        for (int c = 0; c < 6; ++c)
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            mma_bf16_16816(ch[nt][2 * (c & 1)], alo[c].x, ahi[c].x, alo[c].y, ahi[c].y,
                           xb[nt][c].x, xb[nt][c].y);
            mma_bf16_16816(ch[nt][2 * (c & 1) + 1], alo[c].z, ahi[c].z, alo[c].w, ahi[c].w,
                           xb[nt][c].z, xb[nt][c].w);
          }
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[nt][e] = (ch[nt][0][e] + ch[nt][1][e]) + (ch[nt][2][e] + ch[nt][3][e]);
      }
      if (!task) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      // ---- split-K partials -> shared, one barrier ----------------------
      float* red = redp + (k & 1) * S::kRedBuf;
      {
        float* rw = red + warp * NT * kRedTok;
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) {
          const int t0 = 8 * nt + 2 * q;
          rw[t0 * kRedTok + g] = acc[nt][0];
          rw[(t0 + 1) * kRedTok + g] = acc[nt][1];
          rw[t0 * kRedTok + g + 8] = acc[nt][2];
          rw[(t0 + 1) * kRedTok + g + 8] = acc[nt][3];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rbar[k & 1]);
      if (!mbar_wait_bounded(&rbar[k & 1], (uint32_t)((k >> 1) & 1), kWaitLimit)) timed_out = true;

      if (!task) {
        // ---- rope rows -> q_pe ------------------------------------------
        const int r0 = seq.r0 + (k - seq.tasks()) * kTaskRows;
        const int nrows = min(kTaskRows, seq.r1 - r0);
        for (int e = tid; e < kTaskRows * NT; e += kConsumers) {
          const int row = e & (kTaskRows - 1), tok = e >> 4;
          if (row < nrows && tok < a.batch &&
              MLA_IN_BOUNDS(a, r0 + row >= 0 && r0 + row < a.heads * kRope, 2)) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * NT + tok) * kRedTok + row];
            const int r = r0 + row;
            put_q(a, a.q_pe, (int64_t)tok * a.qp_ts + (int64_t)(r / kRope) * a.qp_hs + r % kRope, v,
                  load_qsi(a));
          }
        }
        continue;
      }
      // ---- task: BF16 q of the 16 rows, absorption into dacc -------------
      uint32_t qb[NTL][2];
#pragma unroll
      for (int nt = 0; nt < NTL; ++nt) {
        const int tok = 8 * nt + g;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float* rr = red + (w * NT + tok) * kRedTok;
          const float2 lo = *reinterpret_cast<const float2*>(rr + 2 * q);
          const float2 hi = *reinterpret_cast<const float2*>(rr + 2 * q + 8);
          s0 += lo.x;
          s1 += lo.y;
          s2 += hi.x;
          s3 += hi.y;
        }
        qb[nt][0] = pack_bf16x2(s0, s1);
        qb[nt][1] = pack_bf16x2(s2, s3);
      }
      const int u = k & 3;  // task of the head: 0..3
      if (u == 0) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt)
            dacc[mt][nt][0] = dacc[mt][nt][1] = dacc[mt][nt][2] = dacc[mt][nt][3] = 0.f;
      }
      const uint32_t uk = smem_u32(buf + kTaskQbBytes);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int m = lane >> 3;
        const int p = (lane & 7) + 8 * (m >> 1);
        const int c = 64 * warp + 16 * mt + 8 * (m & 1);
        uint32_t af[4];
        ldmatrix_x4_trans(af, uk + p * kUkPitchM + 2 * c);
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt)
          mma_bf16_16816(dacc[mt][nt], af[0], af[1], af[2], af[3], qb[nt][0], qb[nt][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // W_QB and W_UK of the slot are read
      if (u == 3) {
        const int j = k >> 2;  // head of the pair: 0 or 1
        if (own) {
          if constexpr (S::kKeepInSmem) {
            uint8_t* kp = smem + S::oKeep + j * S::kRecvBytes + slot_off;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
              for (int nt = 0; nt < NTL; ++nt)
                *reinterpret_cast<float4*>(kp + ((mt * NTL + nt) * 32 + lane) * 16) =
                    make_float4(dacc[mt][nt][0], dacc[mt][nt][1], dacc[mt][nt][2], dacc[mt][nt][3]);
          } else {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (j == 0) keep[0][mt][e] = dacc[mt][0][e];
                else keep[1][mt][e] = dacc[mt][0][e];
              }
          }
        } else if (MLA_IN_BOUNDS(a, j >= 0 && j < 2 && slot_off + (4 * NTL * 32 * 16) <=
                                                               S::kRecvBytes, 4)) {
          // to the other CTA: same warp slot (w & 3), same lane, head slot j
          const uint32_t peer = (uint32_t)(rank ^ 1);
          const uint32_t rbar_remote = mapa_shared(smem_u32(&recvbar[j]), peer);
          const uint32_t base = smem_u32(smem + S::oRecv + j * S::kRecvBytes + slot_off);
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTL; ++nt)
              st_async_v4(mapa_shared(base + (uint32_t)(((mt * NTL + nt) * 32 + lane) * 16), peer),
                          dacc[mt][nt][0], dacc[mt][nt][1], dacc[mt][nt][2], dacc[mt][nt][3],
                          rbar_remote);
        }
      }
    }
    if (tid == 0) trace_stamp(a, 6);

    // ---- owned columns: rows 0..63 (rank 0) + rows 64..127 (rank 1) ------
    // The BF16 results go back into this warp's receive slot as
    // [token][64 columns], then out as 16-byte stores.
    if (own) {
      for (int j = 0; j < seq.nh; ++j) {
        if (!mbar_wait_bounded(&recvbar[j], 0u, kWaitLimit)) timed_out = true;
        const int h = seq.h0 + j;
        if (!MLA_IN_BOUNDS(a, h >= 0 && h < a.heads && j < 2, 3)) break;
        uint8_t* slotp = smem + S::oRecv + j * S::kRecvBytes + slot_off;
        float v[4][NTL][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int nt = 0; nt < NTL; ++nt) {
            const float4 o = *reinterpret_cast<const float4*>(slotp + ((mt * NTL + nt) * 32 + lane) * 16);
            const float pv[4] = {o.x, o.y, o.z, o.w};
            float mine[4];
            if constexpr (S::kKeepInSmem) {
              const float4 kv = *reinterpret_cast<const float4*>(
                  smem + S::oKeep + j * S::kRecvBytes + slot_off + ((mt * NTL + nt) * 32 + lane) * 16);
              mine[0] = kv.x;
              mine[1] = kv.y;
              mine[2] = kv.z;
              mine[3] = kv.w;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) mine[e] = j == 0 ? keep[0][mt][e] : keep[1][mt][e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) v[mt][nt][e] = rank == 0 ? mine[e] + pv[e] : pv[e] + mine[e];
          }
        __syncwarp();
        if (a.q_scale_inv == nullptr) {
          uint16_t* stage = reinterpret_cast<uint16_t*>(slotp);  // [NT tokens][64 columns]
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTL; ++nt) {
              const int cl = 16 * mt + g, t0 = 8 * nt + 2 * q;  // column within the warp's 64
              stage[t0 * 64 + cl] = f2bf_bits(v[mt][nt][0]);
              stage[(t0 + 1) * 64 + cl] = f2bf_bits(v[mt][nt][1]);
              stage[t0 * 64 + cl + 8] = f2bf_bits(v[mt][nt][2]);
              stage[(t0 + 1) * 64 + cl + 8] = f2bf_bits(v[mt][nt][3]);
            }
          __syncwarp();
          for (int e = lane; e < a.batch * 8; e += 32) {  // 8 chunks of 16 B per token
            const int t = e >> 3, ch = e & 7;
            *reinterpret_cast<uint4*>(a.q_latent + (int64_t)t * a.ql_ts + (int64_t)h * a.ql_hs +
                                      64 * warp + 8 * ch) =
                *reinterpret_cast<const uint4*>(stage + t * 64 + 8 * ch);
          }
        } else {
          const float qsi = *a.q_scale_inv;
          uint8_t* stage = slotp;  // [NT tokens][64 columns] E4M3
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTL; ++nt) {
              const int cl = 16 * mt + g, t0 = 8 * nt + 2 * q;
              stage[t0 * 64 + cl] = q_fp8(v[mt][nt][0], qsi);
              stage[(t0 + 1) * 64 + cl] = q_fp8(v[mt][nt][1], qsi);
              stage[t0 * 64 + cl + 8] = q_fp8(v[mt][nt][2], qsi);
              stage[(t0 + 1) * 64 + cl + 8] = q_fp8(v[mt][nt][3], qsi);
            }
          __syncwarp();
          uint8_t* ql8 = reinterpret_cast<uint8_t*>(a.q_latent);
          for (int e = lane; e < a.batch * 4; e += 32) {  // 4 chunks of 16 B per token
            const int t = e >> 2, ch = e & 3;
            *reinterpret_cast<uint4*>(ql8 + (int64_t)t * a.ql_ts + (int64_t)h * a.ql_hs + 64 * warp +
                                      16 * ch) =
                *reinterpret_cast<const uint4*>(stage + t * 64 + 16 * ch);
          }
        }
      }
    }
  }

  if (timed_out) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  __syncthreads();
  // Neither CTA leaves while the other may still write into its shared memory
  // (every owner waited for its received bytes above; this only holds both).
  cluster_sync_relaxed();
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

template <int NT>
cudaError_t launch_abs_mma(const DecodeArgs& a, const AbsSplit& sp, int ctas, cudaStream_t stream) {
  using S = AbsMmaSmem<NT>;
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
  return cudaLaunchKernelEx(&cfg, mla_absorb_mma_kernel<NT>, a, sp);
}

template <int NT>
cudaError_t prepare_abs_mma() {
  using S = AbsMmaSmem<NT>;
  static_assert(S::kAlloc <= 232448, "shared memory budget");
  return cudaFuncSetAttribute(mla_absorb_mma_kernel<NT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
}

namespace {
template <int NT>
cudaLaunchConfig_t pair_config(int ctas, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(pair_threads<NT>(), 1, 1);
  cfg.dynamicSmemBytes = PairSmem<NT>::kAlloc;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}
}  // namespace

template <int NT>
bool pair_fits(int ctas) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<NT>(ctas, nullptr, attr);
  cfg.numAttrs = 1;  // the cluster shape only
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, mla_absorb_pair_kernel<NT>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return clusters >= ctas / 2;
}

bool pair_kernel_fits(int ctas, int nt) {
  return nt == 8 ? pair_fits<8>(ctas) : nt == 16 ? pair_fits<16>(ctas) : false;
}

cudaError_t launch_pair(const DecodeArgs& a, const PairSplit& sp, int ctas, int nt,
                        cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  if (nt == 8) {
    cudaLaunchConfig_t cfg = pair_config<8>(ctas, stream, attr);
    return cudaLaunchKernelEx(&cfg, mla_absorb_pair_kernel<8>, a, sp);
  }
  if (nt == 16) {
    cudaLaunchConfig_t cfg = pair_config<16>(ctas, stream, attr);
    return cudaLaunchKernelEx(&cfg, mla_absorb_pair_kernel<16>, a, sp);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_fused_kernels() {
  static_assert(PairSmem<8>::kAlloc <= 232448, "shared memory budget");
  static_assert(PairSmem<16>::kAlloc <= 232448, "shared memory budget");
  {
    cudaError_t e = cudaFuncSetAttribute(mla_absorb_pair_kernel<8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairSmem<8>::kAlloc);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mla_absorb_pair_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PairSmem<16>::kAlloc);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e;
  if ((e = prepare_abs_mma<8>()) != cudaSuccess) return e;
  if ((e = prepare_abs_mma<16>()) != cudaSuccess) return e;
  if ((e = prepare_one<1, false>()) != cudaSuccess) return e;
  if ((e = prepare_one<2, false>()) != cudaSuccess) return e;
  if ((e = prepare_one<8, true>()) != cudaSuccess) return e;
  if ((e = prepare_one<16, true>()) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_absorb(const DecodeArgs& a, const AbsSplit& sp, int nt, int ctas,
                          cudaStream_t stream) {
  if (nt == 8) return launch_abs_mma<8>(a, sp, ctas, stream);
  if (nt == 16) return launch_abs_mma<16>(a, sp, ctas, stream);
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
