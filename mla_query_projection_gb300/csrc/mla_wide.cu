// mla_wide.cu - the decode step for wide batches (17 to 64 tokens per launch)
// on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// What it computes is the step of page "mla.query", class MlaQuery (methods
// kernel / tiled / insert / insert_ds / store_qc): q_a RMSNorm -> xq (q_c),
// Q_B rows -> q (BF16, FP32 accumulate), rope rows -> q_pe, nope rows through
// W_UK -> q_latent, and the paged FP8 KV insert.
//
// GB300 design.  A thread-block cluster of two CTAs splits K = 1536 in halves:
// each CTA keeps its half of the normalised xq of all 64 tokens resident in
// shared memory (the B operand, 96 KiB) and streams only its half of every
// weight row, so each weight byte enters the GPU once for all the tokens.
//  * Units of a pair (the same list on both CTAs): for each of its heads (at
//    most two) NOPE (the head's 128 nope rows: one M = 128 tile, N = 64
//    tokens, K = 768) then ABS (the absorption of that head), and then a
//    byte-balancing share of ROPE units: the 64 rope rows of two heads (one
//    M = 128 tile), or of one head (an M = 64 tile, six boxes per CTA) where
//    those finer units balance the pairs better (64 heads on 76 pairs).
//  * The weights are copied at create into 16 KiB tiles (128 rows x 64
//    K-columns, already in the swizzled shared-memory layout), so a producer
//    thread streams each tile with one 16 KiB 1-D bulk TMA copy into a 5-slot
//    ring (one large copy per tile: the copies one thread issues complete
//    one after another, so a 16 KiB copy keeps an SM near its share of HBM
//    bandwidth, and L2 prefetches would queue behind the copies);
//    one thread issues tcgen05.mma from the ring and the resident xq,
//    accumulating in TMEM, and commits each slot back to the producer.  Its
//    shared-memory descriptors are precomputed once and advanced by adding
//    the 16-byte-unit offset of the slot and k step, so an MMA costs about
//    as much to issue as the tensor core takes to run it.
//  * The two K-half partial sums of a NOPE or ROPE tile are exchanged through
//    distributed shared memory (st.async): rank r finishes tokens 32r..32r+31,
//    adding the half of K 0..767 first.  For NOPE it writes the BF16 q of its
//    32 tokens into the B operand of the absorption (64 tokens x 128 rows,
//    swizzled) and copies those rows into the other CTA's, so both hold the
//    q of all 64 tokens; each CTA then multiplies its half of W_UK^T (a copy
//    made at create, [h][c][p]: latent columns 256 r..256 r + 255) by it into
//    TMEM, and the epilogue writes those columns of q_latent.  Every W_UK
//    byte is streamed once.
// Every wait is bounded (MLA_DEVERR_TIMEOUT instead of a hang).
#include <cuda.h>
#include <cuda_bf16.h>

#include "../../include/mla_query.h"
#include "mla_common.cuh"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

namespace {

constexpr int kWideTok = 64;                 // tokens per launch (N of the Q_B GEMM)
constexpr int kWideHalfTok = 32;             // tokens each CTA of the pair finishes
constexpr int kWideKHalf = kQLora / 2;       // 768
constexpr int kWideAtoms = kWideKHalf / 64;  // 12 K atoms of 64 columns (128 B)
static_assert(kWideAtoms == kWideRopeBoxes && kWideAtoms / 2 == kWideSingleBoxes,
              "rope unit boxes");
constexpr int kWideSlots = 5;
// Boxes past the ring that a CTA prefetches into L2 when it starts, before
// the programmatic-dependent-launch wait: the ring fills in about 2 us, and
// the MMAs cannot start before the normalising kernel has run and xq has
// landed, so without them the CTA's share of HBM would idle meanwhile.
// Measured (us per step, B = 64): H = 128 21.35 / 20.95 / 20.95 with 0 / 4 /
// 8 boxes, H = 64 14.69 / 14.55 / 15.37; 16 boxes 22.5 and 17.6.
#ifndef MLA_WIDE_PREFETCH
#define MLA_WIDE_PREFETCH 4
#endif
constexpr int kWidePrefetch = MLA_WIDE_PREFETCH;
constexpr int kWidePrefetch2 = 4;  // the second wave, after the wait (see the xq copies)
constexpr int kWideBox = 128 * 128;          // one 128-row x 128 B box (16 KiB)
constexpr int kWideThreads = 256;
// TMEM columns: Q_B tiles [2 buffers][2 K-quarter partials][64 tokens] at
// 0..255, absorptions [2 heads][2 column tiles][64 tokens] at 256..511.
constexpr int kWideTmemCols = 512;
constexpr int kWideAbsCol = 256;

enum WideUnit { kUnitNope = 0, kUnitAbs = 1, kUnitRope = 2 };

struct WideSmem {
  static constexpr int oXq = 0;                                  // [12][64 rows][128 B]
  static constexpr int oRing = oXq + kWideAtoms * kWideTok * 128;   // 98304
  static constexpr int kQtAtom = kWideTok * 128;                   // 64 token rows of 128 B
  static constexpr int kQtBytes = 2 * kQtAtom;                      // one head: 2 atoms
  static constexpr int oQt = oRing + kWideSlots * kWideBox;         // [2 heads][2][64 rows][128 B]
  static constexpr int oRecv = oQt + 2 * kQtBytes;                  // [128][32] FP32
  static constexpr int oBar = oRecv + 128 * kWideHalfTok * 4;
  // barriers: full[5] empty[5] dready[2] dfree[2] qready[2] absready[2] absfree[2]
  //           recvfull sendok xqready
  static constexpr int kBars = 2 * kWideSlots + 2 + 2 + 2 + 2 + 2 + 1 + 1 + 1;
  static constexpr int oTslot = oBar + kBars * 8;
  static constexpr int kBytes = oTslot + 16;
  static constexpr int kAlloc = kBytes + 1024;  // base aligned up to 1 KiB (swizzle atoms)
};

// K-major SWIZZLE_128B shared-memory matrix descriptor (tcgen05): start
// address, leading offset unused (1), 1024 B between 8-row groups, version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: BF16 x BF16 -> FP32, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of FP32 from TMEM in one load and one wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// The two K-quarter partials of a Q_B tile (columns c and c + 64), added in
// FP32: first quarter first.
__device__ __forceinline__ void tmem_ld_pair(uint32_t taddr, float (&v)[32]) {
  float w[32];
  tmem_ld32(taddr, v);
  tmem_ld32(taddr + kWideTok, w);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __fadd_rn(v[j], w[j]);
}

// 1-D bulk copy from this CTA's shared memory to the shared memory of a CTA
// of the cluster (dst and the mbarrier given as shared::cluster addresses),
// completion counted on that mbarrier in bytes.  16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_s2s_cluster(uint32_t dst, const void* src, uint32_t bytes,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Arrive on the mbarrier at `remote` (a shared::cluster address in the other
// CTA of the pair).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}

// Offset of element (row, col) of a K-major 128 B-swizzled block (col < 64).
__device__ __forceinline__ int sw128(int row, int col) {
  return row * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2;
}

// Units of pair c, heads [h0, h0 + nh) (nh <= 2) and rope units [r0, r0 + nr):
// NOPE of every head, then the ROPE units, then ABS of every head.  The Q_B
// tiles in between give the epilogue time to finish each head's q before its
// absorption needs it, and the step ends on absorptions, whose epilogue needs
// nothing from the other CTA.
// A CTA's units in order: NOPE (one per head of the pair), ROPE (the pair's
// two-head units, then its one-head units), ABS (one per head).
struct WideSeq {
  int h0, nh, d0, nd, s0, ns, ndouble;
  __device__ int units() const { return 2 * nh + nd + ns; }
  __device__ int kind(int u) const {
    if (u < nh) return kUnitNope;
    if (u < nh + nd + ns) return kUnitRope;
    return kUnitAbs;
  }
  __device__ bool single(int u) const { return u >= nh + nd && u < nh + nd + ns; }
  // head of a NOPE/ABS unit; for a ROPE unit, the two-head unit's index
  // (heads 2 i, 2 i + 1), or the head of a one-head unit
  __device__ int head(int u) const {
    if (u < nh) return h0 + u;
    if (u < nh + nd) return d0 + (u - nh);
    if (u < nh + nd + ns) return 2 * ndouble + s0 + (u - nh - nd);
    return h0 + (u - nh - nd - ns);
  }
  __device__ int boxes(int u) const {
    const int k = kind(u);
    return k == kUnitAbs ? 4 : single(u) ? kWideSingleBoxes : kWideAtoms;
  }
};

// Tile index in the packed copies (pack_wide_weights): NOPE tile (h, K half,
// atom); two-head ROPE tile (unit, K half, atom) after all NOPE tiles;
// one-head ROPE tile (head, K half, pair of atoms) after the ndouble
// two-head units' tiles; W_UK^T tile (h, 128-column tile ct, 64-row atom
// pa), where the CTA of rank `half` takes latent columns 256 half.. (ct =
// 2 half + bx / 2, pa = bx % 2).
__device__ __forceinline__ int64_t wide_qb_tile(int heads, int ndouble, int kind, int h, int half,
                                                int bx, bool single) {
  if (kind == kUnitNope) return (int64_t)(h * 2 + half) * kWideAtoms + bx;
  const int64_t rope0 = (int64_t)heads * 2 * kWideAtoms;
  if (!single) return rope0 + (int64_t)(h * 2 + half) * kWideAtoms + bx;
  return rope0 + (int64_t)ndouble * 2 * kWideAtoms +
         (int64_t)((h - 2 * ndouble) * 2 + half) * kWideSingleBoxes + bx;
}
__device__ __forceinline__ const uint8_t* wide_tile(const DecodeArgs& a, int ndouble, int kind,
                                                    int h, int half, int bx, bool single) {
  if (kind == kUnitAbs) return a.wide_ukt + ((size_t)h * 8 + 4 * half + bx) * kWideBox;
  return a.wide_qb + (size_t)wide_qb_tile(a.heads, ndouble, kind, h, half, bx, single) * kWideBox;
}

// Checks builds: whether wide_tile's box lies inside its packed copy (the
// sizes wide_qb_bytes and wide_ukt_bytes allocate) and in its unit's range.
__device__ __forceinline__ bool wide_tile_in_bounds(const DecodeArgs& a, int ndouble, int kind,
                                                    int h, int half, int bx, bool single) {
  const int64_t H = a.heads;
  if (half != 0 && half != 1) return false;
  if (kind == kUnitAbs) return h >= 0 && h < H && bx >= 0 && bx < 4;
  if (kind == kUnitNope) {
    if (h < 0 || h >= H || bx < 0 || bx >= kWideAtoms) return false;
  } else if (!single) {
    if (h < 0 || h >= ndouble || bx < 0 || bx >= kWideAtoms) return false;
  } else if (h < 2 * ndouble || h >= H || bx < 0 || bx >= kWideSingleBoxes) {
    return false;
  }
  const int64_t idx = wide_qb_tile(a.heads, ndouble, kind, h, half, bx, single);
  return idx >= 0 && idx < (H + (H + 1) / 2) * 2 * kWideAtoms;
}

__global__ void __launch_bounds__(kWideThreads, 1)
    mla_wide_kernel(const DecodeArgs a, const __grid_constant__ WideSplit split) {
  using S = WideSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kWideSlots;
  uint64_t* dready = bars + 2 * kWideSlots;
  uint64_t* dfree = dready + 2;
  uint64_t* qready = dfree + 2;
  uint64_t* absready = qready + 2;  // one absorption accumulator per head of the pair
  uint64_t* absfree = absready + 2;
  uint64_t* recvfull = absfree + 2;  // the other CTA's partials landed (one buffer)
  uint64_t* sendok = recvfull + 1;    // the other CTA has read what this one sent
  uint64_t* xqready = sendok + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::oTslot);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x;
  const int pair = i >> 1, rank = i & 1;  // cluster (2, 1, 1)
  const uint32_t peer = (uint32_t)(rank ^ 1);
  const int H = a.heads;
  const WideSeq seq{split.head[pair],     split.head[pair + 1] - split.head[pair],
                    split.dbl[pair],      split.dbl[pair + 1] - split.dbl[pair],
                    split.sgl[pair],      split.sgl[pair + 1] - split.sgl[pair],
                    split.ndouble};
  const int nu = seq.units();

  if (tid == 0) {
    for (int s = 0; s < kWideSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dready[b], 1);
      mbar_init(&dfree[b], 128);
      // q tile of head b: this CTA's rows (one arrival) and the other CTA's
      // (its bulk copies, counted in bytes; armed here)
      mbar_init(&qready[b], 2);
      mbar_arrive_expect_tx(&qready[b], S::kQtBytes / 2);
    }
    mbar_init(recvfull, 1);
    mbar_init(sendok, 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&absready[j], 1);
      mbar_init(&absfree[j], 128);
    }
    mbar_init(xqready, 1);
    // the other CTA's bytes: its first tile half
    mbar_arrive_expect_tx(recvfull, 128 * kWideHalfTok * 4);
    mbar_fence_init();
    pdl_launch_dependents();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tslot)),
                 "r"(kWideTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers initialised and armed
  if (tid == 0) trace_stamp(a, 0);
  const uint32_t tmem = *tslot;
  bool timed_out = false;

  if (warp == 0 || warp == 3) {
    // ================= producers: weight tiles, no PDL wait ============
    // Two issuing threads in different warps, boxes alternating between
    // them: copies one thread issues complete one after another, and two
    // issuers stream about 45 GB/s per SM against 35 for one (16 KiB
    // copies, measured).  Box k goes to slot k % kWideSlots; its issuer
    // waits for the consumption of box k - kWideSlots in that slot, which
    // only box k's own issuer can be waiting for, so no slot runs more than
    // one phase ahead of a wait on it.
    if (lane == 0) {
      const int me = warp == 0 ? 0 : 1;
      const uint64_t pol = l2_policy_evict_first();
      int k = 0;  // box counter over all units
      for (int u = 0; u < nu; ++u) {
        const int kind = seq.kind(u), h = seq.head(u), nb = seq.boxes(u);
        for (int bx = 0; bx < nb; ++bx, ++k) {
          if ((k & 1) != me) continue;
          const int slot = k % kWideSlots;
          if (k >= kWideSlots &&
              !mbar_wait_bounded(&empty[slot], (uint32_t)(((k / kWideSlots) - 1) & 1), kWaitLimit))
            timed_out = true;
          mbar_arrive_expect_tx(&full[slot], kWideBox);
          if (MLA_IN_BOUNDS(a, wide_tile_in_bounds(a, seq.ndouble, kind, h, rank, bx, seq.single(u)), 5) &&
              MLA_IN_BOUNDS(a, slot >= 0 && slot < kWideSlots, 6))
            bulk_g2s_hint(smem + S::oRing + slot * kWideBox,
                          wide_tile(a, seq.ndouble, kind, h, rank, bx, seq.single(u)), kWideBox,
                          &full[slot], pol);
          if (bx == 0 && u < 4) trace_stamp(a, 24 + u);  // unit u's first box issued
        }
      }
      // every box this thread issued is consumed before the CTA may leave
      for (int kk = k - kWideSlots > 0 ? k - kWideSlots : 0; kk < k; ++kk)
        if ((kk & 1) == me)
          (void)mbar_wait_bounded(&empty[kk % kWideSlots], (uint32_t)((kk / kWideSlots) & 1),
                                  kWaitLimit);
    }
  } else if (warp == 1) {
    // ================= MMA issuer ==================================
    if (lane == 0) {
      if (!mbar_wait_bounded(xqready, 0u, kWaitLimit)) timed_out = true;
      trace_stamp(a, 2);
      tc_fence_after();
      // Descriptors of the ring, the resident xq and the q tiles; an operand
      // at byte offset o from one of them is its descriptor plus o / 16 (the
      // start-address field, which no offset here carries out of).
      const uint64_t dring = umma_desc(smem_u32(smem + S::oRing));
      const uint64_t dxq = umma_desc(smem_u32(smem + S::oXq));
      const uint64_t dqt = umma_desc(smem_u32(smem + S::oQt));
      constexpr uint32_t idq = umma_idesc(128, kWideTok);
      constexpr uint32_t idq64 = umma_idesc(64, kWideTok);
      int nq = 0, na = 0;  // Q_B tiles, absorptions so far
      int slot = 0;
      uint32_t fphase = 0;  // parity of the slot's next full phase
      for (int u = 0; u < nu; ++u) {
        const int kind = seq.kind(u), nb = seq.boxes(u);
        uint32_t dcol;
        if (kind == kUnitAbs) {
          // the q tile of this head is written; the previous absorption read out
          if (!mbar_wait_bounded(&qready[na], 0u, kWaitLimit)) timed_out = true;
          if (na >= 2 &&
              !mbar_wait_bounded(&absfree[na & 1], (uint32_t)(((na >> 1) - 1) & 1), kWaitLimit))
            timed_out = true;
          tc_fence_after();
          dcol = kWideAbsCol + 128 * (na & 1);
        } else {
          const int b = nq & 1;
          if (nq >= 2 && !mbar_wait_bounded(&dfree[b], (uint32_t)(((nq >> 1) - 1) & 1), kWaitLimit))
            timed_out = true;
          tc_fence_after();
          dcol = 128 * b;
        }
        // A Q_B tile accumulates its K half in two partials (the first and
        // the second half of its boxes, 24 k16 steps each), which the
        // epilogue adds in FP32: the tensor core's accumulation error grows
        // with the length of the chain.
        const int half_nb = nb / 2;
        for (int bx = 0; bx < nb; ++bx) {
          if (!mbar_wait_bounded(&full[slot], fphase, kWaitLimit)) timed_out = true;
          // TMEM: a Q_B partial at dcol + 64 * (bx >= half_nb), an absorption
          // column tile at dcol + 64 * (bx / 2), each 64 columns wide
          if (!MLA_IN_BOUNDS(a, dcol >= 0 && dcol + (kind == kUnitAbs ? 128 : 128) <= kWideTmemCols, 6))
            break;
          tc_fence_after();
          const uint64_t da = dring + (uint64_t)(slot * (kWideBox >> 4));
          if (kind == kUnitAbs) {
            // W_UK^T rows 128 ct.. of this CTA's half, q^T atom pa (nope rows
            // 64 pa..64 pa + 63) of all 64 tokens
            const int ct = bx >> 1, pa = bx & 1;
            const uint64_t db = dqt + (uint64_t)(na * (S::kQtBytes >> 4) + pa * (S::kQtAtom >> 4));
            const uint32_t dt = tmem + dcol + kWideTok * ct;
            umma(dt, da, db, idq, (uint32_t)pa);
            umma(dt, da + 2, db + 2, idq, 1u);
            umma(dt, da + 4, db + 4, idq, 1u);
            umma(dt, da + 6, db + 6, idq, 1u);
          } else if (kind == kUnitRope && seq.single(u)) {
            // one head's 64 rope rows, K atoms 2 bx and 2 bx + 1 (8 KiB
            // each): M = 64, rows in TMEM lanes 32 (r / 16) + r % 16
            const uint64_t db = dxq + (uint64_t)(2 * bx * ((kWideTok * 128) >> 4));
            const uint64_t da1 = da + (uint64_t)((64 * 128) >> 4);
            const uint64_t db1 = db + (uint64_t)((kWideTok * 128) >> 4);
            const uint32_t dt = tmem + dcol + kWideTok * (bx >= half_nb);
            umma(dt, da, db, idq64, (uint32_t)(bx % half_nb));
            umma(dt, da + 2, db + 2, idq64, 1u);
            umma(dt, da + 4, db + 4, idq64, 1u);
            umma(dt, da + 6, db + 6, idq64, 1u);
            umma(dt, da1, db1, idq64, 1u);
            umma(dt, da1 + 2, db1 + 2, idq64, 1u);
            umma(dt, da1 + 4, db1 + 4, idq64, 1u);
            umma(dt, da1 + 6, db1 + 6, idq64, 1u);
          } else {
            const uint64_t db = dxq + (uint64_t)(bx * ((kWideTok * 128) >> 4));
            const uint32_t dt = tmem + dcol + kWideTok * (bx >= half_nb);
            umma(dt, da, db, idq, (uint32_t)(bx % half_nb));
            umma(dt, da + 2, db + 2, idq, 1u);
            umma(dt, da + 4, db + 4, idq, 1u);
            umma(dt, da + 6, db + 6, idq, 1u);
          }
          umma_commit(&empty[slot]);  // the slot is free once these MMAs are done
          if (++slot == kWideSlots) {
            slot = 0;
            fphase ^= 1u;
          }
        }
        if (kind == kUnitAbs) {
          umma_commit(&absready[na & 1]);
          ++na;
        } else {
          umma_commit(&dready[nq & 1]);
          ++nq;
        }
        if (u < 16) trace_stamp(a, 8 + u);  // unit u's MMAs issued
      }
    }
  } else {
    // ================= warps 2, 4-7: this K half of xq, then the epilogue
    if (warp == 2 && lane == 0 && kWidePrefetch > 0) {
      // the boxes just past the ring, into L2 (weights: no PDL wait)
      int k = 0;
      for (int u = 0; u < nu && k < kWideSlots + kWidePrefetch; ++u) {
        const int kind = seq.kind(u), h = seq.head(u), nb = seq.boxes(u);
        for (int bx = 0; bx < nb && k < kWideSlots + kWidePrefetch; ++bx, ++k)
          if (k >= kWideSlots)
            bulk_prefetch_l2(wide_tile(a, seq.ndouble, kind, h, rank, bx, seq.single(u)),
                             kWideBox);
      }
    }
    // The normalising kernel launched just before wrote xq in this tile's
    // layout; twelve bulk copies (one per 64-column atom) bring this half in.
    pdl_wait();
    if (warp == 2) {
      // one 8 KiB atom per lane: copies issued by different threads proceed
      // side by side
      if (lane == 0) {
        trace_stamp(a, 3);
        mbar_arrive_expect_tx(xqready, kWideAtoms * kWideTok * 128);
      }
      __syncwarp();
      if (lane < kWideAtoms) {
        const uint8_t* src = a.wide_xq + ((size_t)rank * kWideAtoms + lane) * (kWideTok * 128);
        bulk_g2s(smem + S::oXq + lane * (kWideTok * 128), src, kWideTok * 128, xqready);
      }
      // A second wave of kWidePrefetch2 boxes into L2 once xq is on its way:
      // the ring and the first wave have landed by now, and the slots free
      // only when the MMAs start.  Measured at B = 64 (us per step, waves of
      // 3 / 4 / 5 / 6 boxes against none): H = 128 19.70 / 19.65 / 19.66 /
      // 19.72 against 20.19, H = 96 17.31 / 17.26 / 17.24 / 17.28 against
      // 17.56.  CTAs with more than 16 boxes take it (more than 28: H = 96
      // 16.54, H = 64 13.57 us; more than 16: 16.38 and 13.54, 24 and 32
      // tokens at H = 64 unchanged).
      if (lane == 31) {
        int total = 0;
        for (int u = 0; u < nu; ++u) total += seq.boxes(u);
        if (total > 16) {
          const int k0 = kWideSlots + kWidePrefetch, k1 = k0 + kWidePrefetch2;
          int k = 0;
          for (int u = 0; u < nu && k < k1; ++u) {
            const int kind = seq.kind(u), h = seq.head(u), nb = seq.boxes(u);
            for (int bx = 0; bx < nb && k < k1; ++bx, ++k)
              if (k >= k0)
                bulk_prefetch_l2(wide_tile(a, seq.ndouble, kind, h, rank, bx, seq.single(u)),
                                 kWideBox);
          }
        }
      }
    }

    // The paged KV insert of the launch's tokens, one warp a token, before
    // the first epilogue is due (its inputs are current after the wait).
    // In the normalising kernel it lengthened the chain before the MMAs:
    // B = 64 H = 128 fp8_ds_mla 19.73 -> 19.05 us, H = 64 14.40 -> 13.55.
    if (warp == 4)
      for (int t = (int)blockIdx.x; t < a.batch; t += (int)gridDim.x) kv_insert_warp(a, t, lane);
    if (warp >= 4) {
      // ================= epilogue: TMEM lanes 0..127 ===================
      const int m = tid - 128;  // row of the tile = TMEM lane
      const uint32_t lane_base = (uint32_t)(32 * (warp - 4)) << 16;
      const int my0 = kWideHalfTok * rank, peer0 = kWideHalfTok * (rank ^ 1);
      const float qsi = load_qsi(a);
      int nq = 0, na = 0;
      for (int u = 0; u < nu; ++u) {
        const int kind = seq.kind(u), h = seq.head(u);
        if (kind == kUnitAbs) {
          const int ab = na & 1;
          if (!mbar_wait_bounded(&absready[ab], (uint32_t)((na >> 1) & 1), kWaitLimit))
            timed_out = true;
          tc_fence_after();
          // latent column 256 rank + 128 ct + m of all 64 tokens, 32 at a time
#pragma unroll 1
          for (int part = 0; part < 4; ++part) {
            const int ct = part >> 1, t0 = kWideHalfTok * (part & 1);
            float v[32];
            tmem_ld32(tmem + lane_base + kWideAbsCol + 128 * ab + kWideTok * ct + t0, v);
            const int nt_here = min(kWideHalfTok, a.batch - t0);
            if (nt_here > 0 && MLA_IN_BOUNDS(a, h >= 0 && h < H && 256 * rank + 128 * ct + m < kKvLora, 7))
              put_q_run(a, a.q_latent,
                        (int64_t)t0 * a.ql_ts + (int64_t)h * a.ql_hs + 256 * rank + 128 * ct + m,
                        a.ql_ts, v, nt_here, qsi);
          }
          tc_fence_before();
          mbar_arrive(&absfree[ab]);
          ++na;
          if (m == 0 && u < 16) trace_stamp(a, 28 + u);  // unit u's epilogue done
          continue;
        }
        // ---- a Q_B tile: this K half for 64 tokens -> exchange -> q --------
        const int b = nq & 1;
        if (!mbar_wait_bounded(&dready[b], (uint32_t)((nq >> 1) & 1), kWaitLimit)) timed_out = true;
        tc_fence_after();
        float q[kWideHalfTok];
        // the other CTA's tokens of this row go into its receive buffer b
        tmem_ld_pair(tmem + lane_base + 128 * b + peer0, q);
        // the other CTA has read what this one sent for the previous tile
        if (nq >= 1 && !mbar_wait_bounded(sendok, (uint32_t)((nq - 1) & 1), kWaitLimit))
          timed_out = true;
        {
          const uint32_t rb = mapa_shared(smem_u32(recvfull), peer);
          // row m of the other CTA's receive buffer; 16-byte chunk c (tokens
          // 4c..4c+3) at position c ^ (m % 8), so that reading a row chunk by
          // chunk is free of bank conflicts
          const uint32_t dst = smem_u32(smem + S::oRecv + m * kWideHalfTok * 4);
#pragma unroll
          for (int c = 0; c < kWideHalfTok / 4; ++c)
            st_async_v4(mapa_shared(dst + 16 * (c ^ (m & 7)), peer), q[4 * c], q[4 * c + 1],
                        q[4 * c + 2], q[4 * c + 3], rb);
        }
        // this CTA's tokens: its K half plus the other CTA's, K 0..767 first
        tmem_ld_pair(tmem + lane_base + 128 * b + my0, q);
        tc_fence_before();
        mbar_arrive(&dfree[b]);
        if (!mbar_wait_bounded(recvfull, (uint32_t)(nq & 1), kWaitLimit)) timed_out = true;
        const float4* rcv = reinterpret_cast<const float4*>(smem + S::oRecv + m * kWideHalfTok * 4);
#pragma unroll
        for (int c = 0; c < kWideHalfTok / 4; ++c) {
          const float4 r = rcv[c ^ (m & 7)];
          const float rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            q[4 * c + e] = rank == 0 ? q[4 * c + e] + rv[e] : rv[e] + q[4 * c + e];
        }
        // the buffer is read: re-arm it for its next use, then let the other CTA send
        named_barrier(5, 128);
        if (m == 0) {
          mbar_arrive_expect_tx(recvfull, 128 * kWideHalfTok * 4);
          mbar_arrive_remote(mapa_shared(smem_u32(sendok), peer));
        }
        if (kind == kUnitNope) {
          // q^T tile of head j of the pair: [token 0..63][row m] BF16,
          // K-major swizzled, two atoms (each head has its own tile); this
          // CTA writes its 32 token rows and copies them into the other CTA's
          const int j = h - seq.h0;
          if (!MLA_IN_BOUNDS(a, j == 0 || j == 1, 8)) continue;
          uint8_t* qt = smem + S::oQt + j * S::kQtBytes;
          uint8_t* qa = qt + (m >> 6) * S::kQtAtom;
#pragma unroll
          for (int tl = 0; tl < kWideHalfTok; ++tl)
            *reinterpret_cast<uint16_t*>(qa + sw128(my0 + tl, m & 63)) = f2bf_bits(q[tl]);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          named_barrier(5, 128);
          if (m == 0) {
            const uint32_t rq = mapa_shared(smem_u32(&qready[j]), peer);
            for (int at = 0; at < 2; ++at) {
              uint8_t* rows = qt + at * S::kQtAtom + my0 * 128;  // 32 rows of 128 B
              bulk_s2s_cluster(mapa_shared(smem_u32(rows), peer), rows, kWideHalfTok * 128, rq);
            }
            mbar_arrive(&qready[j]);
          }
        } else if (seq.single(u)) {
          // head h: row 16 (m / 32) + m % 32 in TMEM lanes with m % 32 < 16
          if ((m & 31) < 16 && MLA_IN_BOUNDS(a, h >= 0 && h < H, 7)) {
            const int nt_here = min(kWideHalfTok, a.batch - my0);
            put_q_run(a, a.q_pe,
                      (int64_t)my0 * a.qp_ts + (int64_t)h * a.qp_hs + 16 * (m >> 5) + (m & 15),
                      a.qp_ts, q, nt_here, qsi);
          }
        } else if (2 * h + (m >> 6) < H) {  // rows 0..63: head 2h, 64..127: head 2h + 1
          const int hr = 2 * h + (m >> 6);
          const int nt_here = min(kWideHalfTok, a.batch - my0);
          put_q_run(a, a.q_pe, (int64_t)my0 * a.qp_ts + (int64_t)hr * a.qp_hs + (m & 63), a.qp_ts,
                    q, nt_here, qsi);
        }
        ++nq;
        if (m == 0 && u < 16) trace_stamp(a, 28 + u);  // unit u's epilogue done
      }
      if (m == 0) trace_stamp(a, 6);
    }
  }

  if (timed_out) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kWideTmemCols)
                 : "memory");
  }
  // neither CTA leaves while the other may still write into its shared memory
  cluster_sync_relaxed();
  if (tid == 0) trace_stamp(a, 7);
}

// RMSNorm of the q_a rows of up to 64 tokens for the wide kernel (page
// "mla.query": xq = bf16((q_a * rr) * gamma_q), rr = 1/sqrt(sum q_a^2 / 1536 +
// eps)), written as q_c and into the wide CTAs' swizzled tile layout (rows of
// tokens beyond the batch as zeros).  One CTA of 192 threads per token:
// thread j takes columns 8j..8j+7.  (The paged KV insert runs in the wide
// kernel: every microsecond this kernel takes delays the wide kernel's
// MMAs.)
__global__ void __launch_bounds__(192) mla_wide_norm_kernel(const DecodeArgs a) {
  __shared__ float part[6];
  const int t = blockIdx.x, j = threadIdx.x, lane = j & 31, warp = j >> 5;
  pdl_launch_dependents();  // the wide kernel streams weights meanwhile
  if (j == 0) trace_stamp(a, 60);  // normalising CTA t started
  pdl_wait();
  if (j == 0) trace_stamp(a, 61);  // its wait passed
  uint4 o = make_uint4(0, 0, 0, 0);
  if (t < a.batch) {
    const uint4 v = *reinterpret_cast<const uint4*>(a.q_a + (int64_t)t * a.q_a_stride + 8 * j);
    const uint4 gv = *reinterpret_cast<const uint4*>(a.gamma_q + 8 * j);
    const uint32_t ww[4] = {v.x, v.y, v.z, v.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ss = fmaf(bf16lo(ww[e]), bf16lo(ww[e]), ss);
      ss = fmaf(bf16hi(ww[e]), bf16hi(ww[e]), ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    const float total = ((((part[0] + part[1]) + part[2]) + part[3]) + part[4]) + part[5];
    const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, 1536.0f), a.eps));
    uint32_t r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      r[e] = rms_scale_bf16x2(ww[e], rr, gw[e]);
    o = make_uint4(r[0], r[1], r[2], r[3]);
    if (a.q_c != nullptr) *reinterpret_cast<uint4*>(a.q_c + (int64_t)t * kQLora + 8 * j) = o;
  }
  // chunk j: K half j / 96, atom (j % 96) / 8, 16-byte chunk j % 8 of row t
  const int half = j / 96, cc = j % 96, at = cc >> 3, c = cc & 7;
  const size_t xo = ((size_t)(half * kWideAtoms + at) * kWideTok) * 128 + t * 128 + ((c ^ (t & 7)) << 4);
  if (MLA_IN_BOUNDS(a, t < kWideTok && xo + 16 <= (size_t)2 * kWideAtoms * kWideTok * 128, 9))
    *reinterpret_cast<uint4*>(a.wide_xq + xo) = o;
  __syncthreads();
  if (j == 0) trace_stamp(a, 62);  // its rows written
}

// Tiled copies for the wide kernel, each 16-byte chunk (row r, 8 K-columns
// from 8 j) at r * 128 + ((j ^ (r % 8)) * 16) of its 16 KiB tile: the K-major
// 128-byte-swizzled layout the kernel's shared-memory descriptors read.
//   W_QB tiles: NOPE (h, half, atom) = rows 192 h .. 192 h + 127, columns
//   768 half + 64 atom ..; then two-head ROPE units (u, half, atom) = rope
//   rows of head 2u (tile rows 0..63) and 2u + 1 (rows 64..127, zeros past
//   the last head); then one-head ROPE units (head 2 ndouble + v, half, box)
//   = the head's rope rows at atoms 2 box (rows 0..63) and 2 box + 1.
//   W_UK^T tiles (h, ct, pa): row r = latent column 128 ct + r, K = W_UK row
//   64 pa + k.
__global__ void pack_wide_qb_kernel(const uint16_t* __restrict__ w_qb, uint8_t* __restrict__ out,
                                    int heads, int ndouble) {
  const int singles = heads > 2 * ndouble ? heads - 2 * ndouble : 0;
  const int64_t nope_tiles = (int64_t)heads * 2 * kWideAtoms;
  const int64_t double_tiles = (int64_t)ndouble * 2 * kWideAtoms;
  const int64_t tiles = nope_tiles + double_tiles + (int64_t)singles * 2 * kWideSingleBoxes;
  const int64_t n = tiles * 128 * 8;  // 16-byte chunks
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(e & 7), r = (int)((e >> 3) & 127);
    const int64_t tile = e >> 10;
    int64_t row = -1;
    int col = 0;  // first K column of the chunk
    if (tile < nope_tiles) {
      const int at = (int)(tile % kWideAtoms), half = (int)((tile / kWideAtoms) & 1);
      row = (tile / (2 * kWideAtoms)) * kHeadRows + r;
      col = kWideKHalf * half + 64 * at;
    } else if (tile < nope_tiles + double_tiles) {
      // two-head unit (u, half, atom): rows 0..63 = head 2u's rope rows,
      // 64..127 = head 2u + 1's (zeros past the last head)
      const int at = (int)(tile % kWideAtoms), half = (int)((tile / kWideAtoms) & 1);
      const int64_t hd = 2 * (tile / (2 * kWideAtoms) - heads) + (r >> 6);
      if (hd < heads) row = hd * kHeadRows + kNope + (r & 63);
      col = kWideKHalf * half + 64 * at;
    } else {
      // one-head unit (head 2 ndouble + v, half, box): rows 0..63 = its rope
      // rows at K atom 2 box, rows 64..127 = the same rows at K atom 2 box + 1
      const int64_t t = tile - nope_tiles - double_tiles;
      const int bx = (int)(t % kWideSingleBoxes), half = (int)((t / kWideSingleBoxes) & 1);
      row = (2 * (int64_t)ndouble + t / (2 * kWideSingleBoxes)) * kHeadRows + kNope + (r & 63);
      col = kWideKHalf * half + 64 * (2 * bx + (r >> 6));
    }
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row >= 0) v = *reinterpret_cast<const uint4*>(w_qb + row * kQLora + col + 8 * j);
    *reinterpret_cast<uint4*>(out + tile * kWideBox + r * 128 + ((j ^ (r & 7)) << 4)) = v;
  }
}

__global__ void pack_wide_ukt_kernel(const uint16_t* __restrict__ w_uk, uint8_t* __restrict__ out,
                                     int heads) {
  const int64_t n = (int64_t)heads * 8 * 128 * 8;  // 16-byte chunks
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(e & 7), r = (int)((e >> 3) & 127);
    const int64_t tile = e >> 10;
    const int pa = (int)(tile & 1), ct = (int)((tile >> 1) & 3);
    const int64_t h = tile >> 3;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p0 = 64 * pa + 8 * j + 2 * i;
      const uint32_t lo = w_uk[(h * kNope + p0) * kKvLora + 128 * ct + r];
      const uint32_t hi = w_uk[(h * kNope + p0 + 1) * kKvLora + 128 * ct + r];
      w[i] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(out + tile * kWideBox + r * 128 + ((j ^ (r & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaLaunchConfig_t wide_config(int ctas, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(kWideThreads, 1, 1);
  cfg.dynamicSmemBytes = WideSmem::kAlloc;
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

int wide_tokens() { return kWideTok; }

cudaError_t prepare_wide_kernel() {
  static_assert(WideSmem::kAlloc <= 232448, "shared memory budget");
  return cudaFuncSetAttribute(mla_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              WideSmem::kAlloc);
}

bool wide_kernel_fits(int ctas) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = wide_config(ctas, nullptr, attr);
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, mla_wide_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return clusters >= ctas / 2;
}

size_t wide_qb_bytes(int heads) {
  return (size_t)(heads + (heads + 1) / 2) * 2 * kWideAtoms * kWideBox;
}
size_t wide_ukt_bytes(int heads) { return (size_t)heads * 8 * kWideBox; }

cudaError_t pack_wide_weights(const uint16_t* w_qb, const uint16_t* w_uk, uint8_t* qb_tiles,
                              uint8_t* ukt_tiles, int heads, int ndouble, cudaStream_t stream) {
  pack_wide_qb_kernel<<<512, 256, 0, stream>>>(w_qb, qb_tiles, heads, ndouble);
  pack_wide_ukt_kernel<<<512, 256, 0, stream>>>(w_uk, ukt_tiles, heads);
  return cudaGetLastError();
}

size_t wide_xq_bytes() { return (size_t)2 * kWideAtoms * kWideTok * 128; }

cudaError_t launch_wide(const DecodeArgs& a, const WideSplit& sp, int ctas, cudaStream_t stream) {
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kWideTok, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, mla_wide_norm_kernel, a);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = wide_config(ctas, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_wide_kernel, a, sp);
}

}  // namespace mla
