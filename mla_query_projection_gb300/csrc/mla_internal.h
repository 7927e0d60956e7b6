// mla_internal.h - host/device shared definitions of the MLA query library
// (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Geometry fixed by the method (page "mla.query", class MlaQuery).
constexpr int kQLora = 1536;   // q_a width
constexpr int kNope = 128;     // nope rows per head
constexpr int kRope = 64;      // rope rows per head
constexpr int kHeadRows = 192; // Q_B rows per head
constexpr int kKvLora = 512;   // latent width
constexpr int kRowE4m3 = 576;  // per-tensor cache row bytes
constexpr int kRowDs = 656;    // fp8_ds_mla cache row bytes
constexpr int kDsScales = 512; // byte offset of the four FP32 tile scales
constexpr int kDsRope = 528;   // byte offset of the BF16 k_pe
constexpr int kRowElems = 576;   // a gathered query row: 512 latent + 64 rope
constexpr int kMaxRowHeads = 1024;  // heads per token of a gathered query buffer
constexpr int kRowNvfp4 = 352;  // nvfp4_ds_mla cache row bytes
constexpr int kNvScales = 256;  // byte offset of the 32 E4M3 block scales
constexpr int kNvRope = 288;    // byte offset of the E4M3 k_pe

// Work units of the fused kernel.
constexpr int kRowBytes = kQLora * 2;        // one Q_B row in global memory (3072 B)
constexpr int kUkCols = 64;                  // latent columns per W_UK unit
constexpr int kUkUnitsPerHead = kKvLora / kUkCols;  // 8
constexpr int kUkUnitBytes = kNope * kUkCols * 2;   // 16 KiB
// Combined per-head list of the second phase: 8 W_UK units then 64 rope rows.
constexpr int kItemsPerHead = kUkUnitsPerHead + kRope;                       // 72
constexpr int64_t kItemBytesPerHead = (int64_t)kUkUnitsPerHead * kUkUnitBytes +
                                      (int64_t)kRope * kRowBytes;            // 327680

// Tasks of the absorbing kernels: 16 nope rows of one head (their Q_B rows
// and the matching W_UK rows).
constexpr int kTaskRows = 16;
constexpr int kTasksPerHead = kNope / kTaskRows;       // 8
constexpr int kTaskUkBytes = kTaskRows * kKvLora * 2;  // 16 KiB

// Units of the wide kernel in 16 KiB boxes per CTA of a pair: a head (its
// nope rows' K half, 12 boxes, and its half of W_UK^T, 4), a two-head rope
// unit (one box per 64-column K atom of a half), a single-head rope unit
// (one box per two atoms).
constexpr int kWideHeadBoxes = 16;
constexpr int kWideRopeBoxes = 12;
constexpr int kWideSingleBoxes = 6;

struct DecodeArgs {
  const uint16_t* w_qb;      // [H*192][1536]
  // W_UK repacked as contiguous pre-swizzled 64-column units (see
  // repack_w_uk), or null to load the caller's [H][128][512] through the
  // tensor map.
  const uint8_t* w_uk_packed;
  const uint16_t* gamma_q;   // [1536]
  const uint16_t* gamma_kv;  // [512]
  const uint16_t* q_a;       // [B][q_a_stride]
  const uint16_t* kv_c;      // [B][kv_c_stride]
  const uint16_t* k_pe;      // [B][k_pe_stride]
  int64_t q_a_stride, kv_c_stride, k_pe_stride;  // elements
  const int64_t* slots;      // [B]
  uint8_t* cache;            // [num_pages][page_size][row]
  int64_t num_pages;
  int page_size;
  int layout;
  const float* k_scale;      // [1] (per-tensor layout)
  uint16_t* q_latent;        // [B][H][512] by default, see ql_ts / ql_hs
  uint16_t* q_pe;            // [B][H][64] by default, see qp_ts / qp_hs
  // Output element (t, h, i) of q_latent is q_latent[t * ql_ts + h * ql_hs + i],
  // of q_pe q_pe[t * qp_ts + h * qp_hs + i], in output elements (BF16, or
  // bytes for FP8 queries).  Contiguous outputs: H*512, 512, H*64, 64; the
  // gathered query rows [B][q_heads][576]: q_heads*576, 576 for both, with
  // q_pe = q_latent + 512.
  int64_t ql_ts, ql_hs, qp_ts, qp_hs;
  uint16_t* q_c;             // [B][1536] or null
  // scratch (device)
  uint16_t* qn;              // [groups][NT][H][128] BF16 nope values
  const uint16_t* w_uk;      // [H][128][512] (absorbing kernel)
  float* partial;            // [H*8 tasks][NT][512] FP32 partial absorptions
  uint32_t* ready;           // [groups][H] nope rows finished per head
  uint32_t* finished;        // [1] CTAs finished (last one re-arms the counters)
  uint32_t* err;             // [1] MLA_DEVERR_* bits
  int heads;
  int batch;
  int groups;                // token groups (grid.y)
  float eps;
  // Per-tensor FP8 query outputs (page "mla.query", method kernel, the FP8
  // query epilogue): q_latent and q_pe hold E4M3 codes of
  // bf16(v) * *q_scale_inv; nullptr for BF16 outputs.
  const float* q_scale_inv;
  // Wide kernel: normalised xq of up to 64 tokens, laid out as the wide CTAs'
  // swizzled shared-memory tiles ([2 K halves][12 atoms][64 rows][128 B]).
  uint8_t* wide_xq;
  // Wide kernel: W_QB and W_UK^T copied at create into 16 KiB tiles in the
  // swizzled shared-memory layout (see pack_wide_weights).
  const uint8_t* wide_qb;
  const uint8_t* wide_ukt;
  // Timeline records (builds with MLA_TRACE only; null otherwise):
  // per CTA kTraceSlots globaltimer stamps, see mla_fused.cu.
  uint64_t* trace;
};

constexpr int kTraceSlots = 64;

// Per-CTA ranges of the absorbing kernel (tasks of 16 nope rows + W_UK rows,
// then rope rows), computed on the host.
constexpr int kMaxCtas = 256;
struct AbsSplit {
  uint16_t task[kMaxCtas + 1];
  uint16_t rope[kMaxCtas + 1];
};
void make_abs_split(int heads, int ctas, AbsSplit* sp);
// Split of the paired absorbing kernel (clusters of two CTAs): the heads of
// pair c are [head[c], head[c + 1]) (at most two), rank r of the pair takes
// nope tasks 4r..4r+3 of each; rope rows [rope[i], rope[i + 1]) of CTA i.
struct PairSplit {
  uint16_t head[kMaxCtas / 2 + 1];
  uint16_t rope[kMaxCtas + 1];
};
// Fills `sp` for `ctas` (even) CTAs; false if some pair would get more than
// two heads.  Heads are spread evenly over the pairs, or, with `heads_first`
// and no more heads than pairs, pair c takes head c and the pairs past the
// last head take rope rows only.
bool make_pair_split(int heads, int ctas, bool heads_first, PairSplit* sp);
// Weight bytes of the most loaded CTA of a paired split.
int64_t pair_split_max_bytes(int ctas, const PairSplit& sp);
// Whether `ctas` CTAs of the paired kernel (nt = 8 or 16 tokens) can all be
// resident at once.
bool pair_kernel_fits(int ctas, int nt);
// Small-batch FMA kernel (1, 2, 4 or 8 tokens, clusters of `cluster` CTAs,
// one CTA per SM): the heads of cluster g are
// [head[g], head[g + 1]) (at most two), rank r of the cluster takes nope rows
// [r * 128 / cluster, (r + 1) * 128 / cluster) of each of them with their
// W_UK rows, and CTA i the rope rows [rope[i], rope[i + 1]).
struct SmallSplit {
  int cluster;
  uint16_t head[kMaxCtas / 2 + 1];
  uint16_t rope[kMaxCtas + 1];
};
// Fills `sp` for `ctas` CTAs (a multiple of `cluster`, 2, 4 or 8); false if
// some cluster would get more than two heads.
bool make_small_split(int heads, int ctas, int cluster, SmallSplit* sp);
// Weight bytes of the most loaded CTA of a split.
int64_t small_split_max_bytes(int heads, int ctas, const SmallSplit& sp);
// Chooses the cluster size (fewest bytes on the most loaded CTA) and fills
// `sp`; returns the grid, or 0 if no cluster size can serve `heads`.  A grid
// has at most num_sms / C clusters of C, and at most max_clusters[k] for
// C = 2 << k (how many can be resident at once; 0 = no limit, negative = that
// cluster size cannot run).
int choose_small_split(int heads, int num_sms, const int* max_clusters, SmallSplit* sp);
// Clusters of `cluster` CTAs of the small-batch kernel (nt tokens) that can
// be resident at once on this device (0 on error).
int small_kernel_max_clusters(int cluster, int nt);
cudaError_t prepare_small_kernels();
cudaError_t launch_small(const DecodeArgs& a, const SmallSplit& sp, int ctas, int nt,
                         cudaStream_t stream);
// Wide kernel (17-64 tokens, tcgen05, clusters of two CTAs splitting K): the
// heads of pair c are [head[c], head[c + 1]) (at most two).  The rope rows
// come in two unit shapes: a two-head unit u covers heads 2u and 2u + 1 (one
// 128-row tile; heads 0 .. 2 ndouble - 1, a missing last head's rows zero),
// a one-head unit v covers head 2 ndouble + v (a 64-row tile, computed as
// M = 64: finer, but slower to issue).  Pair c takes the two-head units
// [dbl[c], dbl[c + 1]) and the one-head units [sgl[c], sgl[c + 1]).  Mixing
// the shapes evens out pairs that one shape alone cannot: 128 heads on 76
// pairs, at most 44 boxes of 16 KiB per CTA with two-head units only, 40
// with 48 of them and 32 one-head units.
struct WideSplit {
  uint16_t head[kMaxCtas / 2 + 1];
  uint16_t dbl[kMaxCtas / 2 + 1];
  uint16_t sgl[kMaxCtas / 2 + 1];
  int ndouble;
};
int wide_tokens();
cudaError_t prepare_wide_kernel();
bool wide_kernel_fits(int ctas);
bool make_wide_split(int heads, int ctas, WideSplit* sp);
// Tiled copies of the weights for the wide kernel (bytes, and the packing).
size_t wide_qb_bytes(int heads);
size_t wide_ukt_bytes(int heads);
cudaError_t pack_wide_weights(const uint16_t* w_qb, const uint16_t* w_uk, uint8_t* qb_tiles,
                              uint8_t* ukt_tiles, int heads, int ndouble, cudaStream_t stream);
// Bounded poll of a gathered query buffer [batch][q_heads][576] (mla_gather.cu):
// returns once no element of the first wait_heads rows of every token is the
// all-ones sentinel, or sets MLA_DEVERR_TIMEOUT in *err after limit_ns.
cudaError_t launch_rows_wait(const void* rows, int batch, int q_heads, int wait_heads,
                             int elem_bytes, int64_t limit_ns, uint32_t* err, int num_sms,
                             cudaStream_t stream);
cudaError_t launch_wide(const DecodeArgs& a, const WideSplit& sp, int ctas, cudaStream_t stream);
size_t wide_xq_bytes();
cudaError_t launch_pair(const DecodeArgs& a, const PairSplit& sp, int ctas, int nt,
                        cudaStream_t stream);
cudaError_t launch_absorb(const DecodeArgs& a, const AbsSplit& sp, int nt, int ctas,
                          cudaStream_t stream);

// Scratch sizes for `heads` heads at the largest batch.
size_t scratch_qn_elems(int heads);
size_t scratch_ready_elems(int heads);

// Launch of the fused kernel; nt = tokens per CTA (template), mma = flavour.
// Returns a cudaError_t.
cudaError_t launch_fused(const DecodeArgs& a, const CUtensorMap* uk_map, int nt, bool mma,
                         int num_sms, cudaStream_t stream);
cudaError_t prepare_fused_kernels();

// Repack W_UK [H][128][512] BF16 into H*8 contiguous 16 KiB units: unit
// (h, cb) holds columns 64*cb..64*cb+63 as 128 rows of 128 B, the 16-byte
// chunk j of row p stored at chunk position j ^ (p % 8) (the layout a 2-D
// tensor copy with 128-byte swizzle produces).  dst: H * 131072 bytes.
cudaError_t repack_w_uk(const uint16_t* w_uk, uint8_t* dst, int heads, cudaStream_t stream);

int tokens_per_cta(int batch, bool mma);

}  // namespace mla
