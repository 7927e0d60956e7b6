// mla_api.cu - the C ABI (include/mla_query.h): argument checks, the handle
// with its device scratch, the W_UK tensor map, and path dispatch.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/mla_query.h"
#include "mla_internal.h"

struct mla_query {
  int device;
  int heads;
  int num_sms;
  int path;  // MLA_PATH_*
  const uint16_t* w_qb;
  const uint16_t* w_uk;
  const uint16_t* gamma_q;
  const uint16_t* gamma_kv;
  float eps;
  CUtensorMap uk_map;
  void* scratch;  // one cudaMalloc: err | finished | ready[] | qn[]
  uint32_t* err;
  uint32_t* finished;
  uint32_t* ready;
  uint16_t* qn;
  uint64_t* trace;  // MLA_TRACE builds: per-CTA timeline stamps
  uint8_t* w_uk_packed;  // library-owned repacked copy of W_UK
  float* partial;        // absorbing kernel: FP32 partial absorptions
  mla::AbsSplit split;   // absorbing kernel: per-CTA ranges
  mla::PairSplit pair_split;    // paired absorbing kernel, up to 8 tokens: heads first
  mla::PairSplit pair_split16;  // its 16-token flavour: heads spread evenly
  int pair_ctas;              // its grid (even), 0 if it cannot run on this device
  bool pair16;                // its 16-token flavour can run too
  bool pair_balanced;         // no CTA of it holds more than 10% above the mean bytes
  bool fma_first;             // one token takes the FMA kernel (pick_kernel)
  uint8_t* wide_qb;           // wide kernel: library-owned W_QB tiles
  uint8_t* wide_ukt;          // wide kernel: library-owned W_UK^T tiles
  uint8_t* wide_xq;           // wide kernel: normalised xq in tile layout
  mla::WideSplit wide_split;  // per-pair heads and rope units
  int wide_ctas;              // its grid (even), 0 if it cannot run on this device
  mla::SmallSplit small_split;  // small-batch FMA kernel: cluster size, heads, rope rows
  int small_ctas;               // its grid, 0 if it cannot run on this device
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// W_UK [H*128 rows][512 columns] BF16, boxes of 128 rows x 64 columns (128 B
// rows, 128 B swizzle).
int encode_uk_map(CUtensorMap* map, const void* w_uk, int heads) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return MLA_ECUDA;
  cuuint64_t dims[2] = {(cuuint64_t)mla::kKvLora, (cuuint64_t)heads * mla::kNope};
  cuuint64_t strides[1] = {(cuuint64_t)mla::kKvLora * 2};
  cuuint32_t box[2] = {(cuuint32_t)mla::kUkCols, (cuuint32_t)mla::kNope};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_uk), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ECUDA;
}

// The kernel a decode call launches:
//   absorbing kernel, FP32 FMA flavour (1 or 2 tokens per CTA);
//   absorbing kernel, tensor-core flavour (8 or 16 tokens per CTA, B <= 16);
//   hand-off kernel, tensor cores, token groups of 8 or 16 (any B).
enum class Kernel { kSmall, kAbsorbMma, kAbsorbPair, kWide, kHandoff };

// The default path (measured on GB300, us per step, FMA kernel against the
// tensor-core kernel the batch would otherwise take):
//  * one token where the FMA kernel's most loaded CTA carries at most 80% of
//    the paired kernel's bytes (up to 36 heads on GB300: clusters of 4 or
//    8 CTAs split a head four or eight ways, the paired kernel two ways):
//    FP32 FMAs, 8 heads 4.00 against 4.83, 16 heads 4.73 / 5.43, 32 heads
//    5.72 / 6.85, 36 heads 5.72 / 6.78;
//  * everything else: tensor cores.  One token where both put the same
//    bytes on their most loaded CTA: 40 heads 7.26 against 6.82, 48 heads
//    7.29 / 6.98, 64 heads 8.51 / 7.85, 80 heads 13.32 / 12.98, 88 heads
//    13.04 / 12.90, 96 heads 12.93 / 12.98, 104 heads 12.66 / 12.88, 128
//    heads 14.59 / 14.40; 2, 4 and 8 tokens: 16 heads 6.32 / 6.11, 8.72 /
//    6.94, 13.73 / 7.02, and at 64 and 128 heads the FMA kernel is 1.4 to
//    3.6 times slower.
// Both stream every weight byte once; after the programmatic-dependent-launch
// wait a step is bound by its consumers: the FMA kernel's clusters close each
// head through distributed shared memory, where the partials kernel makes an
// L2 round trip, but its per-row FMA work is slower than the paired kernel's
// tensor-core tiles.
//
// Among the tensor-core kernels up to 16 tokens: the paired kernel, even
// where whole half-heads leave its CTAs unbalanced (its time hardly grows
// with the tokens: 80 heads, 8 tokens 13.0 against 20.9 us for the partials
// kernel; 96 heads 13.0 / 24.6; 48 heads 7.4 / 12.4; 16 heads and 16 tokens
// 9.9 / 12.2), except at few heads and tokens, where the partials kernel's
// even split wins (8 heads, 2 tokens 5.0 against 7.3; 16 heads, 4 tokens
// 6.9 / 7.3; 32 heads, 2 tokens 8.0 / 7.3 goes to the paired kernel).
bool partials_first(const mla_query* h, int batch) {
  return !h->pair_balanced && h->heads <= 24 && h->heads * batch <= 64;
}

int pick_kernel(const mla_query* h, int batch, Kernel* k, int* nt) {
  int path = h->path;
  if (path == MLA_PATH_AUTO)
    path = batch == 1 && h->fma_first ? MLA_PATH_FMA : MLA_PATH_MMA;
  if (path == MLA_PATH_FMA) {
    if (batch > 8 || h->small_ctas == 0) return MLA_EUNSUPPORTED;
    *k = Kernel::kSmall;
    *nt = batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8;
  } else if (path == MLA_PATH_MMA) {
    if (batch <= 16 && partials_first(h, batch)) {
      *k = Kernel::kAbsorbMma;
      *nt = batch <= 8 ? 8 : 16;
    } else if (batch <= 8 && h->pair_ctas > 0) {
      *k = Kernel::kAbsorbPair;
      *nt = 8;
    } else if (batch <= 16 && h->pair_ctas > 0 && h->pair16) {
      *k = Kernel::kAbsorbPair;
      *nt = 16;
    } else if (batch > 16 && h->wide_ctas > 0) {
      *k = Kernel::kWide;  // one launch per 64 tokens
      *nt = mla::wide_tokens();
    } else if (h->pair_ctas > 0 && h->pair16) {
      *k = Kernel::kAbsorbPair;  // above 16 tokens: one launch per 16 tokens
      *nt = 16;
    } else if (batch <= 16) {
      *k = Kernel::kAbsorbMma;
      *nt = batch <= 8 ? 8 : 16;
    } else {
      *k = Kernel::kHandoff;
      *nt = mla::tokens_per_cta(batch, true);
    }
  } else {
    return MLA_EINVAL;
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

const char* mla_query_strerror(int code) {
  switch (code) {
    case MLA_OK: return "ok";
    case MLA_EINVAL: return "invalid argument";
    case MLA_ENOMEM: return "device allocation failed";
    case MLA_ECUDA: return "CUDA call failed";
    case MLA_EUNSUPPORTED: return "unsupported shape or path";
    default: return "unknown error";
  }
}

int mla_query_create(mla_query_t* out, int num_heads, const void* w_qb, const void* w_uk,
                     const void* gamma_q, const void* gamma_kv, float eps) {
  if (out == nullptr) return MLA_EINVAL;
  *out = nullptr;
  if (num_heads < 1 || num_heads > MLA_MAX_HEADS) return MLA_EINVAL;
  if (w_qb == nullptr || w_uk == nullptr || gamma_q == nullptr || gamma_kv == nullptr)
    return MLA_EINVAL;
  if (!aligned16(w_qb) || !aligned16(w_uk) || !aligned16(gamma_q) || !aligned16(gamma_kv))
    return MLA_EINVAL;
  if (!(eps >= 0.0f)) return MLA_EINVAL;

  mla_query* h = static_cast<mla_query*>(calloc(1, sizeof(mla_query)));
  if (h == nullptr) return MLA_ENOMEM;
  h->heads = num_heads;
  h->w_qb = static_cast<const uint16_t*>(w_qb);
  h->w_uk = static_cast<const uint16_t*>(w_uk);
  h->gamma_q = static_cast<const uint16_t*>(gamma_q);
  h->gamma_kv = static_cast<const uint16_t*>(gamma_kv);
  h->eps = eps;
  h->path = MLA_PATH_AUTO;
  int rc = MLA_ECUDA;
  if (cudaGetDevice(&h->device) != cudaSuccess) goto fail;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
      cudaSuccess)
    goto fail;
  if (mla::prepare_fused_kernels() != cudaSuccess || mla::prepare_small_kernels() != cudaSuccess)
    goto fail;
  if ((rc = encode_uk_map(&h->uk_map, w_uk, num_heads)) != MLA_OK) goto fail;
  if (h->num_sms > mla::kMaxCtas) {
    rc = MLA_EUNSUPPORTED;
    goto fail;
  }
  mla::make_abs_split(num_heads, h->num_sms, &h->split);
  // The small-batch FMA kernel: the cluster size whose split puts the fewest
  // bytes on the most loaded CTA.  Each grid is sized so that all its
  // clusters can be resident at once, one CTA per SM, for every token count
  // (1, 2, 4, 8) the kernel is built for.
  {
    int most[3];
    for (int k = 0; k < 3; ++k) {
      const int c = 2 << k;
      most[k] = mla::small_kernel_max_clusters(c, 1);
      for (int nt = 2; nt <= 8; nt *= 2) {
        const int m = mla::small_kernel_max_clusters(c, nt);
        if (m < most[k]) most[k] = m;
      }
      if (most[k] <= 0) most[k] = -1;  // cannot run: no cluster of this size
    }
    h->small_ctas = 0;
    mla::SmallSplit trial;
    trial.cluster = 0;
    const int ctas = mla::choose_small_split(num_heads, h->num_sms, most, &trial);
    if (ctas > 0) {
      h->small_split = trial;
      h->small_ctas = ctas;
    }
#ifdef MLA_DEBUG_SPLIT
    fprintf(stderr, "small split: heads %d sms %d max clusters %d %d %d -> ctas %d cluster %d\n",
            num_heads, h->num_sms, most[0], most[1], most[2], h->small_ctas, trial.cluster);
#endif
  }
  // The paired kernel gives each CTA whole half-heads (256 KiB of weights per
  // head). Balanced means no CTA holds more than 10% above the average bytes
  // per CTA; where it is not, one token takes the FMA kernel and few heads
  // and tokens the partials kernel (pick_kernel).
  h->pair_ctas = h->num_sms & ~1;
  {
    const int pairs = h->pair_ctas / 2;
    // Where the heads do not fill every pair, one head on each of the first
    // pairs measured faster than heads spread evenly for launches of up to 8
    // tokens (at 64 heads on 76 pairs, one token: 7.85 against 7.92 us; 40
    // heads, two tokens: 6.80 against 7.32), and slower for 16 tokens (11.25
    // against 11.04 us at 64 heads); each flavour takes the faster order.
    if (pairs < 1 || !mla::make_pair_split(num_heads, h->pair_ctas, true, &h->pair_split) ||
        !mla::make_pair_split(num_heads, h->pair_ctas, false, &h->pair_split16) ||
        !mla::pair_kernel_fits(h->pair_ctas, 8))
      h->pair_ctas = 0;
    h->pair16 = h->pair_ctas > 0 && mla::pair_kernel_fits(h->pair_ctas, 16);
    const int64_t most = (int64_t)((num_heads + pairs - 1) / (pairs > 0 ? pairs : 1)) * 4 * 65536;
    const int64_t avg = (int64_t)num_heads * (8 * 65536 + 64 * 3072) / (h->pair_ctas > 0 ? h->pair_ctas : 1);
    h->pair_balanced = h->pair_ctas > 0 && 10 * most <= 11 * avg;
  }
  // One token takes the FMA kernel where its most loaded CTA carries at most
  // 80% of the paired kernel's (clusters of 4 or 8 CTAs split a head four or
  // eight ways where the paired kernel splits it two ways), or where the
  // paired kernel cannot run.
  h->fma_first =
      h->small_ctas > 0 &&
      (h->pair_ctas == 0 ||
       5 * mla::small_split_max_bytes(num_heads, h->small_ctas, h->small_split) <=
           4 * mla::pair_split_max_bytes(h->pair_ctas, h->pair_split));
  // Wide kernel (17 tokens and more): its split decides the rope tiles' shape.
  if (mla::prepare_wide_kernel() != cudaSuccess) goto fail;
  h->wide_ctas = h->num_sms & ~1;
  if (!mla::make_wide_split(num_heads, h->wide_ctas, &h->wide_split) ||
      !mla::wide_kernel_fits(h->wide_ctas))
    h->wide_ctas = 0;
  {
    // Device memory for the kernels the dispatch can reach with this head
    // count on this device, and nothing else: the partials kernel where the
    // paired kernel cannot serve every batch of up to 16 tokens or leaves it
    // to the partials kernel (few heads and tokens), the wide kernel's tiled
    // weight copies where it runs, and the hand-off kernel's packed W_UK and
    // q buffer only where neither the wide nor the 16-token paired kernel
    // covers batches above 16.
    const bool partials = h->pair_ctas == 0 || !h->pair16 || partials_first(h, 1);
    const bool handoff = h->wide_ctas == 0 && !(h->pair_ctas > 0 && h->pair16);
    const bool wide = h->wide_ctas > 0;
    const size_t head = 256;  // err, finished
    const size_t ready_bytes = mla::scratch_ready_elems(num_heads) * sizeof(uint32_t);
    const size_t qn_off = head + ((ready_bytes + 255) / 256) * 256;
    const size_t bytes =
        qn_off + (handoff ? mla::scratch_qn_elems(num_heads) * sizeof(uint16_t) : 0);
    if (cudaMalloc(&h->scratch, bytes) != cudaSuccess) {
      rc = MLA_ENOMEM;
      goto fail;
    }
    if (cudaMemset(h->scratch, 0, bytes) != cudaSuccess) goto fail;
    uint8_t* base = static_cast<uint8_t*>(h->scratch);
    h->err = reinterpret_cast<uint32_t*>(base);
    h->finished = reinterpret_cast<uint32_t*>(base + 4);
    h->ready = reinterpret_cast<uint32_t*>(base + head);
    h->qn = handoff ? reinterpret_cast<uint16_t*>(base + qn_off) : nullptr;
    // FP32 partial absorptions of the partials kernel: [task][token < 16][512]
    if (partials &&
        cudaMalloc(&h->partial, (size_t)num_heads * 8 * 16 * mla::kKvLora * sizeof(float)) !=
            cudaSuccess) {
      rc = MLA_ENOMEM;
      goto fail;
    }
    // W_UK copy in contiguous pre-swizzled units (one 1-D bulk copy per unit)
    if (handoff) {
      if (cudaMalloc(&h->w_uk_packed,
                     (size_t)num_heads * mla::kUkUnitsPerHead * mla::kUkUnitBytes) != cudaSuccess) {
        rc = MLA_ENOMEM;
        goto fail;
      }
      if (mla::repack_w_uk(h->w_uk, h->w_uk_packed, num_heads, 0) != cudaSuccess ||
          cudaStreamSynchronize(0) != cudaSuccess)
        goto fail;
    }
    if (wide) {
      if (cudaMalloc(&h->wide_xq, mla::wide_xq_bytes()) != cudaSuccess ||
          cudaMalloc(&h->wide_qb, mla::wide_qb_bytes(num_heads)) != cudaSuccess ||
          cudaMalloc(&h->wide_ukt, mla::wide_ukt_bytes(num_heads)) != cudaSuccess) {
        rc = MLA_ENOMEM;
        goto fail;
      }
      if (mla::pack_wide_weights(h->w_qb, h->w_uk, h->wide_qb, h->wide_ukt, num_heads,
                                 h->wide_split.ndouble, 0) != cudaSuccess ||
          cudaStreamSynchronize(0) != cudaSuccess)
        goto fail;
    }
  }
#ifdef MLA_TRACE
  {
    const size_t tb = (size_t)h->num_sms * mla::kTraceSlots * 8;
    if (cudaMalloc(&h->trace, tb) != cudaSuccess || cudaMemset(h->trace, 0, tb) != cudaSuccess)
      goto fail;
  }
#endif
  *out = h;
  return MLA_OK;
fail:
  if (h->scratch) cudaFree(h->scratch);
  if (h->partial) cudaFree(h->partial);
  if (h->w_uk_packed) cudaFree(h->w_uk_packed);
  if (h->wide_qb) cudaFree(h->wide_qb);
  if (h->wide_ukt) cudaFree(h->wide_ukt);
  if (h->wide_xq) cudaFree(h->wide_xq);
  if (h->trace) cudaFree(h->trace);
  free(h);
  cudaGetLastError();
  return rc;
}

}  // extern "C"

namespace {

// The decode step behind both entry points: BF16 query outputs, or
// (q_scale_inv != nullptr) per-tensor FP8 ones.
// Addressing of the q outputs, in output elements: token and head strides of
// q_latent and of q_pe (see DecodeArgs).  All zero: contiguous [B][H][512] and
// [B][H][64].
struct QStrides {
  int64_t ql_ts, ql_hs, qp_ts, qp_hs;
};

int decode_impl(mla_query_t h, int batch, const void* q_a, int64_t q_a_stride, const void* kv_c,
                int64_t kv_c_stride, const void* k_pe, int64_t k_pe_stride,
                const int64_t* slot_mapping, void* kv_cache, int64_t num_pages, int page_size,
                int layout, const float* k_scale, const float* q_scale_inv, void* q_latent,
                void* q_pe, void* q_c, void* stream, QStrides qs = {0, 0, 0, 0}) {
  if (h == nullptr) return MLA_EINVAL;
  if (batch < 1 || batch > MLA_MAX_BATCH) return MLA_EINVAL;
  if (q_a == nullptr || kv_c == nullptr || k_pe == nullptr || slot_mapping == nullptr ||
      kv_cache == nullptr || q_latent == nullptr || q_pe == nullptr)
    return MLA_EINVAL;
  if (layout != MLA_KV_FP8_E4M3 && layout != MLA_KV_FP8_DS_MLA && layout != MLA_KV_NVFP4_DS_MLA)
    return MLA_EINVAL;
  if (layout == MLA_KV_FP8_E4M3 && k_scale == nullptr) return MLA_EINVAL;
  if (num_pages < 1 || page_size < 1) return MLA_EINVAL;
  if (q_a_stride == 0) q_a_stride = mla::kQLora;
  if (kv_c_stride == 0) kv_c_stride = mla::kKvLora;
  if (k_pe_stride == 0) k_pe_stride = mla::kRope;
  if (q_a_stride < mla::kQLora || kv_c_stride < mla::kKvLora || k_pe_stride < mla::kRope)
    return MLA_EINVAL;
  if ((q_a_stride | kv_c_stride | k_pe_stride) & 7) return MLA_EINVAL;
  if (!aligned16(q_a) || !aligned16(kv_c) || !aligned16(k_pe) || !aligned16(kv_cache) ||
      !aligned16(q_latent) || !aligned16(q_pe) || !aligned16(q_c) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(q_scale_inv) & 3u))
    return MLA_EINVAL;

  Kernel kern = Kernel::kSmall;
  int nt = 1;
  int rc = pick_kernel(h, batch, &kern, &nt);
  if (rc != MLA_OK) return rc;
  const bool contiguous = qs.ql_ts == 0;
  if ((q_scale_inv != nullptr || !contiguous) && kern == Kernel::kHandoff) return MLA_EUNSUPPORTED;
  if (contiguous)
    qs = {(int64_t)h->heads * mla::kKvLora, mla::kKvLora, (int64_t)h->heads * mla::kRope,
          mla::kRope};

  mla::DecodeArgs a;
  a.w_qb = h->w_qb;
  a.w_uk_packed = h->w_uk_packed;
  a.w_uk = h->w_uk;
  a.partial = h->partial;
  a.gamma_q = h->gamma_q;
  a.gamma_kv = h->gamma_kv;
  a.q_a = static_cast<const uint16_t*>(q_a);
  a.kv_c = static_cast<const uint16_t*>(kv_c);
  a.k_pe = static_cast<const uint16_t*>(k_pe);
  a.q_a_stride = q_a_stride;
  a.kv_c_stride = kv_c_stride;
  a.k_pe_stride = k_pe_stride;
  a.slots = slot_mapping;
  a.cache = static_cast<uint8_t*>(kv_cache);
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.layout = layout;
  a.k_scale = k_scale;
  a.q_latent = static_cast<uint16_t*>(q_latent);
  a.q_pe = static_cast<uint16_t*>(q_pe);
  a.ql_ts = qs.ql_ts;
  a.ql_hs = qs.ql_hs;
  a.qp_ts = qs.qp_ts;
  a.qp_hs = qs.qp_hs;
  a.q_c = static_cast<uint16_t*>(q_c);
  a.qn = h->qn;
  a.ready = h->ready;
  a.finished = h->finished;
  a.err = h->err;
  a.heads = h->heads;
  a.batch = batch;
  a.groups = (batch + nt - 1) / nt;
  a.eps = h->eps;
  a.trace = h->trace;
  a.q_scale_inv = q_scale_inv;
  a.wide_xq = h->wide_xq;
  a.wide_qb = h->wide_qb;
  a.wide_ukt = h->wide_ukt;
  if (a.groups > h->num_sms) return MLA_EUNSUPPORTED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // bytes per q_latent / q_pe element: BF16, or E4M3 with the FP8 query
  const int64_t qbytes = q_scale_inv != nullptr ? 1 : 2;
  cudaError_t e;
  if (kern == Kernel::kSmall)
    e = mla::launch_small(a, h->small_split, h->small_ctas, nt, st);
  else if (kern == Kernel::kHandoff)
    e = mla::launch_fused(a, &h->uk_map, nt, true, h->num_sms, st);
  else if (kern == Kernel::kWide) {
    // one launch per slice of 64 tokens, every per-token pointer offset
    e = cudaSuccess;
    const int tw = mla::wide_tokens();
    for (int t0 = 0; t0 < batch && e == cudaSuccess; t0 += tw) {
      mla::DecodeArgs s64 = a;
      s64.batch = batch - t0 < tw ? batch - t0 : tw;
      s64.groups = 1;
      s64.q_a = a.q_a + (int64_t)t0 * a.q_a_stride;
      s64.kv_c = a.kv_c + (int64_t)t0 * a.kv_c_stride;
      s64.k_pe = a.k_pe + (int64_t)t0 * a.k_pe_stride;
      s64.slots = a.slots + t0;
      s64.q_latent = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.q_latent) +
                                                 (int64_t)t0 * a.ql_ts * qbytes);
      s64.q_pe = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.q_pe) +
                                             (int64_t)t0 * a.qp_ts * qbytes);
      s64.q_c = a.q_c != nullptr ? a.q_c + (int64_t)t0 * mla::kQLora : nullptr;
      e = mla::launch_wide(s64, h->wide_split, h->wide_ctas, st);
    }
  } else if (kern == Kernel::kAbsorbPair && batch <= 16)
    e = mla::launch_pair(a, nt == 16 ? h->pair_split16 : h->pair_split, h->pair_ctas, nt, st);
  else if (kern == Kernel::kAbsorbPair) {
    // Batches above 16: the 16-token paired kernel once per slice of 16
    // tokens, every per-token pointer offset to the slice.  Each launch
    // streams the weights again; each slice inserts its own KV rows.
    e = cudaSuccess;
    for (int t0 = 0; t0 < batch && e == cudaSuccess; t0 += 16) {
      mla::DecodeArgs s16 = a;
      s16.batch = batch - t0 < 16 ? batch - t0 : 16;
      s16.groups = 1;
      s16.q_a = a.q_a + (int64_t)t0 * a.q_a_stride;
      s16.kv_c = a.kv_c + (int64_t)t0 * a.kv_c_stride;
      s16.k_pe = a.k_pe + (int64_t)t0 * a.k_pe_stride;
      s16.slots = a.slots + t0;
      s16.q_latent = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.q_latent) +
                                                 (int64_t)t0 * a.ql_ts * qbytes);
      s16.q_pe = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(a.q_pe) +
                                             (int64_t)t0 * a.qp_ts * qbytes);
      s16.q_c = a.q_c != nullptr ? a.q_c + (int64_t)t0 * mla::kQLora : nullptr;
      e = s16.batch <= 8 ? mla::launch_pair(s16, h->pair_split, h->pair_ctas, 8, st)
                         : mla::launch_pair(s16, h->pair_split16, h->pair_ctas, 16, st);
    }
  }
  else
    e = mla::launch_absorb(a, h->split, nt, h->num_sms, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_query_decode(mla_query_t h, int batch, const void* q_a, int64_t q_a_stride,
                     const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                     int64_t k_pe_stride, const int64_t* slot_mapping, void* kv_cache,
                     int64_t num_pages, int page_size, int layout, const float* k_scale,
                     void* q_latent, void* q_pe, void* q_c, void* stream) {
  return decode_impl(h, batch, q_a, q_a_stride, kv_c, kv_c_stride, k_pe, k_pe_stride,
                     slot_mapping, kv_cache, num_pages, page_size, layout, k_scale, nullptr,
                     q_latent, q_pe, q_c, stream);
}

int mla_query_decode_fp8q(mla_query_t h, int batch, const void* q_a, int64_t q_a_stride,
                          const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                          int64_t k_pe_stride, const int64_t* slot_mapping, void* kv_cache,
                          int64_t num_pages, int page_size, int layout, const float* k_scale,
                          const float* q_scale_inv, void* q_latent_fp8, void* q_pe_fp8,
                          void* q_c, void* stream) {
  if (q_scale_inv == nullptr) return MLA_EINVAL;
  return decode_impl(h, batch, q_a, q_a_stride, kv_c, kv_c_stride, k_pe, k_pe_stride,
                     slot_mapping, kv_cache, num_pages, page_size, layout, k_scale, q_scale_inv,
                     q_latent_fp8, q_pe_fp8, q_c, stream);
}

int mla_query_decode_rows(mla_query_t h, int batch, const void* q_a, int64_t q_a_stride,
                          const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                          int64_t k_pe_stride, const int64_t* slot_mapping, void* kv_cache,
                          int64_t num_pages, int page_size, int layout, const float* k_scale,
                          const float* q_scale_inv, void* q_rows, int q_heads, int head_offset,
                          void* q_c, void* stream) {
  if (h == nullptr || q_rows == nullptr) return MLA_EINVAL;
  if (head_offset < 0 || q_heads < 1 || q_heads > mla::kMaxRowHeads ||
      head_offset + h->heads > q_heads)
    return MLA_EINVAL;
  const int64_t e = q_scale_inv != nullptr ? 1 : 2;  // bytes per element
  uint8_t* base = static_cast<uint8_t*>(q_rows) + (int64_t)head_offset * mla::kRowElems * e;
  const int64_t ts = (int64_t)q_heads * mla::kRowElems;
  return decode_impl(h, batch, q_a, q_a_stride, kv_c, kv_c_stride, k_pe, k_pe_stride,
                     slot_mapping, kv_cache, num_pages, page_size, layout, k_scale, q_scale_inv,
                     base, base + mla::kKvLora * e, q_c, stream,
                     QStrides{ts, mla::kRowElems, ts, mla::kRowElems});
}

int mla_query_rows_arm(void* q_rows, int batch, int q_heads, int elem_bytes, void* stream) {
  if (q_rows == nullptr || batch < 1 || batch > MLA_MAX_BATCH || q_heads < 1 ||
      q_heads > mla::kMaxRowHeads || (elem_bytes != 1 && elem_bytes != 2) || !aligned16(q_rows))
    return MLA_EINVAL;
  const size_t bytes = (size_t)batch * q_heads * mla::kRowElems * elem_bytes;
  if (cudaMemsetAsync(q_rows, 0xFF, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  return MLA_OK;
}

int mla_query_rows_wait(mla_query_t h, const void* q_rows, int batch, int q_heads,
                        int wait_heads, int elem_bytes, int64_t limit_ns, void* stream) {
  if (h == nullptr || q_rows == nullptr || batch < 1 || batch > MLA_MAX_BATCH || q_heads < 1 ||
      q_heads > mla::kMaxRowHeads || wait_heads < 1 || wait_heads > q_heads ||
      (elem_bytes != 1 && elem_bytes != 2) || !aligned16(q_rows) || limit_ns < 0 ||
      limit_ns > MLA_ROWS_WAIT_MAX_NS)
    return MLA_EINVAL;
  if (mla::launch_rows_wait(q_rows, batch, q_heads, wait_heads, elem_bytes, limit_ns, h->err,
                            h->num_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  return MLA_OK;
}

int mla_query_get_error(mla_query_t h, unsigned* device_flags, void* stream) {
  if (h == nullptr || device_flags == nullptr) return MLA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, h->err, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(h->err, 0, sizeof(uint32_t), s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  *device_flags = v;
  return MLA_OK;
}

int mla_query_set_path(mla_query_t h, int path) {
  if (h == nullptr) return MLA_EINVAL;
  if (path != MLA_PATH_AUTO && path != MLA_PATH_FMA && path != MLA_PATH_MMA) return MLA_EINVAL;
  h->path = path;
  return MLA_OK;
}

int mla_query_path_for(mla_query_t h, int batch) {
  if (h == nullptr || batch < 1 || batch > MLA_MAX_BATCH) return MLA_EINVAL;
  Kernel kern = Kernel::kSmall;
  int nt = 1;
  int rc = pick_kernel(h, batch, &kern, &nt);
  if (rc != MLA_OK) return rc;
  return kern == Kernel::kSmall ? MLA_PATH_FMA : MLA_PATH_MMA;
}

const char* mla_query_kernel_for(mla_query_t h, int batch) {
  if (h == nullptr || batch < 1 || batch > MLA_MAX_BATCH) return nullptr;
  Kernel kern = Kernel::kSmall;
  int nt = 1;
  if (pick_kernel(h, batch, &kern, &nt) != MLA_OK) return nullptr;
  switch (kern) {
    case Kernel::kSmall: {
      static const char* names[4][3] = {
          {"mla_small_kernel<1,2>", "mla_small_kernel<1,4>", "mla_small_kernel<1,8>"},
          {"mla_small_kernel<2,2>", "mla_small_kernel<2,4>", "mla_small_kernel<2,8>"},
          {"mla_small_kernel<4,2>", "mla_small_kernel<4,4>", "mla_small_kernel<4,8>"},
          {"mla_small_kernel<8,2>", "mla_small_kernel<8,4>", "mla_small_kernel<8,8>"}};
      const int c = h->small_split.cluster;
      const int row = nt <= 1 ? 0 : nt == 2 ? 1 : nt == 4 ? 2 : 3;
      return names[row][c == 2 ? 0 : c == 4 ? 1 : 2];
    }
    case Kernel::kAbsorbMma: return nt == 8 ? "mla_absorb_mma_kernel<8>" : "mla_absorb_mma_kernel<16>";
    case Kernel::kAbsorbPair: return nt == 8 ? "mla_absorb_pair_kernel<8>" : "mla_absorb_pair_kernel<16>";
    case Kernel::kWide: return "mla_wide_norm_kernel+mla_wide_kernel";
    case Kernel::kHandoff: return "mla_fused_kernel";
  }
  return nullptr;
}

#ifdef MLA_TRACE
// Timeline readout of trace builds: copies the per-CTA stamps to `host` and
// clears them for the next call.
MLA_API int mla_query_trace_read(mla_query_t h, void* host, size_t bytes) {
  if (h == nullptr || h->trace == nullptr) return MLA_EINVAL;
  if (cudaMemcpy(host, h->trace, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ECUDA;
  return cudaMemset(h->trace, 0, bytes) == cudaSuccess ? MLA_OK : MLA_ECUDA;
}
#endif

void mla_query_destroy(mla_query_t h) {
  if (h == nullptr) return;
  if (h->trace) cudaFree(h->trace);
  if (h->scratch) cudaFree(h->scratch);
  if (h->w_uk_packed) cudaFree(h->w_uk_packed);
  if (h->wide_qb) cudaFree(h->wide_qb);
  if (h->wide_ukt) cudaFree(h->wide_ukt);
  if (h->wide_xq) cudaFree(h->wide_xq);
  if (h->partial) cudaFree(h->partial);
  free(h);
}

}  // extern "C"
