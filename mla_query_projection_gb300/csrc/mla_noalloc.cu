// mla_noalloc.cu - mla_query_decode_noalloc: the decode step for callers that
// are not allowed to allocate device memory.
//
// The fused decode kernel needs a little global scratch (the BF16 nope q
// values handed from the CTAs that compute them to the CTAs that absorb them,
// per-head completion counters, a CTA counter and an error word).  The
// handle-based entry point allocates that scratch in mla_query_create.  This
// entry point instead uses one file-scope device array, sized for at most
// MLA_NOALLOC_MAX_BATCH tokens and MLA_MAX_HEADS heads, that every GPU which
// loads the library holds until the process exits.  It calls no cudaMalloc,
// cudaFree or other allocating routine.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/mla_query.h"
#include "mla_internal.h"

namespace {

// Layout of the array: [0, 256) error word (unused when the caller passes
// its own flag word) and CTA counter; [256, 256 + kReadyBytes) per-head
// counters; then the q hand-off buffer [tokens][heads][128] BF16.
constexpr size_t kHeaderBytes = 256;
constexpr size_t kMaxGroups = MLA_NOALLOC_MAX_BATCH / 16;  // 16 tokens per CTA above 8
constexpr size_t kReadyBytes = kMaxGroups * MLA_MAX_HEADS * sizeof(uint32_t);
constexpr size_t kQnBytes = (size_t)MLA_NOALLOC_MAX_BATCH * MLA_MAX_HEADS * 128 * sizeof(uint16_t);
constexpr size_t kScratchBytes = kHeaderBytes + kReadyBytes + kQnBytes;  // 2,099,456 B

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Per-device set-up, done by the first call on each device (with that device
// current): the device address of the array and the kernels' shared-memory
// opt-in.  In host code g_noalloc_scratch is only a stand-in symbol; the
// kernel must be given the address cudaGetSymbolAddress returns.  The address
// is kept for the life of the process, so the entry point must not be used
// on a device after cudaDeviceReset (the module, and the array with it, would
// be loaded again at another address).
constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  unsigned char* scratch = nullptr;
  int num_sms = 0;
};
DeviceState g_devices[kMaxDevices];
std::mutex g_setup_mutex;

int setup_device(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return MLA_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceState& d = g_devices[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ECUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        mla::prepare_fused_kernels() != cudaSuccess) {
      cudaGetLastError();
      return MLA_ECUDA;
    }
    d.scratch = static_cast<unsigned char*>(p);
    d.num_sms = sms;
    d.ready = true;
  }
  *out = &d;
  return MLA_OK;
}

int encode_uk_map_noalloc(CUtensorMap* map, const void* w_uk, int heads) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return MLA_ECUDA;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  cuuint64_t dims[2] = {(cuuint64_t)mla::kKvLora, (cuuint64_t)heads * mla::kNope};
  cuuint64_t strides[1] = {(cuuint64_t)mla::kKvLora * 2};
  cuuint32_t box[2] = {(cuuint32_t)mla::kUkCols, (cuuint32_t)mla::kNope};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_uk), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" MLA_API int mla_query_decode_noalloc(
    int num_heads, const void* w_qb, const void* w_uk, const void* gamma_q, const void* gamma_kv,
    float eps, int batch, const void* q_a, int64_t q_a_stride, const void* kv_c,
    int64_t kv_c_stride, const void* k_pe, int64_t k_pe_stride, const int64_t* slot_mapping,
    void* kv_cache, int64_t num_pages, int page_size, int layout, const float* k_scale,
    void* q_latent, void* q_pe, void* q_c, unsigned* device_flags, void* stream) {
  if (num_heads < 1 || num_heads > MLA_MAX_HEADS) return MLA_EINVAL;
  if (batch < 1) return MLA_EINVAL;
  if (batch > MLA_NOALLOC_MAX_BATCH) return MLA_EUNSUPPORTED;  // beyond the fixed array
  if (w_qb == nullptr || w_uk == nullptr || gamma_q == nullptr || gamma_kv == nullptr ||
      q_a == nullptr || kv_c == nullptr || k_pe == nullptr || slot_mapping == nullptr ||
      kv_cache == nullptr || q_latent == nullptr || q_pe == nullptr)
    return MLA_EINVAL;
  if (!(eps >= 0.0f)) return MLA_EINVAL;
  if (layout != MLA_KV_FP8_E4M3 && layout != MLA_KV_FP8_DS_MLA && layout != MLA_KV_NVFP4_DS_MLA)
    return MLA_EINVAL;
  if (layout == MLA_KV_FP8_E4M3 && k_scale == nullptr) return MLA_EINVAL;
  if (num_pages < 1 || page_size < 1) return MLA_EINVAL;
  if (q_a_stride == 0) q_a_stride = mla::kQLora;
  if (kv_c_stride == 0) kv_c_stride = mla::kKvLora;
  if (k_pe_stride == 0) k_pe_stride = mla::kRope;
  if (q_a_stride < mla::kQLora || kv_c_stride < mla::kKvLora || k_pe_stride < mla::kRope ||
      ((q_a_stride | kv_c_stride | k_pe_stride) & 7))
    return MLA_EINVAL;
  if (!aligned16(w_qb) || !aligned16(w_uk) || !aligned16(gamma_q) || !aligned16(gamma_kv) ||
      !aligned16(q_a) || !aligned16(kv_c) || !aligned16(k_pe) || !aligned16(kv_cache) ||
      !aligned16(q_latent) || !aligned16(q_pe) || !aligned16(q_c) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(device_flags) & 3u))
    return MLA_EINVAL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  DeviceState* d = nullptr;
  int rc = setup_device(dev, &d);
  if (rc != MLA_OK) return rc;

  const bool mma = batch > 2;
  const int nt = mla::tokens_per_cta(batch, mma);
  const int groups = (batch + nt - 1) / nt;
  // The kernel writes the q hand-off rows of every token slot of every group
  // (padding slots past the batch included) and one counter per group and
  // head: both must fit the array as sized above.
  if (groups > (int)kMaxGroups || (int64_t)groups * nt > MLA_NOALLOC_MAX_BATCH)
    return MLA_EUNSUPPORTED;

  CUtensorMap uk_map;
  if ((rc = encode_uk_map_noalloc(&uk_map, w_uk, num_heads)) != MLA_OK) return rc;

  unsigned char* base = d->scratch;
  mla::DecodeArgs a;
  a.w_qb = static_cast<const uint16_t*>(w_qb);
  a.w_uk_packed = nullptr;  // W_UK is read in place through the tensor map
  a.w_uk = static_cast<const uint16_t*>(w_uk);
  a.partial = nullptr;
  a.gamma_q = static_cast<const uint16_t*>(gamma_q);
  a.gamma_kv = static_cast<const uint16_t*>(gamma_kv);
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
  a.ql_ts = (int64_t)num_heads * mla::kKvLora;
  a.ql_hs = mla::kKvLora;
  a.qp_ts = (int64_t)num_heads * mla::kRope;
  a.qp_hs = mla::kRope;
  a.q_c = static_cast<uint16_t*>(q_c);
  a.err = device_flags != nullptr ? reinterpret_cast<uint32_t*>(device_flags)
                                  : reinterpret_cast<uint32_t*>(base);
  a.finished = reinterpret_cast<uint32_t*>(base + 4);
  a.ready = reinterpret_cast<uint32_t*>(base + kHeaderBytes);
  a.qn = reinterpret_cast<uint16_t*>(base + kHeaderBytes + kReadyBytes);
  a.heads = num_heads;
  a.batch = batch;
  a.groups = groups;
  a.eps = eps;
  a.trace = nullptr;
  a.q_scale_inv = nullptr;
  a.wide_xq = nullptr;
  a.wide_qb = nullptr;
  a.wide_ukt = nullptr;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the error word and the
  // counters must start at zero (the q buffer is fully rewritten before it is
  // read).
  if (cudaMemsetAsync(base, 0, kHeaderBytes + kReadyBytes, s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  if (mla::launch_fused(a, &uk_map, nt, mma, d->num_sms, s) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  return MLA_OK;
}
