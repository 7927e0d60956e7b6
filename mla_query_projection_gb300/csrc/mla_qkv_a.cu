// mla_qkv_a.cu - the down-projection that produces the fused q_a | kv_c | k_pe
// row the query path reads: y[b][n] = bf16(sum_k x[b][k] * W[n][k]), BF16
// operands, FP32 accumulation (vLLM API page "ws_gemm", class WsGemm:
// y[M, N] = x[M, K] @ W[N, K]^T; page "mla.query", method kernel: the qkv row,
// q_a at columns 0..1535, kv_c at 1536..2047, k_pe at 2048..2111).
//
// Weight streaming: each CTA owns R <= 15 consecutive rows of W over the whole
// K, so the bytes per CTA are even to within one row and no partial sum
// crosses a CTA.  Each of the 8 warps takes one eighth of K; its lanes issue
// one 1-D bulk copy per row of that slice, all of them before the
// programmatic-dependent-launch wait (W is static), into a row pitch of
// 2 * K/8 + 64 bytes (conflict-free 16-byte fragment loads).  Tokens are the
// n = 8 side of mma.sync m16n8k16 (swap-AB): 8 tokens per launch, larger
// batches in 8-token slices.  Each lane's 16-byte loads of a weight row and of
// x feed two k-steps (the same permutation of k on both operands).
#include <stdlib.h>

#include "../../include/mla_query.h"
#include "mla_device.cuh"

struct mla_qkv_a {
  int device;
  int n, k;
  int rows;  // rows of W per CTA
  int ctas;
  const uint16_t* w;
  uint32_t* err;
};

namespace mla {
namespace {

constexpr int kQkvWarps = 8;
constexpr int kQkvThreads = 32 * kQkvWarps;
constexpr int kQkvMaxRows = 15;    // rows per CTA (one m16 tile, smem bound at K = 7168)
constexpr int kQkvMaxBlocks = 28;  // 32-column blocks per warp: K <= 8 * 28 * 32 = 7168
constexpr int kQkvTok = 8;         // tokens per launch: one n8 tile
constexpr long long kQkvWaitLimit = 2000000000LL;

struct QkvArgs {
  const uint16_t* w;  // [n][k]
  const uint16_t* x;  // [batch][x_stride]
  uint16_t* y;        // [batch][y_stride]
  uint32_t* err;
  int64_t x_stride, y_stride;
  int n, k, rows, batch;
  int evict_first;  // the weights are read once: mark their lines first to go
};

__host__ __device__ constexpr int qkv_pitch(int k) { return 2 * (k / kQkvWarps) + 64; }
__host__ __device__ constexpr int qkv_red_offset(int rows, int k) {
  return kQkvWarps * rows * qkv_pitch(k);
}
// weights | FP32 partials [warp][16 rows][8 tokens] | one mbarrier per warp
__host__ __device__ constexpr int qkv_smem_bytes(int rows, int k) {
  return qkv_red_offset(rows, k) + kQkvWarps * 16 * kQkvTok * 4 + kQkvWarps * 8;
}

__global__ void __launch_bounds__(kQkvThreads, 1) mla_qkv_a_kernel(QkvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int kw = a.k / kQkvWarps;  // K columns of this warp
  const int nb = kw / 32;          // 32-column blocks of this warp
  const int pitch = qkv_pitch(a.k);
  const int row0 = blockIdx.x * a.rows;
  const int rc = min(a.rows, a.n - row0);  // rows this CTA owns
  uint8_t* wsm = smem + warp * a.rows * pitch;
  float* red = reinterpret_cast<float*>(smem + qkv_red_offset(a.rows, a.k));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + qkv_red_offset(a.rows, a.k) +
                                              kQkvWarps * 16 * kQkvTok * 4) +
                  warp;

  // ---- this warp's K slice of its rows: static weights, before the wait
  if (lane == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(bar, (uint32_t)(rc * 2 * kw));
  }
  __syncwarp();
  if (lane < rc) {
    const uint16_t* src = a.w + (int64_t)(row0 + lane) * a.k + warp * kw;
    if (a.evict_first)
      bulk_g2s_hint(wsm + lane * pitch, src, (uint32_t)(2 * kw), bar, l2_policy_evict_first());
    else
      bulk_g2s(wsm + lane * pitch, src, (uint32_t)(2 * kw), bar);
  }
  pdl_launch_dependents();
  pdl_wait();

  // ---- x fragments: token g, columns 8t..8t+7 of every block of the slice
  uint4 xr[kQkvMaxBlocks];
  const uint16_t* xs = a.x + (int64_t)g * a.x_stride + warp * kw + 8 * t;
#pragma unroll
  for (int j = 0; j < kQkvMaxBlocks; ++j) {
    xr[j] = make_uint4(0, 0, 0, 0);
    if (j < nb && g < a.batch) xr[j] = *reinterpret_cast<const uint4*>(xs + 32 * j);
  }

  float acc[4][4] = {};
  if (mbar_wait_bounded(bar, 0u, kQkvWaitLimit)) {
    const uint8_t* lo = wsm + g * pitch + 16 * t;
    const uint8_t* hi = wsm + (g + 8) * pitch + 16 * t;
    const bool has_lo = g < rc, has_hi = g + 8 < rc;
#pragma unroll
    for (int j = 0; j < kQkvMaxBlocks; ++j) {
      if (j < nb) {
        uint4 al = make_uint4(0, 0, 0, 0), ah = make_uint4(0, 0, 0, 0);
        if (has_lo) al = *reinterpret_cast<const uint4*>(lo + 64 * j);
        if (has_hi) ah = *reinterpret_cast<const uint4*>(hi + 64 * j);
        mma_bf16_16816(acc[(2 * j) & 3], al.x, ah.x, al.y, ah.y, xr[j].x, xr[j].y);
        mma_bf16_16816(acc[(2 * j + 1) & 3], al.z, ah.z, al.w, ah.w, xr[j].z, xr[j].w);
      }
    }
  } else {
    atomicOr(a.err, MLA_DEVERR_TIMEOUT);
  }

  // ---- split-K: the 8 warps' partial tiles, added in warp order
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = ((acc[0][i] + acc[1][i]) + acc[2][i]) + acc[3][i];
  float* r = red + warp * 16 * kQkvTok;
  r[g * kQkvTok + 2 * t] = v[0];
  r[g * kQkvTok + 2 * t + 1] = v[1];
  r[(g + 8) * kQkvTok + 2 * t] = v[2];
  r[(g + 8) * kQkvTok + 2 * t + 1] = v[3];
  __syncthreads();
  if (tid < 16 * kQkvTok) {
    const int row = tid / kQkvTok, tok = tid % kQkvTok;
    if (row < rc && tok < a.batch) {
      float s = red[row * kQkvTok + tok];
#pragma unroll
      for (int w = 1; w < kQkvWarps; ++w) s += red[(w * 16 + row) * kQkvTok + tok];
      a.y[(int64_t)tok * a.y_stride + row0 + row] = f2bf_bits(s);
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

extern "C" {

int mla_qkv_a_create(mla_qkv_a_t* out, int n, int k, const void* w) {
  using namespace mla;
  if (out == nullptr) return MLA_EINVAL;
  *out = nullptr;
  if (w == nullptr || !aligned16(w) || n < 1 || k < 512 || k % 512 != 0) return MLA_EINVAL;
  if (k > kQkvWarps * kQkvMaxBlocks * 32) return MLA_EUNSUPPORTED;
  int dev = 0, sms = 0, smem_max = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  const int rows = (n + sms - 1) / sms;
  if (rows > kQkvMaxRows || qkv_smem_bytes(rows, k) > smem_max) return MLA_EUNSUPPORTED;
  if (cudaFuncSetAttribute(mla_qkv_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           qkv_smem_bytes(kQkvMaxRows, kQkvWarps * kQkvMaxBlocks * 32) <= smem_max
                               ? qkv_smem_bytes(kQkvMaxRows, kQkvWarps * kQkvMaxBlocks * 32)
                               : smem_max) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ECUDA;
  }
  mla_qkv_a* h = static_cast<mla_qkv_a*>(calloc(1, sizeof(mla_qkv_a)));
  if (h == nullptr) return MLA_ENOMEM;
  h->device = dev;
  h->n = n;
  h->k = k;
  h->rows = rows;
  h->ctas = (n + rows - 1) / rows;
  h->w = static_cast<const uint16_t*>(w);
  if (cudaMalloc(&h->err, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    free(h);
    return MLA_ENOMEM;
  }
  if (cudaMemset(h->err, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->err);
    free(h);
    return MLA_ECUDA;
  }
  *out = h;
  return MLA_OK;
}

int mla_qkv_a_run(mla_qkv_a_t h, int batch, const void* x, int64_t x_stride, void* y,
                  int64_t y_stride, void* stream) {
  using namespace mla;
  if (h == nullptr || x == nullptr || y == nullptr) return MLA_EINVAL;
  if (batch < 1 || batch > MLA_MAX_BATCH) return MLA_EINVAL;
  if (x_stride == 0) x_stride = h->k;
  if (y_stride == 0) y_stride = h->n;
  if (x_stride < h->k || x_stride % 8 != 0 || !aligned16(x)) return MLA_EINVAL;
  if (y_stride < h->n || (reinterpret_cast<uintptr_t>(y) & 1u) != 0) return MLA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  QkvArgs a = {};
  a.w = h->w;
  a.err = h->err;
  a.x_stride = x_stride;
  a.y_stride = y_stride;
  a.n = h->n;
  a.k = h->k;
  a.rows = h->rows;
  a.evict_first = batch <= kQkvTok;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)h->ctas, 1, 1);
  cfg.blockDim = dim3(kQkvThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)qkv_smem_bytes(h->rows, h->k);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int t0 = 0; t0 < batch; t0 += kQkvTok) {
    a.x = static_cast<const uint16_t*>(x) + (int64_t)t0 * x_stride;
    a.y = static_cast<uint16_t*>(y) + (int64_t)t0 * y_stride;
    a.batch = batch - t0 < kQkvTok ? batch - t0 : kQkvTok;
    if (cudaLaunchKernelEx(&cfg, mla_qkv_a_kernel, a) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ECUDA;
    }
  }
  return MLA_OK;
}

int mla_qkv_a_get_error(mla_qkv_a_t h, unsigned* device_flags, void* stream) {
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

void mla_qkv_a_destroy(mla_qkv_a_t h) {
  if (h == nullptr) return;
  if (h->err) cudaFree(h->err);
  free(h);
}

}  // extern "C"
