// mla_gather.cu - the wait side of the gathered query rows (vLLM API page
// "mla.query", class MlaQuery, methods publish and gathered: under decode
// context parallelism every rank's query rows land in head block `rank` of a
// [B][q_heads][576] buffer armed with a sentinel, and readers poll until no
// word is the sentinel).  On one GPU the ranks are the decode calls that wrote
// their head blocks earlier on the stream; the poll is the same bounded check:
// every element of the buffer differs from the all-ones sentinel (an E4M3 or
// BF16 NaN pattern, which the decode never writes).  A wait that runs past
// its limit sets MLA_DEVERR_TIMEOUT and returns.
#include "../../include/mla_query.h"
#include "mla_internal.h"

namespace mla {
namespace {

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint4 ld_volatile_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// True if any byte (elem_bytes 1) or any 16-bit element (elem_bytes 2) of the
// chunk is all ones.
__device__ __forceinline__ bool has_sentinel(uint4 v, int elem_bytes) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t any = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    any |= elem_bytes == 1 ? __vcmpeq4(w[i], 0xFFFFFFFFu) : __vcmpeq2(w[i], 0xFFFFFFFFu);
  return any != 0;
}

// Chunk c of the polled region: token c / per_token, chunk c % per_token of
// that token's first heads; a token's rows start every `pitch` chunks.
__global__ void __launch_bounds__(256) mla_rows_wait_kernel(const uint4* rows, int64_t chunks,
                                                            int64_t per_token, int64_t pitch,
                                                            int elem_bytes, int64_t limit_ns,
                                                            uint32_t* err) {
  const uint64_t t0 = global_ns();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += stride) {
    const uint4* p = rows + (c / per_token) * pitch + c % per_token;
    while (has_sentinel(ld_volatile_v4(p), elem_bytes)) {
      if ((int64_t)(global_ns() - t0) > limit_ns) {
        atomicOr(err, MLA_DEVERR_TIMEOUT);
        return;
      }
      __nanosleep(256);
    }
  }
}

}  // namespace

cudaError_t launch_rows_wait(const void* rows, int batch, int q_heads, int wait_heads,
                             int elem_bytes, int64_t limit_ns, uint32_t* err, int num_sms,
                             cudaStream_t stream) {
  const int64_t row_chunks = (int64_t)kRowElems * elem_bytes / 16;
  const int64_t per_token = wait_heads * row_chunks;
  const int64_t chunks = (int64_t)batch * per_token;
  const int64_t want = (chunks + 255) / 256;
  const int ctas = (int)(want < 2 * num_sms ? want : 2 * num_sms);
  mla_rows_wait_kernel<<<ctas, 256, 0, stream>>>(static_cast<const uint4*>(rows), chunks,
                                                 per_token, q_heads * row_chunks, elem_bytes,
                                                 limit_ns, err);
  return cudaGetLastError();
}

}  // namespace mla
