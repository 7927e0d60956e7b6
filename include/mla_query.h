/*
 * mla_query.h - C ABI of the GB300 (sm_103a) decode-step MLA query library.
 *
 * One call of mla_query_decode runs the query side of one Multi-head Latent
 * Attention decode step on one GPU, as the vLLM API page "mla.query" (module
 * vllm/models/kimi_k3/nvidia/specialized_decode/cutedsl/mla/query.py, class
 * MlaQuery) defines it:
 *
 *   1. q_a RMSNorm (class MlaQuery, method kernel):
 *        xq[b,k] = bf16((q_a[b,k] * rr) * gamma_q[k]),
 *        rr = 1/sqrt(sum_k q_a[b,k]^2 / 1536 + eps);          xq is also q_c.
 *   2. Q_B projection (method kernel): for every head h and p < 192,
 *        q[b,h,p] = bf16(sum_k xq[b,k] * W_QB[h*192+p, k])  (FP32 accumulate).
 *   3. rope split: q_pe[b,h,i] = q[b,h,128+i], i < 64 (no rotation here).
 *   4. W_UK absorption (method kernel):
 *        q_latent[b,h,c] = bf16(sum_{p<128} q[b,h,p] * W_UK[h,p,c]).
 *   5. KV insert (methods insert, kv_fp8, insert_ds; function pow2_ceil):
 *        n = bf16((kv_c * rr_kv) * gamma_kv), rr_kv = 1/sqrt(sum kv_c^2/512 + eps),
 *        written with k_pe into the paged FP8 cache row of slot_mapping[b].
 *
 * Conventions.  All tensors are caller-owned device memory unless stated.
 * BF16 is IEEE bfloat16 stored as 16-bit words; arrays are row-major and
 * dense unless a stride argument says otherwise.  Every pointer must be
 * 16-byte aligned.  Calls are asynchronous on the given CUDA stream
 * (a cudaStream_t passed as void*; NULL = the legacy default stream), never
 * synchronise the host and never allocate.  Host-checkable argument errors
 * return a negative code and launch nothing; errors only the device can see
 * (a slot beyond the cache) set a sticky device flag read by
 * mla_query_get_error.  No call ever traps the GPU.
 */
#ifndef MLA_QUERY_H
#define MLA_QUERY_H

#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MLA_OK 0
#define MLA_EINVAL (-1)       /* bad argument (null, size, alignment, layout) */
#define MLA_ENOMEM (-2)       /* device allocation failed in create           */
#define MLA_ECUDA (-3)        /* a CUDA runtime/driver call failed            */
#define MLA_EUNSUPPORTED (-4) /* shape the library does not handle            */

/* KV cache layouts (page "mla.query", methods insert, insert_ds and
   insert_nvfp4). */
#define MLA_KV_FP8_E4M3 0   /* 576-byte row: 512 E4M3 latent + 64 E4M3 k_pe,
                               each value divided by k_scale                 */
#define MLA_KV_FP8_DS_MLA 1 /* 656-byte row: 512 E4M3 latent scaled per 128
                               columns by a power of two, 4 FP32 scales at
                               byte 512, 64 raw BF16 k_pe at byte 528        */
#define MLA_KV_NVFP4_DS_MLA 2 /* 352-byte row: 512 E2M1 latent, two to a byte
                               (value 2k in the low half of byte k), scaled
                               per 16 values by the E4M3 scale
                               max(amax / 6, 2^-9); the 32 scales at byte
                               256, block s at 256 + 8 * (s % 4) + s / 4;
                               64 unscaled E4M3 k_pe at byte 288          */

/* Bits of the device error flag (mla_query_get_error). */
#define MLA_DEVERR_BAD_SLOT 1u /* a slot >= num_pages * page_size was skipped   */
#define MLA_DEVERR_TIMEOUT 2u  /* an internal bounded wait gave up (results of
                                  that call are not valid)                     */
#define MLA_DEVERR_CHECK 4u    /* builds compiled with -DMLA_CHECKS only: an
                                  index or address failed its bounds check and
                                  the access was skipped; bit 8 + s is set for
                                  check site s (results are not valid)        */

/* Compute paths (mla_query_set_path). */
#define MLA_PATH_AUTO 0 /* the default: MLA_PATH_FMA for one token at small
                           head counts (where the FMA kernel's most loaded
                           CTA carries at most 80% of the paired
                           tensor-core kernel's bytes; it measured faster
                           there), MLA_PATH_MMA otherwise                  */
#define MLA_PATH_FMA 1  /* FP32 FMA dot products: the small-batch kernel
                           (batch <= 8 only; MLA_EUNSUPPORTED above)       */
#define MLA_PATH_MMA 2  /* BF16 tensor-core tiles, FP32 accumulate           */

#define MLA_MAX_BATCH 256 /* largest batch one decode call accepts           */
#define MLA_MAX_HEADS 128 /* largest number of local heads                   */

typedef struct mla_query* mla_query_t;

/*
 * mla_query_create - bind one layer's static weights (page "mla.query", class
 * MlaQuery, constructor and the argument list of method kernel: w_qa (gamma_q),
 * w_kva (gamma_kv), w_qb, w_uk, eps).
 *
 *   out       receives the handle (host pointer, must not be NULL).
 *   num_heads local heads H, 1 <= H <= MLA_MAX_HEADS.
 *   w_qb      device BF16 [H*192][1536], row h*192+p is Q_B row p of head h
 *             (p < 128 nope, p >= 128 rope).
 *   w_uk      device BF16 [H][128][512], element (h, p, c).
 *   gamma_q   device BF16 [1536], gamma_kv device BF16 [512].
 *   eps       RMSNorm epsilon used by both norms.
 *
 * W_QB, W_UK and the gammas are borrowed: they must stay valid and unchanged
 * until mla_query_destroy.  Batches of up to 16 tokens read W_QB, W_UK and
 * the gammas in place at every call.  Batches above 16 run the wide kernel,
 * which reads copies of W_QB (H * 576 KiB) and W_UK^T (H * 128 KiB) that
 * create makes once, in swizzled 16 KiB tiles; they read only the gammas in
 * place.  So a weight changed after create is seen by batches of up to 16
 * tokens and not by larger ones: create a new handle to change weights.
 *
 * Device memory: create allocates, with cudaMalloc on the current device,
 * only what the kernels its dispatch can reach need for this head count on
 * this device: the error flag and counters (under 20 KiB); the wide kernel's
 * weight tiles (H * 704 KiB) and normalised-row buffer (192 KiB); where the
 * paired kernel cannot serve every batch of up to 16 tokens (small head
 * counts), the partials kernel's FP32 buffer (H * 256 KiB); and only on a
 * device where neither the wide nor the 16-token paired kernel can run, the
 * hand-off kernel's packed W_UK (H * 128 KiB) and q buffer.  On a GB300 at
 * 64 or 128 heads that is the wide tiles and 192 KiB.  create synchronises
 * the legacy default stream; the handle may only be used on that device.
 * Returns MLA_OK, MLA_EINVAL, MLA_ENOMEM or MLA_ECUDA.
 */
MLA_API int mla_query_create(mla_query_t* out, int num_heads, const void* w_qb,
                     const void* w_uk, const void* gamma_q,
                     const void* gamma_kv, float eps);

/*
 * mla_query_decode - run one decode step (all five steps above) on `stream`.
 *
 *   batch         B tokens, 1 <= B <= MLA_MAX_BATCH.
 *   q_a           device BF16 [B][q_a_stride] (first 1536 used);
 *                 q_a_stride in elements, 0 means 1536; multiple of 8.
 *   kv_c          device BF16 [B][kv_c_stride] (first 512), 0 means 512.
 *   k_pe          device BF16 [B][k_pe_stride] (first 64), 0 means 64.
 *                 (A fused [B][2112] q_a|kv_c|k_pe row is q_a = row,
 *                 kv_c = row + 1536, k_pe = row + 2048, all strides 2112.)
 *   slot_mapping  device int64 [B]; a slot < 0 skips the token's cache row
 *                 (page "mla.query", method insert); a slot >= num_pages *
 *                 page_size is skipped and sets MLA_DEVERR_BAD_SLOT.
 *   kv_cache      device uint8 [num_pages][page_size][row], row = 576
 *                 (MLA_KV_FP8_E4M3), 656 (MLA_KV_FP8_DS_MLA) or 352
 *                 (MLA_KV_NVFP4_DS_MLA) bytes; slot s lives at page
 *                 s / page_size, offset s % page_size.
 *   layout        MLA_KV_FP8_E4M3, MLA_KV_FP8_DS_MLA or MLA_KV_NVFP4_DS_MLA.
 *   k_scale       device FP32 [1]; the per-tensor layout divides by it
 *                 (ignored by the two ds layouts, may then be NULL).
 *   q_latent      device BF16 [B][H][512] output.
 *   q_pe          device BF16 [B][H][64] output.
 *   q_c           device BF16 [B][1536] output, or NULL to skip it.
 *   stream        cudaStream_t as void*.
 *
 * Inputs are read, and outputs written, only after the previous kernel on
 * the stream has completed (programmatic dependent launch: weights may be
 * prefetched earlier).  Calls sharing one handle must be ordered on one
 * stream: they share the handle's scratch.
 * Returns MLA_OK, MLA_EINVAL, MLA_EUNSUPPORTED or MLA_ECUDA (launch error).
 */
MLA_API int mla_query_decode(mla_query_t h, int batch, const void* q_a,
                     int64_t q_a_stride, const void* kv_c, int64_t kv_c_stride,
                     const void* k_pe, int64_t k_pe_stride,
                     const int64_t* slot_mapping, void* kv_cache,
                     int64_t num_pages, int page_size, int layout,
                     const float* k_scale, void* q_latent, void* q_pe,
                     void* q_c, void* stream);

/*
 * mla_query_decode_fp8q - the same decode step with per-tensor FP8 query
 * outputs (page "mla.query", method kernel, the FP8 query epilogue used with
 * the per-tensor FP8 cache for dense MLA): each q_latent and q_pe element is
 * the OCP E4M3 code (round to nearest even, saturating to +-448) of
 * bf16(v) * q_scale_inv, the product rounded to binary32.
 *
 *   q_scale_inv   device FP32 [1] (must not be NULL).
 *   q_latent_fp8  device uint8 [B][H][512] output.
 *   q_pe_fp8      device uint8 [B][H][64] output.
 *   Every other argument, the ordering and the errors as mla_query_decode;
 *   q_c stays BF16.  Returns MLA_EUNSUPPORTED where only the hand-off kernel
 *   could serve the batch (not on a GB300).
 */
MLA_API int mla_query_decode_fp8q(mla_query_t h, int batch, const void* q_a,
                          int64_t q_a_stride, const void* kv_c, int64_t kv_c_stride,
                          const void* k_pe, int64_t k_pe_stride,
                          const int64_t* slot_mapping, void* kv_cache,
                          int64_t num_pages, int page_size, int layout,
                          const float* k_scale, const float* q_scale_inv,
                          void* q_latent_fp8, void* q_pe_fp8, void* q_c, void* stream);

/* ---------------------------------------------------------------------------
 * Gathered query rows (page "mla.query", class MlaQuery, methods publish and
 * gathered: under decode context parallelism each rank writes its query into
 * head block `rank` of a [B][q_heads][576] buffer armed with a sentinel, and
 * the attention side polls until no element is the sentinel).  On one GPU the
 * ranks are decode calls ordered on a stream; each writes its heads' rows in
 * place, and the wait is the same bounded check.
 *
 * A query row is 576 elements: q_latent (512) then q_pe (64), BF16 (2 bytes)
 * or, with q_scale_inv, E4M3 (1 byte).  The sentinel is all ones in every
 * element (a NaN pattern in both types, never written by the decode).
 * ------------------------------------------------------------------------- */
#define MLA_MAX_ROW_HEADS 1024           /* q_heads limit of a row buffer    */
#define MLA_ROWS_WAIT_MAX_NS 2000000000  /* longest wait mla_query_rows_wait accepts */

/*
 * mla_query_decode_rows - the decode step with the query written as rows:
 * q_rows[t][head_offset + h][0..511] = q_latent[t][h], [512..575] = q_pe[t][h].
 *
 *   Arguments up to k_scale as mla_query_decode.
 *   q_scale_inv  device FP32 [1] for E4M3 rows (as mla_query_decode_fp8q),
 *                or NULL for BF16 rows.
 *   q_rows       device [batch][q_heads][576] elements, 16-byte aligned.
 *   q_heads      heads per token in the buffer, <= MLA_MAX_ROW_HEADS (for
 *                example ranks * H, or a padded count the attention kernel
 *                wants); head_offset + H <= q_heads.
 *   head_offset  first head of this call's rows (rank * H).
 *   q_c, stream  as mla_query_decode.
 * Rows of other heads are not touched.  Returns as mla_query_decode, and
 * MLA_EUNSUPPORTED where only the hand-off kernel could run the batch.
 */
MLA_API int mla_query_decode_rows(mla_query_t h, int batch, const void* q_a,
                                  int64_t q_a_stride, const void* kv_c, int64_t kv_c_stride,
                                  const void* k_pe, int64_t k_pe_stride,
                                  const int64_t* slot_mapping, void* kv_cache,
                                  int64_t num_pages, int page_size, int layout,
                                  const float* k_scale, const float* q_scale_inv, void* q_rows,
                                  int q_heads, int head_offset, void* q_c, void* stream);

/*
 * mla_query_rows_arm - set every element of q_rows [batch][q_heads][576]
 * (elem_bytes 1 or 2 per element) to the sentinel, on `stream`.
 * Returns MLA_OK, MLA_EINVAL or MLA_ECUDA.
 */
MLA_API int mla_query_rows_arm(void* q_rows, int batch, int q_heads, int elem_bytes,
                               void* stream);

/*
 * mla_query_rows_wait - on `stream`, poll heads 0..wait_heads-1 of every token
 * of q_rows [batch][q_heads][576] (wait_heads = ranks * H; heads beyond it,
 * padding, are not polled) until no element is the sentinel.  If some
 * element still is after limit_ns nanoseconds (0 <= limit_ns <=
 * MLA_ROWS_WAIT_MAX_NS), the kernel sets MLA_DEVERR_TIMEOUT in the handle's
 * device flags (mla_query_get_error) and returns; the context stays usable.
 * Asynchronous.  Returns MLA_OK, MLA_EINVAL or MLA_ECUDA.
 */
MLA_API int mla_query_rows_wait(mla_query_t h, const void* q_rows, int batch, int q_heads,
                                int wait_heads, int elem_bytes, int64_t limit_ns, void* stream);

/*
 * mla_query_get_error - read and clear the handle's device error flag.
 * Synchronises `stream` (host wait).  *device_flags receives the OR of the
 * MLA_DEVERR_* bits raised since the last call (0 if none).
 */
MLA_API int mla_query_get_error(mla_query_t h, unsigned* device_flags, void* stream);

/*
 * mla_query_set_path - force a compute path (MLA_PATH_*) for later decode
 * calls on this handle; MLA_PATH_AUTO restores the default dispatch.
 * A forced path that cannot serve a batch makes decode return
 * MLA_EUNSUPPORTED.  For tests and tuning; results of every path agree within
 * the library's stated tolerance.
 */
MLA_API int mla_query_set_path(mla_query_t h, int path);

/*
 * mla_query_path_for - the path (MLA_PATH_FMA / MLA_PATH_MMA) a decode call
 * with `batch` tokens takes on this handle; negative on error.
 */
MLA_API int mla_query_path_for(mla_query_t h, int batch);

#define MLA_NOALLOC_MAX_BATCH 64 /* largest batch of mla_query_decode_noalloc */

/*
 * mla_query_decode_noalloc - the same decode step as mla_query_decode, for
 * callers that must not allocate device memory: a serving runtime that
 * reserves all GPU memory for its own pool at start-up, or a plugin loaded
 * into a framework whose allocator owns the device, cannot let a library call
 * cudaMalloc behind its back.  The pages define no such entry point; it has
 * no counterpart there.
 *
 * No handle: the weights, eps and every per-call argument are passed
 * directly (same meaning, layout and alignment rules as mla_query_create and
 * mla_query_decode).  The kernel's scratch (q hand-off buffer and counters)
 * is one fixed device array inside the library, about 2 MiB, that every GPU
 * which loads the library holds until the process exits.  The call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 *   batch         1 <= B <= MLA_NOALLOC_MAX_BATCH (64); a larger batch
 *                 returns MLA_EUNSUPPORTED; num_heads <= MLA_MAX_HEADS.
 *   device_flags  optional caller-owned device word (4-byte aligned) into
 *                 which the call ORs MLA_DEVERR_* bits.  NULL discards them:
 *                 a bad slot then goes unreported, and so does a hand-off
 *                 wait that ran out (its CTAs wait on one another through
 *                 global memory, for up to about a second when other work
 *                 holds the SMs), after which q_latent is not valid.  Pass a
 *                 word where the outputs must be trusted.
 *
 * The first call on a device sets that device up (looks up the array's
 * device address, opts the kernels into their shared memory); make that first
 * call before any stream capture.  The address is kept until the process
 * exits: do not call this entry point on a device after cudaDeviceReset.  Every call shares the one array, and each
 * call clears its counters on `stream` before launching: calls that may
 * overlap on the GPU (different streams, or threads without ordering) race on
 * it and must not be issued; order them on one stream.
 * Returns MLA_OK, MLA_EINVAL, MLA_EUNSUPPORTED or MLA_ECUDA.
 */
MLA_API int mla_query_decode_noalloc(int num_heads, const void* w_qb, const void* w_uk,
                                     const void* gamma_q, const void* gamma_kv, float eps,
                                     int batch, const void* q_a, int64_t q_a_stride,
                                     const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                                     int64_t k_pe_stride, const int64_t* slot_mapping,
                                     void* kv_cache, int64_t num_pages, int page_size,
                                     int layout, const float* k_scale, void* q_latent,
                                     void* q_pe, void* q_c, unsigned* device_flags,
                                     void* stream);

/* mla_query_kernel_for - static text naming the kernels one decode of
 * `batch` tokens launches on this handle and its path, "+" between kernels
 * launched in sequence (a diagnostic: the split by batch size, head count and
 * path).  NULL for a null handle or a batch outside 1..MLA_MAX_BATCH. */
MLA_API const char* mla_query_kernel_for(mla_query_t h, int batch);

/* mla_query_destroy - free the handle and its scratch (NULL is a no-op).
 * The caller must ensure no decode on the handle is still in flight. */
MLA_API void mla_query_destroy(mla_query_t h);

/* mla_query_strerror - static text for a return code. */
MLA_API const char* mla_query_strerror(int code);

/* ---------------------------------------------------------------------------
 * The qkv_a down-projection: the step that produces the fused row the decode
 * step reads (page "ws_gemm", class WsGemm: y[M, N] = x[M, K] @ W[N, K]^T,
 * BF16 operands, FP32 accumulation, BF16 outputs; page "mla.query", method
 * kernel: the qkv row holds q_a at columns 0..1535, kv_c at 1536..2047 and
 * k_pe at 2048..2111).  With W = the stacked q_a / kv_a projections
 * [2112][7168], y[b] can be handed to mla_query_decode as a fused row
 * (q_a = y, kv_c = y + 1536, k_pe = y + 2048, all strides 2112); run on the
 * same stream, the decode's weight streaming overlaps this call's tail.
 * ------------------------------------------------------------------------- */
typedef struct mla_qkv_a* mla_qkv_a_t;

/*
 * mla_qkv_a_create - bind the projection weight.
 *
 *   out  receives the handle.
 *   n    output columns (rows of W), 1 <= n; n / SMs rounded up must be at
 *        most 15 (n <= 2280 on 152 SMs).
 *   k    input columns, a multiple of 512, 512 <= k <= 7168.
 *   w    device BF16 [n][k], row-major, 16-byte aligned.  Borrowed: read in
 *        place at every call, so it must stay valid and unchanged until
 *        mla_qkv_a_destroy.
 *
 * Allocates a 4-byte device error word.  Returns MLA_OK, MLA_EINVAL (null or
 * misaligned pointer, bad n or k), MLA_EUNSUPPORTED (n or k beyond the limits
 * above), MLA_ENOMEM or MLA_ECUDA.
 */
MLA_API int mla_qkv_a_create(mla_qkv_a_t* out, int n, int k, const void* w);

/*
 * mla_qkv_a_run - y[b][j] = bf16(sum_i x[b][i] * W[j][i]) for b < batch, on
 * `stream`, asynchronously (no host sync, no allocation).
 *
 *   batch     1 <= batch <= MLA_MAX_BATCH; one launch per 8 tokens.
 *   x         device BF16 [batch][x_stride] (first k used), 16-byte aligned;
 *             x_stride in elements, 0 means k; a multiple of 8.
 *   y         device BF16 [batch][y_stride] output (first n written);
 *             y_stride in elements, 0 means n.
 *   stream    cudaStream_t as void*.
 *
 * W is streamed before the previous kernel on the stream completes
 * (programmatic dependent launch); x is read, and y written, only after it.
 * Returns MLA_OK, MLA_EINVAL or MLA_ECUDA (launch error).
 */
MLA_API int mla_qkv_a_run(mla_qkv_a_t h, int batch, const void* x, int64_t x_stride, void* y,
                          int64_t y_stride, void* stream);

/* mla_qkv_a_get_error - read and clear the handle's device error word
 * (MLA_DEVERR_TIMEOUT if a bounded wait gave up); synchronises `stream`. */
MLA_API int mla_qkv_a_get_error(mla_qkv_a_t h, unsigned* device_flags, void* stream);

/* mla_qkv_a_destroy - free the handle (NULL is a no-op).  No call on it may
 * still be in flight. */
MLA_API void mla_qkv_a_destroy(mla_qkv_a_t h);

#ifdef __cplusplus
}
#endif

#endif /* MLA_QUERY_H */
