/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged KV-cache library.
 *
 * Operations of the decode/prefill hot path of a paged-KV serving engine:
 *   pa_reshape_and_cache           scatter per-token K/V into a paged cache
 *   pa_concat_mla_k                assemble MLA K from k_nope and a shared k_rope
 *   pa_concat_and_cache_mla        write MLA latent rows [c_kv | k_pe] into a paged cache
 *   pa_paged_decode_attention      GQA decode attention over the paged cache
 *   pa_paged_decode_attention_fp8  the same over an FP8 E4M3 cache with scales
 *   pa_paged_decode_step           new-token cache write + decode attention, one launch
 *   pa_paged_prefill_attention     causal varlen prefill attention over the paged cache
 *   pa_mla_absorb_q                MLA: absorbed query [W_UK_h q_nope | q_pe]
 *   pa_mla_decode_attention        MLA: decode attention over the paged latent cache
 *   pa_mla_project_out             MLA: latent output times W_UV_h
 *
 * Common rules
 *   - Every pointer argument except the `*_host` ones is a DEVICE pointer on
 *     the current CUDA device.  The caller owns every buffer; the library
 *     never allocates, frees or synchronises, and keeps no state besides
 *     per-device caches of the SM count, of one driver entry point and of
 *     the address of the static decode scratch (see the _static call).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and
 *     runs asynchronously.  No call reads device memory on the host or
 *     branches on device data, so every call can be captured in a CUDA graph
 *     (the PagedAttention-principle post, section on host->device metadata
 *     transfer, explains why host-side branching on device state is
 *     incompatible with graph capture).
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error code and launches nothing.  Index values
 *     that live in device memory (slots, SWA entries, block ids, context
 *     lengths) are checked on the device: an out-of-range value is skipped,
 *     never dereferenced.
 *   - "Elements" in strides are elements of the array's own dtype.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (the runtime's typedef of this pointer). */
typedef struct CUstream_st *pa_stream_t;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,     /* null pointer, bad size, inconsistent arguments */
  PA_ERR_UNSUPPORTED = 2, /* valid but not implemented (dtype pair, head size) */
  PA_ERR_ALIGN = 3,       /* pointer or stride breaks the vector-access rules */
  PA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  PA_ERR_CUDA = 5         /* a CUDA runtime call or a launch failed */
} pa_status;

typedef enum {
  PA_BF16 = 0,
  PA_FP16 = 1,
  PA_FP32 = 2,
  PA_FP8_E4M3 = 3 /* OCP FP8 E4M3 (max 448, no inf, 0x7F/0xFF NaN) */
} pa_dtype;

/* Bits of the device-side error word (first 4 bytes of a decode workspace). */
#define PA_DEVERR_WAIT_TIMEOUT 0x1u   /* a pipeline wait gave up (should never happen) */
#define PA_DEVERR_CONTEXT_CLIPPED 0x2u /* some context_lens[b] exceeded the planned range */
#define PA_DEVERR_SLOT_MISMATCH 0x4u   /* decode step: a slot was not position L-1's slot */

/* ------------------------------------------------------------------------
 * pa_reshape_and_cache
 *
 * Defined by sglang kernels/ops/kvcache/cache_ops.py, reshape_and_cache_flash
 * and launch_reshape_and_cache_flash ("slot mapping", "optional scale" and
 * "target layout" blocks), and the nano-vLLM walkthrough, section 2.6
 * Attention (store_kvcache_kernel).  For every token t:
 *     s = slot_mapping[t]
 *     if s < 0: skip                                  (-1 marks padding)
 *     if swa_slot_mapping: if s >= swa_len: skip; s = swa_slot_mapping[s];
 *                          if s < 0: skip
 *     if s >= num_blocks * block_size: skip
 *     for h, i:  y = x[t, h, i]  (as float);  if scales: y = y / scale (IEEE)
 *         cache[s / block_size, s % block_size, h, i] = cast(y)
 * for K and V.  The cast rounds to nearest-even; to E4M3 it saturates to
 * +-448.  Two tokens that resolve to the same slot: unspecified winner.
 *
 * key, value:   [num_tokens, num_heads, head_size], key_stride/value_stride
 *               elements between tokens; heads and elements contiguous.
 *               value may be NULL (K-only cache, e.g. an MLA latent cache);
 *               then value_cache must be NULL too.
 * key_cache, value_cache: [num_blocks, block_size, num_heads, head_size],
 *               block_stride elements between blocks, the rest contiguous.
 * src_dtype:    PA_BF16, PA_FP16 or PA_FP32.
 * cache_dtype:  PA_BF16, PA_FP16, PA_FP32 or PA_FP8_E4M3.
 * slot_mapping: [num_tokens] int64.
 * swa_slot_mapping: NULL or [swa_len] int64 second-stage table.
 * k_scale, v_scale: both NULL or both device pointers to one float (> 0).
 * Alignment: key/value/caches 16-byte aligned; num_heads*head_size,
 *   key_stride, value_stride and block_stride multiples of 8 elements.
 * Errors: PA_ERR_INVALID (null/negative/inconsistent), PA_ERR_UNSUPPORTED
 *   (dtype pair), PA_ERR_ALIGN, PA_ERR_CUDA (launch failed).
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache(const void *key, const void *value, pa_dtype src_dtype,
                               int64_t num_tokens, int32_t num_heads, int32_t head_size,
                               int64_t key_stride, int64_t value_stride, void *key_cache,
                               void *value_cache, pa_dtype cache_dtype, int64_t num_blocks,
                               int32_t block_size, int64_t block_stride,
                               const int64_t *slot_mapping, const int64_t *swa_slot_mapping,
                               int64_t swa_len, const float *k_scale, const float *v_scale,
                               pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_concat_mla_k
 *
 * Defined by sglang cache_ops.py, concat_and_cast_mha_k_kernel and
 * concat_and_cast_mha_k_triton:
 *     k[n, h, 0:nope_dim]                  = k_nope[n, h, :]
 *     k[n, h, nope_dim:nope_dim+rope_dim]  = k_rope[n, 0, :]   (all heads)
 * with an implicit round-to-nearest-even cast to k_dtype (E4M3 saturates).
 * Shapes: k [num_tokens, num_heads, nope_dim + rope_dim],
 *         k_nope [num_tokens, num_heads, nope_dim], k_rope [num_tokens, 1, rope_dim];
 *         the wrapper's shape checks become num_heads >= 1, equal token
 *         counts (a single num_tokens) and k's last size = nope + rope.
 * Strides in elements of each tensor; the last dimension is contiguous.
 * src_dtype: PA_BF16, PA_FP16 or PA_FP32; k_dtype: any pa_dtype.
 * Alignment: pointers 16-byte aligned; nope_dim, rope_dim and every stride
 *   multiples of 8 elements.
 * ---------------------------------------------------------------------- */
pa_status pa_concat_mla_k(void *k, pa_dtype k_dtype, const void *k_nope, const void *k_rope,
                          pa_dtype src_dtype, int64_t num_tokens, int32_t num_heads,
                          int32_t nope_dim, int32_t rope_dim, int64_t k_stride0,
                          int64_t k_stride1, int64_t nope_stride0, int64_t nope_stride1,
                          int64_t rope_stride0, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_concat_and_cache_mla -- the MLA latent-cache write in one pass.
 *
 * PagedAttention-principle post, MLA section: what a token caches is its
 * latent c_kv (d_c elements) with the rope part of its key, k_pe (d_r,
 * shared by the heads), beside it.  For every token t:
 *     s = slot_mapping[t];  skip if s < 0 or s >= num_blocks * block_size
 *     latent_cache[s / block_size, s % block_size, 0:d_c]       = cast(kv_c[t] / scale)
 *     latent_cache[s / block_size, s % block_size, d_c:d_c+d_r] = cast(k_pe[t] / scale)
 * (without a scale, a plain cast), i.e. the same bytes as pa_concat_mla_k
 * with one head (assembling [kv_c | k_pe]) followed by pa_reshape_and_cache
 * with head_size d_c + d_r and no value cache, but with one read and one
 * write of each row.  Casts and the scale division as in
 * pa_reshape_and_cache.
 *
 * kv_c [num_tokens, latent_dim], k_pe [num_tokens, rope_dim]: kv_c_stride,
 *   k_pe_stride elements between tokens, rows contiguous; src_dtype PA_BF16,
 *   PA_FP16 or PA_FP32.
 * latent_cache [num_blocks, block_size, latent_dim + rope_dim] of
 *   cache_dtype (any pa_dtype), block_stride elements between blocks.
 * slot_mapping [num_tokens] int64.  scale: NULL or a device pointer to one
 *   float (> 0).
 * Alignment: pointers 16-byte aligned; latent_dim, rope_dim and the strides
 *   multiples of 8 elements.
 * Errors: PA_ERR_INVALID, PA_ERR_UNSUPPORTED (dtype pair), PA_ERR_ALIGN,
 *   PA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
pa_status pa_concat_and_cache_mla(const void *kv_c, const void *k_pe, pa_dtype src_dtype,
                                  int64_t num_tokens, int32_t latent_dim, int32_t rope_dim,
                                  int64_t kv_c_stride, int64_t k_pe_stride, void *latent_cache,
                                  pa_dtype cache_dtype, int64_t num_blocks, int32_t block_size,
                                  int64_t block_stride, const int64_t *slot_mapping,
                                  const float *scale, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * Paged GQA decode attention.
 *
 * The cache is read back along the block table (nano-vLLM walkthrough,
 * section 2.6: the decode attention kernel reads the physical blocks via
 * block_tables; PagedAttention-principle post, "paged attention原理": blocks
 * are physically scattered and the table keeps their logical order).  For
 * sequence b and query head h, with G = num_q_heads / num_kv_heads and
 * L = context_lens[b]:
 *     kv head g = h / G; logical token j lives at physical row
 *         block_tables[b][j / block_size] * block_size + j % block_size
 *     out[b, h] = softmax_j(scale * q[b, h] . K_j) @ V_j,   j < L
 * L counts the token just written (write, then attend).  L = 0 gives a
 * zero row.  A block id outside [0, num_blocks) drops its tokens from the
 * softmax.
 *
 * q, out: [num_seqs, num_q_heads, head_size] bf16, contiguous.
 * k_cache, v_cache: [num_blocks, block_size, num_kv_heads, head_size],
 *   contiguous, cache_dtype PA_BF16, or PA_FP8_E4M3 read with unit scales
 *   (see pa_paged_decode_attention_fp8); other dtypes: PA_ERR_UNSUPPORTED.
 * block_tables: [num_seqs, max_blocks_per_seq] int32; context_lens [num_seqs] int32.
 * head_size: 128.  block_size: a power of two in [8, 256].
 * G: 1, 2, 4, 8 or 16.  num_seqs above 65535: PA_ERR_UNSUPPORTED (one grid
 * dimension per sequence).
 * max_context_len: host-side upper bound on every context_lens[b]; it sets
 *   the split plan.  Larger lengths are clipped to the plan (and to
 *   max_blocks_per_seq * block_size) and flag PA_DEVERR_CONTEXT_CLIPPED.
 * workspace: device buffer of at least pa_paged_decode_workspace_size(...)
 *   bytes, 256-byte aligned, ZEROED ONCE by the caller before first use.
 *   Its first 4 bytes are a sticky device-side error word (PA_DEVERR_*);
 *   the caller reads it whenever it likes and clears it to reset.  It also
 *   holds per-(sequence, kv head) split counters that every call leaves at
 *   zero.  Calls that share a workspace must be ordered on one stream.
 * Alignment: q, out, caches 16-byte aligned.
 *
 * The context is split into equal token ranges (a plan computed from
 * num_seqs, num_kv_heads, max_context_len and the SM count); each
 * (kv head, range, sequence) is one CTA, kv heads adjacent in launch order
 * (the CTAs of one range read the same token rows together), that streams
 * its K/V blocks through shared memory, computes the grouped products on
 * the tensor cores and keeps an fp32 online softmax; the last CTA of each
 * (sequence, kv head) merges the ranges by log-sum-exp.  One launch per call.
 *
 * pa_paged_decode_workspace_size returns the bytes the call above needs
 * (0 for invalid sizes).  It takes num_kv_heads and no block_size: the
 * split plan counts CTAs per (sequence, kv head) and cuts token ranges in
 * multiples of 64 tokens whatever the block size, so the partials depend on
 * num_seqs, num_q_heads, num_kv_heads, head_size and max_context_len only.
 * ---------------------------------------------------------------------- */
size_t pa_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_size,
                                      int32_t max_context_len);

pa_status pa_paged_decode_attention(void *out, const void *q, const void *k_cache,
                                    const void *v_cache, pa_dtype cache_dtype,
                                    const int32_t *block_tables, const int32_t *context_lens,
                                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_size, int32_t block_size,
                                    int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                                    int32_t max_context_len, void *workspace,
                                    size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_paged_decode_attention_fp8 -- decode attention over an FP8 E4M3 cache.
 *
 * The cache holds x / k_scale and x / v_scale rounded to e4m3 (written by
 * pa_reshape_and_cache with the same scales: sglang cache_ops.py,
 * reshape_and_cache_flash, "optional scale"), so a code stands for
 * code * scale.  Computes the same attention as pa_paged_decode_attention
 * with K_j = code * k_scale and V_j = code * v_scale; the codes are read as
 * they are (half the bytes of bf16), k_scale folds into the score scale and
 * v_scale into the output.  k_scale, v_scale: both NULL (unit scales) or
 * both device pointers to one float.  Other arguments, the workspace and the
 * error word as for pa_paged_decode_attention (which also accepts
 * PA_FP8_E4M3 caches, with unit scales).  The grouped products run in f16
 * on the tensor cores: q is carried with a power-of-two prescale, so q
 * values must be finite.
 * ---------------------------------------------------------------------- */
pa_status pa_paged_decode_attention_fp8(void *out, const void *q, const void *k_cache,
                                        const void *v_cache, const float *k_scale,
                                        const float *v_scale, const int32_t *block_tables,
                                        const int32_t *context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_size, int32_t block_size,
                                        int32_t max_blocks_per_seq, int64_t num_blocks,
                                        float scale, int32_t max_context_len, void *workspace,
                                        size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_paged_decode_step -- one decode step in one launch: write each
 * sequence's newest K/V token into the cache, then attend.
 *
 * Same result as pa_reshape_and_cache(new_k, new_v, ..., slot_mapping,
 * k_scale, v_scale) followed by pa_paged_decode_attention(_fp8) (the
 * PagedAttention-principle post, decode dataflow: compute the new token's
 * q/k/v, write the KV cache, then compute attention).  The CTA that holds
 * position context_lens[b] - 1 converts the new row exactly as the cache
 * write does, stores it at slot_mapping[b] and uses it directly.
 *
 * new_k, new_v: [num_seqs, num_kv_heads, head_size] bf16, contiguous,
 *   16-byte aligned.  slot_mapping: [num_seqs] int64; -1 (or any slot
 *   outside the pool) skips that sequence's write.  A slot that is not the
 *   slot of position context_lens[b] - 1 is still written but not attended
 *   to in this call, and sets PA_DEVERR_SLOT_MISMATCH (no other CTA may be
 *   reading it: keep slot_mapping consistent with the block table).
 * cache_dtype PA_BF16 (k_scale, v_scale NULL) or PA_FP8_E4M3 (scales as in
 *   pa_paged_decode_attention_fp8).  Other arguments as for
 *   pa_paged_decode_attention.
 * ---------------------------------------------------------------------- */
pa_status pa_paged_decode_step(void *out, const void *q, const void *new_k, const void *new_v,
                               const int64_t *slot_mapping, void *k_cache, void *v_cache,
                               pa_dtype cache_dtype, const float *k_scale, const float *v_scale,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_size, int32_t block_size, int32_t max_blocks_per_seq,
                               int64_t num_blocks, float scale, int32_t max_context_len,
                               void *workspace, size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_paged_prefill_attention -- causal varlen prefill attention over the
 * paged cache (the nano-vLLM walkthrough names varlen flash attention with
 * cu_seqlens_q for prefill; section 2.6: attention reads the cache along
 * block_tables).
 *
 * Sequence b has n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens; they
 * are the last n_b of its L_b = context_lens[b] tokens, whose K/V are already
 * in the cache (pa_reshape_and_cache first).  New token j of sequence b is
 * at position p = L_b - n_b + j and
 *     out[cu_seqlens_q[b] + j, h] = softmax_{t <= p}(scale q.K_t) @ V_t
 * with K_t, V_t of kv head h / (H_Q / H_KV) read through the block table.
 * Positions below zero (n_b > L_b) give zero rows; a block id outside the
 * pool drops its tokens.
 *
 * q, out: [total_new_tokens, num_q_heads, 128] bf16, contiguous;
 * cu_seqlens_q [num_seqs + 1] int32 (device), context_lens [num_seqs] int32;
 * caches, block table, block_size, G as for pa_paged_decode_attention
 * (bf16 caches).  max_q_len: host upper bound on every n_b (sets the grid;
 * tokens past it are not computed).  error_word: device pointer to one
 * 4-byte word receiving PA_DEVERR_* bits (the caller clears it).
 * Numerics: fp32 accumulation and softmax; the softmax weights enter the
 * P.V product rounded to bf16.
 * ---------------------------------------------------------------------- */
pa_status pa_paged_prefill_attention(void *out, const void *q, const void *k_cache,
                                     const void *v_cache, pa_dtype cache_dtype,
                                     const int32_t *block_tables, const int32_t *cu_seqlens_q,
                                     const int32_t *context_lens, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int32_t max_blocks_per_seq,
                                     int64_t num_blocks, float scale, int32_t max_q_len,
                                     unsigned *error_word, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_paged_decode_attention_static -- the same decode attention for callers
 * that cannot allocate device memory.
 *
 * No counterpart in the paper: this is a deployment variant of the call
 * above.  Some callers never get to call cudaMalloc: a plugin inside a host
 * runtime that owns every device buffer and hands the plugin only its input
 * and output tensors, or a latency-critical loop that must not risk the
 * device-wide synchronisation an allocation can cause.  Such a caller
 * cannot provide the split-K workspace, so this entry point uses a scratch
 * area compiled into the library instead (a 16 MiB __device__ array that
 * every GPU loading the library holds until the process exits).  It
 * allocates nothing and calls no allocating routine.
 *
 * Arguments are those of pa_paged_decode_attention without the workspace;
 * the caller still passes every input and the output.  error_word: NULL or
 * a device pointer to one 4-byte word that receives the PA_DEVERR_* bits of
 * this call (OR-ed in; the caller clears it).  With NULL the bits go to the
 * first word of the library's own scratch, which no call reads or clears:
 * they are lost, harmlessly.
 * Limits: a problem whose split-K partials need more than 16 MiB (see
 * pa_paged_decode_workspace_size) returns PA_ERR_WORKSPACE and launches
 * nothing.  The first call on a device looks up the scratch's device
 * address (once per device, with that device current) and keeps it for the
 * life of the process; make that first call before any stream capture.  A
 * device reset (cudaDeviceReset) after the first call is not supported: the
 * kept address would be stale.  All calls share the one scratch area,
 * and each call overwrites what the last one left there (the split counters
 * in it, which must start at zero, are zero when the library loads and every
 * completed call returns them to zero): calls that may
 * overlap on the GPU (different streams, no ordering between them) race and
 * give wrong results -- order them on one stream.
 * ---------------------------------------------------------------------- */
pa_status pa_paged_decode_attention_static(void *out, const void *q, const void *k_cache,
                                           const void *v_cache, pa_dtype cache_dtype,
                                           const int32_t *block_tables,
                                           const int32_t *context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_size, int32_t block_size,
                                           int32_t max_blocks_per_seq, int64_t num_blocks,
                                           float scale, int32_t max_context_len,
                                           unsigned *error_word, pa_stream_t stream);

/* The split plan the decode calls above use: *num_splits token ranges of
 * *tokens_per_split tokens each.  num_sms <= 0 means "the current
 * device's SM count".  Host only; launches nothing. */
pa_status pa_paged_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len,
                               int32_t num_sms, int32_t *num_splits_host,
                               int32_t *tokens_per_split_host);

/* ========================================================================
 * MLA decode over the latent cache
 *
 * PagedAttention-principle post, MLA section ("MLA 不直接缓存 k 和 v"): a
 * token's cache entry is its latent c_kv = x W_DKV ([d_c]); head h's K and
 * V are c_kv W_UK_h and c_kv W_UV_h, with W_UK, W_UV: [d_c, H * d_h] and
 * head h owning columns h*d_h .. (h+1)*d_h - 1; the rope part of K (k_pe,
 * [d_r], shared by the heads) is added separately.  The cache row of a
 * token is [c_kv | k_pe] (d_c + d_r elements), the layout
 * [num_blocks, block_size, 1, d_c + d_r] that pa_reshape_and_cache writes
 * with num_heads = 1, head_size = d_c + d_r and no value cache.
 *
 * Decode runs in the absorbed form (associativity of the products):
 *   q_lat[b,h] = [W_UK_h q_nope[b,h] | q_pe[b,h]]            pa_mla_absorb_q
 *   o_lat[b,h] = sum_j softmax_j(scale q_lat[b,h] . row_j) row_j[0:d_c]
 *                                                   pa_mla_decode_attention
 *   out[b,h]   = o_lat[b,h] W_UV_h                          pa_mla_project_out
 * which equals attention with the explicitly reconstructed K and V.
 * ====================================================================== */

/* q_latent [num_seqs, num_heads, latent_dim + rope_dim] bf16 (written) from
 * q_nope [num_seqs, num_heads, nope_dim], q_pe [num_seqs, num_heads,
 * rope_dim] and w_uk [latent_dim, num_heads * nope_dim], all bf16 and
 * contiguous.  nope_dim and latent_dim must be multiples of 64, rope_dim of
 * 8; pointers 16-byte aligned.  fp32 accumulation, one bf16 rounding. */
pa_status pa_mla_absorb_q(void *q_latent, const void *q_nope, const void *q_pe, const void *w_uk,
                          int32_t num_seqs, int32_t num_heads, int32_t nope_dim, int32_t rope_dim,
                          int32_t latent_dim, pa_stream_t stream);

/* Bytes of workspace pa_mla_decode_attention needs for these sizes on the
 * current device (0 for invalid sizes).  The first 4 bytes are the device
 * error word (PA_DEVERR_* bits; the caller clears it); the rest must be zero
 * before the first call and is left zero by every completed call. */
size_t pa_mla_decode_workspace_size(int32_t num_seqs, int32_t num_heads,
                                    int32_t max_context_len);

/* out_latent [num_seqs, num_heads, latent_dim] bf16 = the attention of each
 * q_latent row [num_seqs, num_heads, latent_dim + rope_dim] (bf16) over the
 * first context_lens[b] tokens of latent_cache [num_blocks, block_size,
 * latent_dim + rope_dim] (bf16), read through block_tables [num_seqs,
 * max_blocks_per_seq] (int32, logical block i of sequence b is physical
 * block block_tables[b][i]); scores over all latent_dim + rope_dim
 * elements, values = the first latent_dim.  Supported: latent_dim 512,
 * rope_dim 64, num_heads a multiple of 16, block_size a power of two in
 * [8, 256].  max_context_len: host hint on context_lens (0 or less: a
 * one-chunk plan); the work is cut into equal token chunks from the actual
 * context_lens on the device, so no length is clipped to the hint.  A
 * length beyond max_blocks_per_seq * block_size is clipped to the table and
 * flagged (PA_DEVERR_CONTEXT_CLIPPED).
 * A block id outside [0, num_blocks) drops its tokens; an empty context
 * gives a zero row.  Numerics: fp32 scores, softmax and accumulation; the
 * softmax weights enter the weighted sum rounded to bf16.  Pointers
 * 16-byte aligned (workspace 256). */
pa_status pa_mla_decode_attention(void *out_latent, const void *q_latent,
                                  const void *latent_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int32_t num_seqs,
                                  int32_t num_heads, int32_t latent_dim, int32_t rope_dim,
                                  int32_t block_size, int32_t max_blocks_per_seq,
                                  int64_t num_blocks, float scale, int32_t max_context_len,
                                  void *workspace, size_t workspace_bytes, pa_stream_t stream);

/* out [num_seqs, num_heads, v_head_dim] bf16 = out_latent[b, h, :] (bf16,
 * [num_seqs, num_heads, latent_dim]) times W_UV_h, w_uv [latent_dim,
 * num_heads * v_head_dim] bf16.  latent_dim and v_head_dim multiples of 64;
 * pointers 16-byte aligned.  fp32 accumulation, one bf16 rounding. */
pa_status pa_mla_project_out(void *out, const void *out_latent, const void *w_uv,
                             int32_t num_seqs, int32_t num_heads, int32_t latent_dim,
                             int32_t v_head_dim, pa_stream_t stream);

/* Diagnostic of the failure path every pipeline kernel shares: launches one
 * CTA whose threads wait, with the same bounded wait the pipelines use, on a
 * barrier that nothing completes.  After the wait limit (2 s) the kernel
 * sets PA_DEVERR_WAIT_TIMEOUT in *error_word (a device pointer to one 4-byte
 * word, 4-byte aligned; the caller clears it) and exits, leaving the context
 * usable.  Stream-ordered; returns PA_ERR_INVALID for a null word and
 * PA_ERR_CUDA if the launch fails. */
pa_status pa_selftest_bounded_wait(unsigned *error_word, pa_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
