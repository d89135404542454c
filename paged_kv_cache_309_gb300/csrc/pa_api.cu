// pa_api.cu -- extern "C" entry points of libpa: argument checks, then the
// launchers.  Nothing here allocates, synchronises or reads device memory.
#include <atomic>
#include <cmath>

#include "pa_internal.cuh"

namespace pa_detail {

int num_sms_current_device() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev].load();
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n);
  return n;
}

}  // namespace pa_detail

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_src_dtype(pa_dtype d) { return d == PA_BF16 || d == PA_FP16 || d == PA_FP32; }
bool is_any_dtype(pa_dtype d) { return is_src_dtype(d) || d == PA_FP8_E4M3; }

// Host-side checks shared by both decode entry points; fills *a (all but the
// workspace) on success.
pa_status check_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                       pa_dtype cache_dtype, const int32_t* block_tables,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                       int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                       int32_t max_context_len, pa_detail::DecodeArgs* a) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 ||
      max_context_len > (1 << 30))
    return PA_ERR_INVALID;
  if (out == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr ||
      block_tables == nullptr || context_lens == nullptr)
    return PA_ERR_INVALID;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID;
  if (!std::isfinite(scale)) return PA_ERR_INVALID;
  if (cache_dtype != PA_BF16 && cache_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (head_size != 128) return PA_ERR_UNSUPPORTED;
  const int32_t G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return PA_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)) != 0)
    return PA_ERR_UNSUPPORTED;
  if (num_blocks * block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PA_ERR_ALIGN;
  a->out = out;
  a->q = q;
  a->k_cache = k_cache;
  a->v_cache = v_cache;
  a->block_tables = block_tables;
  a->context_lens = context_lens;
  a->num_seqs = num_seqs;
  a->num_q_heads = num_q_heads;
  a->num_kv_heads = num_kv_heads;
  a->head_size = head_size;
  a->block_size = block_size;
  a->max_blocks_per_seq = max_blocks_per_seq;
  a->num_blocks = num_blocks;
  a->scale = scale;
  a->cache_dtype = cache_dtype;
  a->k_scale = nullptr;
  a->v_scale = nullptr;
  a->plan = pa_detail::make_decode_plan(num_seqs, num_kv_heads, max_context_len,
                                        pa_detail::num_sms_current_device());
  return PA_OK;
}

// One CTA waits on a barrier nothing arrives on: the bounded wait gives up
// after its limit and the error bit is set, as in any pipeline kernel.
__global__ void selftest_bounded_wait_kernel(unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pa::mbar_init(&bar, 1);
    pa::mbar_init_fence();
  }
  __syncthreads();
  const bool ok = pa::mbar_wait_bounded(&bar, 0, nullptr);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicOr(err, PA_DEVERR_WAIT_TIMEOUT);
}

}  // namespace

extern "C" {

pa_status pa_selftest_bounded_wait(unsigned* error_word, pa_stream_t stream) {
  if (error_word == nullptr || !aligned(error_word, 4)) return PA_ERR_INVALID;
  selftest_bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(error_word);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: unsupported configuration";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer or stride misaligned for vector access";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime or launch failure";
  }
  return "unknown pa_status";
}

pa_status pa_reshape_and_cache(const void* key, const void* value, pa_dtype src_dtype,
                               int64_t num_tokens, int32_t num_heads, int32_t head_size,
                               int64_t key_stride, int64_t value_stride, void* key_cache,
                               void* value_cache, pa_dtype cache_dtype, int64_t num_blocks,
                               int32_t block_size, int64_t block_stride,
                               const int64_t* slot_mapping, const int64_t* swa_slot_mapping,
                               int64_t swa_len, const float* k_scale, const float* v_scale,
                               pa_stream_t stream) {
  if (num_tokens < 0 || num_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
    return PA_ERR_INVALID;
  if (num_tokens == 0) return PA_OK;  // nothing to write; pointers may be null
  if (key == nullptr || key_cache == nullptr || slot_mapping == nullptr) return PA_ERR_INVALID;
  if ((value == nullptr) != (value_cache == nullptr)) return PA_ERR_INVALID;
  if ((k_scale == nullptr) != (v_scale == nullptr)) return PA_ERR_INVALID;
  if (swa_slot_mapping != nullptr && swa_len < 0) return PA_ERR_INVALID;
  if (!is_src_dtype(src_dtype) || !is_any_dtype(cache_dtype)) return PA_ERR_UNSUPPORTED;
  const int64_t row = static_cast<int64_t>(num_heads) * head_size;
  if (row % 8 != 0) return PA_ERR_ALIGN;
  if (row / 8 > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
  if (key_stride % 8 != 0 || block_stride % 8 != 0 || (value && value_stride % 8 != 0))
    return PA_ERR_ALIGN;
  if (num_tokens > 1 && (key_stride < row || (value && value_stride < row))) return PA_ERR_INVALID;
  if (num_blocks > 1 && block_stride < row * block_size) return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(key_cache, 16) || (value && !aligned(value, 16)) ||
      (value_cache && !aligned(value_cache, 16)))
    return PA_ERR_ALIGN;

  pa_detail::ReshapeArgs a{};
  a.key = key;
  a.value = value;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.slot_mapping = slot_mapping;
  a.swa = swa_slot_mapping;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.swa_len = swa_slot_mapping ? swa_len : 0;
  a.num_tokens = num_tokens;
  a.key_stride = key_stride;
  a.value_stride = value ? value_stride : 0;
  a.block_stride = block_stride;
  a.num_slots = num_blocks * block_size;
  a.row_chunks = static_cast<int32_t>(row / 8);
  a.block_size = block_size;
  return pa_detail::launch_reshape_and_cache(a, src_dtype, cache_dtype,
                                             reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_concat_mla_k(void* k, pa_dtype k_dtype, const void* k_nope, const void* k_rope,
                          pa_dtype src_dtype, int64_t num_tokens, int32_t num_heads,
                          int32_t nope_dim, int32_t rope_dim, int64_t k_stride0,
                          int64_t k_stride1, int64_t nope_stride0, int64_t nope_stride1,
                          int64_t rope_stride0, pa_stream_t stream) {
  if (num_tokens < 0 || num_heads <= 0 || nope_dim <= 0 || rope_dim <= 0) return PA_ERR_INVALID;
  if (num_tokens == 0) return PA_OK;  // nothing to assemble; pointers may be null
  if (k == nullptr || k_nope == nullptr || k_rope == nullptr) return PA_ERR_INVALID;
  if (!is_src_dtype(src_dtype) || !is_any_dtype(k_dtype)) return PA_ERR_UNSUPPORTED;
  if (nope_dim % 8 != 0 || rope_dim % 8 != 0) return PA_ERR_ALIGN;
  if (k_stride0 % 8 || k_stride1 % 8 || nope_stride0 % 8 || nope_stride1 % 8 || rope_stride0 % 8)
    return PA_ERR_ALIGN;
  if (k_stride1 < 0 || k_stride0 < 0 || nope_stride0 < 0 || nope_stride1 < 0 || rope_stride0 < 0)
    return PA_ERR_INVALID;
  if (num_heads > 1 && (k_stride1 < nope_dim + rope_dim || nope_stride1 < nope_dim))
    return PA_ERR_INVALID;
  if (!aligned(k, 16) || !aligned(k_nope, 16) || !aligned(k_rope, 16)) return PA_ERR_ALIGN;
  pa_detail::ConcatArgs a{};
  a.k = k;
  a.k_nope = k_nope;
  a.k_rope = k_rope;
  a.num_tokens = num_tokens;
  a.k_stride0 = k_stride0;
  a.k_stride1 = k_stride1;
  a.nope_stride0 = nope_stride0;
  a.nope_stride1 = nope_stride1;
  a.rope_stride0 = rope_stride0;
  a.num_heads = num_heads;
  a.nope_chunks = nope_dim / 8;
  a.rope_chunks = rope_dim / 8;
  return pa_detail::launch_concat_mla_k(a, src_dtype, k_dtype,
                                        reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_concat_and_cache_mla(const void* kv_c, const void* k_pe, pa_dtype src_dtype,
                                  int64_t num_tokens, int32_t latent_dim, int32_t rope_dim,
                                  int64_t kv_c_stride, int64_t k_pe_stride, void* latent_cache,
                                  pa_dtype cache_dtype, int64_t num_blocks, int32_t block_size,
                                  int64_t block_stride, const int64_t* slot_mapping,
                                  const float* scale, pa_stream_t stream) {
  if (num_tokens < 0 || latent_dim <= 0 || rope_dim <= 0 || block_size <= 0 || num_blocks < 0)
    return PA_ERR_INVALID;
  if (num_tokens == 0) return PA_OK;  // nothing to write; pointers may be null
  if (kv_c == nullptr || k_pe == nullptr || latent_cache == nullptr || slot_mapping == nullptr)
    return PA_ERR_INVALID;
  if (!is_src_dtype(src_dtype) || !is_any_dtype(cache_dtype)) return PA_ERR_UNSUPPORTED;
  if (latent_dim % 8 != 0 || rope_dim % 8 != 0) return PA_ERR_ALIGN;
  const int64_t row = static_cast<int64_t>(latent_dim) + rope_dim;
  if (row / 8 > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
  if (kv_c_stride % 8 != 0 || k_pe_stride % 8 != 0 || block_stride % 8 != 0) return PA_ERR_ALIGN;
  if (num_tokens > 1 && (kv_c_stride < latent_dim || k_pe_stride < rope_dim))
    return PA_ERR_INVALID;
  if (num_blocks > 1 && block_stride < row * block_size) return PA_ERR_INVALID;
  if (!aligned(kv_c, 16) || !aligned(k_pe, 16) || !aligned(latent_cache, 16)) return PA_ERR_ALIGN;
  pa_detail::ReshapeArgs a{};
  a.key = kv_c;
  a.key2 = k_pe;
  a.key_stride = kv_c_stride;
  a.key2_stride = k_pe_stride;
  a.key_chunks = latent_dim / 8;
  a.key_cache = latent_cache;
  a.slot_mapping = slot_mapping;
  a.k_scale = scale;
  a.v_scale = scale;
  a.num_tokens = num_tokens;
  a.block_stride = block_stride;
  a.num_slots = num_blocks * block_size;
  a.row_chunks = static_cast<int32_t>(row / 8);
  a.block_size = block_size;
  return pa_detail::launch_reshape_and_cache(a, src_dtype, cache_dtype,
                                             reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_paged_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len,
                               int32_t num_sms, int32_t* num_splits_host,
                               int32_t* tokens_per_split_host) {
  if (num_splits_host == nullptr || tokens_per_split_host == nullptr) return PA_ERR_INVALID;
  if (num_seqs < 0 || num_kv_heads <= 0 || max_context_len < 0 || max_context_len > (1 << 30))
    return PA_ERR_INVALID;
  if (num_sms <= 0) num_sms = pa_detail::num_sms_current_device();
  const pa_detail::DecodePlan plan =
      pa_detail::make_decode_plan(num_seqs, num_kv_heads, max_context_len, num_sms);
  *num_splits_host = plan.num_splits;
  *tokens_per_split_host = plan.tokens_per_split;
  return PA_OK;
}

size_t pa_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_size,
                                      int32_t max_context_len) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
      max_context_len < 0 || max_context_len > (1 << 30))
    return 0;
  const pa_detail::DecodePlan plan = pa_detail::make_decode_plan(
      num_seqs, num_kv_heads, max_context_len, pa_detail::num_sms_current_device());
  return pa_detail::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size, plan);
}

pa_status pa_paged_decode_attention(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, pa_dtype cache_dtype,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_size, int32_t block_size,
                                    int32_t max_blocks_per_seq, int64_t num_blocks, float scale,
                                    int32_t max_context_len, void* workspace,
                                    size_t workspace_bytes, pa_stream_t stream) {
  pa_detail::DecodeArgs a{};
  const pa_status st = check_decode(out, q, k_cache, v_cache, cache_dtype, block_tables,
                                    context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                    block_size, max_blocks_per_seq, num_blocks, scale,
                                    max_context_len, &a);
  if (st != PA_OK) return st;
  const size_t need =
      pa_detail::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size, a.plan);
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
  a.workspace = workspace;
  a.error_word = nullptr;
  return pa_detail::launch_paged_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_paged_decode_attention_fp8(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const float* k_scale,
                                        const float* v_scale, const int32_t* block_tables,
                                        const int32_t* context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_size, int32_t block_size,
                                        int32_t max_blocks_per_seq, int64_t num_blocks,
                                        float scale, int32_t max_context_len, void* workspace,
                                        size_t workspace_bytes, pa_stream_t stream) {
  if ((k_scale == nullptr) != (v_scale == nullptr)) return PA_ERR_INVALID;
  pa_detail::DecodeArgs a{};
  const pa_status st = check_decode(out, q, k_cache, v_cache, PA_FP8_E4M3, block_tables,
                                    context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                    block_size, max_blocks_per_seq, num_blocks, scale,
                                    max_context_len, &a);
  if (st != PA_OK) return st;
  const size_t need =
      pa_detail::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size, a.plan);
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
  a.workspace = workspace;
  a.error_word = nullptr;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return pa_detail::launch_paged_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_paged_decode_step(void* out, const void* q, const void* new_k, const void* new_v,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               pa_dtype cache_dtype, const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_size, int32_t block_size, int32_t max_blocks_per_seq,
                               int64_t num_blocks, float scale, int32_t max_context_len,
                               void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if ((k_scale == nullptr) != (v_scale == nullptr)) return PA_ERR_INVALID;
  if (k_scale != nullptr && cache_dtype != PA_FP8_E4M3) return PA_ERR_INVALID;
  pa_detail::DecodeArgs a{};
  const pa_status st = check_decode(out, q, k_cache, v_cache, cache_dtype, block_tables,
                                    context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                    block_size, max_blocks_per_seq, num_blocks, scale,
                                    max_context_len, &a);
  if (st != PA_OK) return st;
  if (num_seqs > 0 && (new_k == nullptr || new_v == nullptr || slot_mapping == nullptr))
    return PA_ERR_INVALID;
  if (!aligned(new_k, 16) || !aligned(new_v, 16)) return PA_ERR_ALIGN;
  const size_t need =
      pa_detail::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size, a.plan);
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
  a.workspace = workspace;
  a.error_word = nullptr;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.new_k = new_k;
  a.new_v = new_v;
  a.slot_mapping = slot_mapping;
  return pa_detail::launch_paged_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_paged_prefill_attention(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, pa_dtype cache_dtype,
                                     const int32_t* block_tables, const int32_t* cu_seqlens_q,
                                     const int32_t* context_lens, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int32_t max_blocks_per_seq,
                                     int64_t num_blocks, float scale, int32_t max_q_len,
                                     unsigned* error_word, pa_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_q_len < 0)
    return PA_ERR_INVALID;
  if (num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (out == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr ||
      block_tables == nullptr || cu_seqlens_q == nullptr || context_lens == nullptr ||
      error_word == nullptr)
    return PA_ERR_INVALID;
  if (num_q_heads % num_kv_heads != 0 || !std::isfinite(scale)) return PA_ERR_INVALID;
  if (cache_dtype != PA_BF16 || head_size != 128) return PA_ERR_UNSUPPORTED;
  const int32_t G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return PA_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)) != 0)
    return PA_ERR_UNSUPPORTED;
  if (num_blocks * block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(error_word, 4))
    return PA_ERR_ALIGN;
  pa_detail::PrefillArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.cu_seqlens_q = cu_seqlens_q;
  a.context_lens = context_lens;
  a.error_word = error_word;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.max_q_len = max_q_len;
  a.num_blocks = num_blocks;
  a.scale = scale;
  return pa_detail::launch_paged_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_paged_decode_attention_static(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, pa_dtype cache_dtype,
                                           const int32_t* block_tables,
                                           const int32_t* context_lens, int32_t num_seqs,
                                           int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_size, int32_t block_size,
                                           int32_t max_blocks_per_seq, int64_t num_blocks,
                                           float scale, int32_t max_context_len,
                                           unsigned* error_word, pa_stream_t stream) {
  pa_detail::DecodeArgs a{};
  const pa_status st = check_decode(out, q, k_cache, v_cache, cache_dtype, block_tables,
                                    context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                    block_size, max_blocks_per_seq, num_blocks, scale,
                                    max_context_len, &a);
  if (st != PA_OK) return st;
  if (error_word != nullptr && !aligned(error_word, 4)) return PA_ERR_ALIGN;
  const size_t need =
      pa_detail::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_size, a.plan);
  if (need > pa_detail::static_decode_scratch_bytes()) return PA_ERR_WORKSPACE;
  if (num_seqs == 0) return PA_OK;
  void* scratch = nullptr;
  const pa_status sst = pa_detail::static_decode_scratch_address(&scratch);
  if (sst != PA_OK) return sst;
  a.workspace = scratch;
  a.error_word = error_word;
  return pa_detail::launch_paged_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_mla_absorb_q(void* q_latent, const void* q_nope, const void* q_pe, const void* w_uk,
                          int32_t num_seqs, int32_t num_heads, int32_t nope_dim, int32_t rope_dim,
                          int32_t latent_dim, pa_stream_t stream) {
  if (num_seqs < 0 || num_heads <= 0 || nope_dim <= 0 || rope_dim < 0 || latent_dim <= 0)
    return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (q_latent == nullptr || q_nope == nullptr || w_uk == nullptr || (rope_dim > 0 && q_pe == nullptr))
    return PA_ERR_INVALID;
  if (nope_dim % 64 != 0 || latent_dim % 64 != 0 || rope_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_heads) * nope_dim >= (1ll << 31) / 2) return PA_ERR_UNSUPPORTED;
  if (!aligned(q_latent, 16) || !aligned(q_nope, 16) || !aligned(w_uk, 16) ||
      (q_pe != nullptr && !aligned(q_pe, 16)))
    return PA_ERR_ALIGN;
  return pa_detail::launch_mla_absorb_q(q_latent, q_nope, rope_dim > 0 ? q_pe : nullptr, w_uk,
                                        num_seqs, num_heads, nope_dim, rope_dim, latent_dim,
                                        reinterpret_cast<cudaStream_t>(stream));
}

size_t pa_mla_decode_workspace_size(int32_t num_seqs, int32_t num_heads,
                                    int32_t max_context_len) {
  if (num_seqs < 0 || num_heads <= 0 || num_heads % 16 != 0 || max_context_len < 0 ||
      max_context_len > (1 << 30))
    return 0;
  const pa_detail::DecodePlan plan = pa_detail::make_mla_plan(
      num_seqs, num_heads, max_context_len, pa_detail::num_sms_current_device());
  return pa_detail::mla_workspace_bytes(num_seqs, num_heads, plan);
}

pa_status pa_mla_decode_attention(void* out_latent, const void* q_latent,
                                  const void* latent_cache, const int32_t* block_tables,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_heads, int32_t latent_dim, int32_t rope_dim,
                                  int32_t block_size, int32_t max_blocks_per_seq,
                                  int64_t num_blocks, float scale, int32_t max_context_len,
                                  void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (num_seqs < 0 || num_heads <= 0 || latent_dim <= 0 || rope_dim < 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 ||
      max_context_len > (1 << 30))
    return PA_ERR_INVALID;
  if (out_latent == nullptr || q_latent == nullptr || latent_cache == nullptr ||
      block_tables == nullptr || context_lens == nullptr)
    return PA_ERR_INVALID;
  if (!std::isfinite(scale)) return PA_ERR_INVALID;
  if (latent_dim != 512 || rope_dim != 64 || num_heads % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)) != 0)
    return PA_ERR_UNSUPPORTED;
  if (num_blocks * block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_seqs) * num_heads >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
  if (!aligned(out_latent, 16) || !aligned(q_latent, 16) || !aligned(latent_cache, 16))
    return PA_ERR_ALIGN;
  pa_detail::MlaDecodeArgs a{};
  a.out_latent = out_latent;
  a.q_latent = q_latent;
  a.latent_cache = latent_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.plan = pa_detail::make_mla_plan(num_seqs, num_heads, max_context_len,
                                    pa_detail::num_sms_current_device());
  const size_t need = pa_detail::mla_workspace_bytes(num_seqs, num_heads, a.plan);
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
  a.workspace = workspace;
  return pa_detail::launch_mla_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_mla_project_out(void* out, const void* out_latent, const void* w_uv,
                             int32_t num_seqs, int32_t num_heads, int32_t latent_dim,
                             int32_t v_head_dim, pa_stream_t stream) {
  if (num_seqs < 0 || num_heads <= 0 || latent_dim <= 0 || v_head_dim <= 0) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (out == nullptr || out_latent == nullptr || w_uv == nullptr) return PA_ERR_INVALID;
  if (latent_dim % 64 != 0 || v_head_dim % 64 != 0) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_heads) * v_head_dim >= (1ll << 31) / 2) return PA_ERR_UNSUPPORTED;
  if (!aligned(out, 16) || !aligned(out_latent, 16) || !aligned(w_uv, 16)) return PA_ERR_ALIGN;
  return pa_detail::launch_mla_project_out(out, out_latent, w_uv, num_seqs, num_heads, latent_dim,
                                           v_head_dim, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
