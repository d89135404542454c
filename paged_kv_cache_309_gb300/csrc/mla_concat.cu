// mla_concat.cu -- MLA K assembly: k = [k_nope | k_rope broadcast over heads].
//
// Follows sglang cache_ops.py, concat_and_cast_mha_k_kernel: per token n and
// head h, k[n, h, :nope] = k_nope[n, h, :] and k[n, h, nope:] = k_rope[n, 0, :],
// cast to k's dtype.  The page runs one program per token over a
// [heads, dim] tile.  Here the output is treated as a stream of 16-byte
// chunks (8 elements): consecutive threads write consecutive chunks of k, so
// every store is coalesced; a chunk either comes from k_nope (coalesced in
// runs of nope/8 chunks) or from the token's single k_rope row, which all
// heads re-read from L1/L2.  Each thread keeps 4 chunks in flight.
#include <type_traits>

#include "pa_internal.cuh"

namespace pa_detail {
namespace {

constexpr int kChunksPerThread = 4;

template <typename S, typename D, bool kRaw>
__global__ void concat_mla_k_kernel(ConcatArgs a) {
  using namespace pa;
  const int64_t n = blockIdx.x;  // token
  const int cpr = a.nope_chunks + a.rope_chunks;  // chunks per head row
  const int total = a.num_heads * cpr;            // chunks per token
  const int c0 = blockIdx.y * (blockDim.x * kChunksPerThread) + threadIdx.x;

  const S* nope = static_cast<const S*>(a.k_nope) + n * a.nope_stride0;
  const S* rope = static_cast<const S*>(a.k_rope) + n * a.rope_stride0;
  D* kout = static_cast<D*>(a.k) + n * a.k_stride0;

  Vec8<S> v[kChunksPerThread];
  int64_t dst[kChunksPerThread];
#pragma unroll
  for (int i = 0; i < kChunksPerThread; ++i) {
    const int c = c0 + i * blockDim.x;
    dst[i] = -1;
    if (c < total) {
      const int h = c / cpr;
      const int j = c - h * cpr;
      const S* src = (j < a.nope_chunks) ? nope + h * a.nope_stride1 + 8 * j
                                         : rope + 8 * (j - a.nope_chunks);
      v[i] = load8(src);
      dst[i] = h * a.k_stride1 + 8 * j;
    }
  }
#pragma unroll
  for (int i = 0; i < kChunksPerThread; ++i) {
    if (dst[i] < 0) continue;
    if constexpr (kRaw) {
      store8(kout + dst[i], v[i]);
    } else {
      float f[8];
      to_f32(v[i], f);
      store8(kout + dst[i], from_f32<D>(f));
    }
  }
}

template <typename S, typename D>
pa_status launch_typed(const ConcatArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0) return PA_OK;
  if (a.num_tokens > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
  const int64_t total = static_cast<int64_t>(a.num_heads) * (a.nope_chunks + a.rope_chunks);
  if (total > 0x3FFFFFFFll) return PA_ERR_UNSUPPORTED;
  // threads: enough for one pass over a token's chunks, 32..256
  int64_t want = (total + kChunksPerThread - 1) / kChunksPerThread;
  int threads = static_cast<int>(want > 256 ? 256 : ((want + 31) / 32) * 32);
  const int64_t per_cta = static_cast<int64_t>(threads) * kChunksPerThread;
  const int64_t gy = (total + per_cta - 1) / per_cta;
  if (gy > 65535) return PA_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(a.num_tokens), static_cast<unsigned>(gy));
  if constexpr (std::is_same<S, D>::value)
    concat_mla_k_kernel<S, D, true><<<grid, threads, 0, stream>>>(a);
  else
    concat_mla_k_kernel<S, D, false><<<grid, threads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename S>
pa_status launch_src(const ConcatArgs& a, pa_dtype dst, cudaStream_t stream) {
  switch (dst) {
    case PA_BF16: return launch_typed<S, pa::bf16>(a, stream);
    case PA_FP16: return launch_typed<S, pa::f16>(a, stream);
    case PA_FP32: return launch_typed<S, float>(a, stream);
    case PA_FP8_E4M3: return launch_typed<S, pa::e4m3>(a, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

}  // namespace

pa_status launch_concat_mla_k(const ConcatArgs& a, pa_dtype src, pa_dtype dst,
                              cudaStream_t stream) {
  switch (src) {
    case PA_BF16: return launch_src<pa::bf16>(a, dst, stream);
    case PA_FP16: return launch_src<pa::f16>(a, dst, stream);
    case PA_FP32: return launch_src<float>(a, dst, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace pa_detail
