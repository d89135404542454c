// cache_write.cu -- reshape_and_cache: scatter per-token K/V rows into the
// paged cache through slot_mapping (optional SWA remap, optional scale, cast).
//
// Follows sglang cache_ops.py, reshape_and_cache_flash ("slot mapping",
// "optional scale", "target layout" blocks) and the nano-vLLM walkthrough,
// section 2.6 (store_kvcache_kernel).  Both pages run one program per
// (token, head block) over a [HEAD_BLOCK, BLOCK_D] tile.  Here one warp owns
// a (token, chunk group): a token's H*d elements are contiguous in the
// source row AND in the destination slot row ([bs, H, d] inside a block),
// so the whole row moves as 16-byte chunks of 8 elements, 32 lanes side by
// side (fully coalesced), up to 4 chunks of K and 4 of V in flight per lane.
// The slot is resolved by every lane from the same address (a broadcast), so
// a skipped token exits the whole warp at once: no divergence.
// The two-source form (kTwoSrc, pa_concat_and_cache_mla) reads the first
// key_chunks chunks of each row from `key` and the rest from `key2`, which
// assembles an MLA latent row [c_kv | k_pe] and stores it in the same pass.
#include <type_traits>

#include "pa_internal.cuh"

namespace pa_detail {
namespace {

constexpr int kWarps = 8;            // warps per CTA
constexpr int kChunksPerLane = 4;    // chunks of 8 elements per lane per tensor
constexpr int kChunksPerWarp = 32 * kChunksPerLane;
constexpr int kTwoSrcRowsPerWarp = 2;
constexpr int kTwoSrcSlotsPerLane = 5;  // 160 chunks: two rows of up to 80 chunks (the
                                        // 576-element MLA latent row is 72)

// Writes token t's row to slot s (already resolved and in the pool): the
// lane's chunks c_begin, c_begin + 32, ... of the row's chunk group.
template <typename S, typename D, bool kRaw, bool kTwoSrc>
__device__ __forceinline__ void write_row(const ReshapeArgs& a, int64_t t, int64_t s, int grp,
                                          int lane) {
  using namespace pa;
  const int64_t blk = (a.block_size & (a.block_size - 1)) == 0
                          ? s >> (__ffs(a.block_size) - 1)
                          : s / a.block_size;
  const int64_t off = s - blk * a.block_size;
  const int64_t row_elems = static_cast<int64_t>(a.row_chunks) * 8;
  const int64_t dst0 = blk * a.block_stride + off * row_elems;

  const S* ksrc = static_cast<const S*>(a.key) + t * a.key_stride;
  const S* vsrc = static_cast<const S*>(a.value) + t * a.value_stride;
  // two-source rows: chunk c >= key_chunks comes from key2 (chunk c - key_chunks)
  const S* k2src = kTwoSrc ? static_cast<const S*>(a.key2) + t * a.key2_stride -
                                 8 * static_cast<int64_t>(a.key_chunks)
                           : nullptr;
  D* kdst = static_cast<D*>(a.key_cache) + dst0;
  D* vdst = static_cast<D*>(a.value_cache) + dst0;
  const bool has_v = a.value != nullptr;
  const int c_begin = grp * kChunksPerWarp + lane;

  Vec8<S> kv[kChunksPerLane], vv[kChunksPerLane];
#pragma unroll
  for (int i = 0; i < kChunksPerLane; ++i) {
    const int c = c_begin + 32 * i;
    if (c < a.row_chunks) {
      kv[i] = load8((kTwoSrc && c >= a.key_chunks ? k2src : ksrc) + 8 * c);
      if (has_v) vv[i] = load8(vsrc + 8 * c);
    }
  }
  if constexpr (kRaw) {
#pragma unroll
    for (int i = 0; i < kChunksPerLane; ++i) {
      const int c = c_begin + 32 * i;
      if (c < a.row_chunks) {
        store8(kdst + 8 * c, kv[i]);
        if (has_v) store8(vdst + 8 * c, vv[i]);
      }
    }
  } else {
    const bool scaled = a.k_scale != nullptr;
    const Divisor ks = make_divisor(scaled ? __ldg(a.k_scale) : 1.0f);
    const Divisor vs = make_divisor(scaled ? __ldg(a.v_scale) : 1.0f);
    constexpr bool kToE4m3 = std::is_same<D, e4m3>::value;
    // largest |x| whose product with r = 1/s stays below FLT_MAX (finite,
    // so that infinities take the library path)
    const float kxmax = fminf(1.7e38f * ks.s, 3.0e38f), vxmax = fminf(1.7e38f * vs.s, 3.0e38f);
#pragma unroll
    for (int i = 0; i < kChunksPerLane; ++i) {
      const int c = c_begin + 32 * i;
      if (c < a.row_chunks) {
        float f[8];
        if (kToE4m3 && scaled) {
          div8_for_e4m3(kv[i], f, ks, kxmax);
        } else {
          to_f32(kv[i], f);
          if (scaled) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = div_rn(f[e], ks);  // IEEE quotient
          }
        }
        store8(kdst + 8 * c, from_f32<D>(f));
        if (has_v) {
          if (kToE4m3 && scaled) {
            div8_for_e4m3(vv[i], f, vs, vxmax);
          } else {
            to_f32(vv[i], f);
            if (scaled) {
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = div_rn(f[e], vs);
            }
          }
          store8(vdst + 8 * c, from_f32<D>(f));
        }
      }
    }
  }
}

// Two-source rows (K only, rows of at most 128 chunks), kRows tokens per
// warp: chunk c of the warp's kRows * row_chunks is chunk c % row_chunks of
// row c / row_chunks; every load of the rows is issued before the first
// store, so a warp keeps kRows rows in flight (the MLA latent row is 72
// chunks, which one warp alone covers with 2.25 chunks per lane).  s[r] < 0:
// row r is skipped.
// s[r] for a row index known only at run time, by selects (no local-memory array)
template <int kRows>
__device__ __forceinline__ int64_t pick_row(const int64_t (&s)[kRows], int r) {
  int64_t v = -1;
#pragma unroll
  for (int i = 0; i < kRows; ++i) v = r == i ? s[i] : v;
  return v;
}

template <typename S, typename D, bool kRaw, int kRows>
__device__ __forceinline__ void write_rows_two_src(const ReshapeArgs& a, int64_t t0,
                                                   const int64_t (&s)[kRows], int lane) {
  using namespace pa;
  constexpr int kMax = kTwoSrcSlotsPerLane;  // chunks per lane (kRows rows fit 32 * kMax)
  const int rc = a.row_chunks;
  Vec8<S> x[kMax];
#pragma unroll
  for (int i = 0; i < kMax; ++i) {
    const int c = lane + 32 * i;
    const int r = c / rc, cc = c - (c / rc) * rc;
    if (r < kRows && pick_row(s, r) >= 0) {
      const int64_t t = t0 + r;
      const S* src = cc < a.key_chunks
                         ? static_cast<const S*>(a.key) + t * a.key_stride + 8 * cc
                         : static_cast<const S*>(a.key2) + t * a.key2_stride +
                               8 * (cc - a.key_chunks);
      x[i] = load8(src);
    }
  }
  const bool scaled = a.k_scale != nullptr;
  const Divisor ks = make_divisor(!kRaw && scaled ? __ldg(a.k_scale) : 1.0f);
  const float kxmax = fminf(1.7e38f * ks.s, 3.0e38f);
  constexpr bool kToE4m3 = std::is_same<D, e4m3>::value;
#pragma unroll
  for (int i = 0; i < kMax; ++i) {
    const int c = lane + 32 * i;
    const int r = c / rc, cc = c - (c / rc) * rc;
    const int64_t sr = pick_row(s, r);
    if (r < kRows && sr >= 0) {
      const int64_t blk = (a.block_size & (a.block_size - 1)) == 0
                              ? sr >> (__ffs(a.block_size) - 1)
                              : sr / a.block_size;
      const int64_t off = sr - blk * a.block_size;
      D* dst = static_cast<D*>(a.key_cache) + blk * a.block_stride +
               off * static_cast<int64_t>(rc) * 8 + 8 * cc;
      if constexpr (kRaw) {
        store8(dst, x[i]);
      } else {
        float f[8];
        if (kToE4m3 && scaled) {
          div8_for_e4m3(x[i], f, ks, kxmax);
        } else {
          to_f32(x[i], f);
          if (scaled) {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = div_rn(f[e], ks);  // IEEE quotient
          }
        }
        store8(dst, from_f32<D>(f));
      }
    }
  }
}

// kTPW = 1: one warp per (token, chunk group); every lane resolves the slot
// from the same address (a broadcast), so a skipped token exits the warp.
// kTPW = 8 (a second-stage SWA table, rows of one chunk group): lanes 0-7
// resolve eight tokens' slots and table entries side by side, then the warp
// writes the rows that survived one after another.  Under a sliding window
// most tokens fall out of the window; batching their two dependent index
// loads keeps the grid to one wave instead of paying both loads per token.
// Warp w takes tokens w, w + NW, w + 2 NW, ... (NW warps in the grid), so a
// window of consecutive surviving tokens spreads over all warps (about one
// row each) instead of queueing eight rows on a few warps.
template <typename S, typename D, bool kRaw, bool kTwoSrc, int kTPW>
__global__ void __launch_bounds__(kWarps * 32, 4) reshape_and_cache_kernel(ReshapeArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if constexpr (kTwoSrc && kTPW > 1) {
    // kTPW two-source rows per warp (rows of one chunk group, no SWA table)
    const int64_t t0 = wid * kTPW;
    if (t0 >= a.num_tokens) return;
    int64_t s[kTPW];
#pragma unroll
    for (int r = 0; r < kTPW; ++r) {
      s[r] = t0 + r < a.num_tokens ? __ldg(a.slot_mapping + t0 + r) : -1;
      if (s[r] >= a.num_slots) s[r] = -1;
    }
    write_rows_two_src<S, D, kRaw, kTPW>(a, t0, s, lane);
  } else if constexpr (kTPW == 1) {
    const int64_t t = a.groups == 1 ? wid : wid / a.groups;  // a 64-bit division is long
    const int grp = static_cast<int>(wid - t * a.groups);
    if (t >= a.num_tokens) return;
    // slot resolution (same value in every lane)
    int64_t s = __ldg(a.slot_mapping + t);
    if (s < 0) return;
    if (a.swa != nullptr) {
      if (s >= a.swa_len) return;
      s = __ldg(a.swa + s);
      if (s < 0) return;
    }
    if (s >= a.num_slots) return;
    write_row<S, D, kRaw, kTwoSrc>(a, t, s, grp, lane);
  } else {
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
    if (wid >= a.num_tokens) return;
    int64_t s = -1;
    const int64_t tl = wid + lane * nw;  // lane j < kTPW resolves token wid + j * NW
    if (lane < kTPW && tl < a.num_tokens) {
      s = __ldg(a.slot_mapping + tl);
      if (s >= 0 && a.swa != nullptr) s = s < a.swa_len ? __ldg(a.swa + s) : -1;
      if (s >= a.num_slots) s = -1;
    }
    uint32_t valid = __ballot_sync(0xffffffffu, s >= 0);
    while (valid != 0u) {
      const int j = __ffs(valid) - 1;
      valid &= valid - 1u;
      write_row<S, D, kRaw, kTwoSrc>(a, wid + j * nw, __shfl_sync(0xffffffffu, s, j), 0, lane);
    }
  }
}

constexpr int kSwaTokensPerWarp = 8;

template <typename S, typename D>
pa_status launch_typed(ReshapeArgs a, cudaStream_t stream) {
  a.groups = (a.row_chunks + kChunksPerWarp - 1) / kChunksPerWarp;
  const bool batched = a.swa != nullptr && a.groups == 1 && a.key2 == nullptr;
  // (32-bit sources keep one row per warp: two rows of them do not fit the registers)
  const bool paired = sizeof(S) == 2 && a.key2 != nullptr && a.swa == nullptr &&
                      kTwoSrcRowsPerWarp * a.row_chunks <= 32 * kTwoSrcSlotsPerLane;
  const int64_t warps = batched ? (a.num_tokens + kSwaTokensPerWarp - 1) / kSwaTokensPerWarp
                        : paired ? (a.num_tokens + kTwoSrcRowsPerWarp - 1) / kTwoSrcRowsPerWarp
                                 : a.num_tokens * a.groups;
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  if (blocks == 0) return PA_OK;
  if (blocks > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
  const bool raw = std::is_same<S, D>::value && a.k_scale == nullptr;
  const unsigned grid = static_cast<unsigned>(blocks);
  if (paired) {
    if constexpr (sizeof(S) == 2) {
      if (raw) {
        if constexpr (std::is_same<S, D>::value)
          reshape_and_cache_kernel<S, D, true, true, kTwoSrcRowsPerWarp>
              <<<grid, kWarps * 32, 0, stream>>>(a);
      } else {
        reshape_and_cache_kernel<S, D, false, true, kTwoSrcRowsPerWarp>
            <<<grid, kWarps * 32, 0, stream>>>(a);
      }
    }
  } else if (a.key2 != nullptr) {
    if (raw) {
      if constexpr (std::is_same<S, D>::value)
        reshape_and_cache_kernel<S, D, true, true, 1><<<grid, kWarps * 32, 0, stream>>>(a);
    } else {
      reshape_and_cache_kernel<S, D, false, true, 1><<<grid, kWarps * 32, 0, stream>>>(a);
    }
  } else if (batched) {
    if (raw) {
      if constexpr (std::is_same<S, D>::value)
        reshape_and_cache_kernel<S, D, true, false, kSwaTokensPerWarp>
            <<<grid, kWarps * 32, 0, stream>>>(a);
    } else {
      reshape_and_cache_kernel<S, D, false, false, kSwaTokensPerWarp>
          <<<grid, kWarps * 32, 0, stream>>>(a);
    }
  } else if (raw) {
    if constexpr (std::is_same<S, D>::value)
      reshape_and_cache_kernel<S, D, true, false, 1><<<grid, kWarps * 32, 0, stream>>>(a);
  } else {
    reshape_and_cache_kernel<S, D, false, false, 1><<<grid, kWarps * 32, 0, stream>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename S>
pa_status launch_src(const ReshapeArgs& a, pa_dtype dst, cudaStream_t stream) {
  switch (dst) {
    case PA_BF16: return launch_typed<S, pa::bf16>(a, stream);
    case PA_FP16: return launch_typed<S, pa::f16>(a, stream);
    case PA_FP32: return launch_typed<S, float>(a, stream);
    case PA_FP8_E4M3: return launch_typed<S, pa::e4m3>(a, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

}  // namespace

pa_status launch_reshape_and_cache(const ReshapeArgs& a, pa_dtype src, pa_dtype dst,
                                   cudaStream_t stream) {
  switch (src) {
    case PA_BF16: return launch_src<pa::bf16>(a, dst, stream);
    case PA_FP16: return launch_src<pa::f16>(a, dst, stream);
    case PA_FP32: return launch_src<float>(a, dst, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace pa_detail
