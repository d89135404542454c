// mla_common.cuh -- pieces shared by the two MLA decode kernels (the
// mma.sync kernel in mla_decode.cu and the tcgen05 kernel in
// mla_decode_tc.cu): the latent row geometry, the kernel parameters, the
// context clipping, the tile loader and the split merge.
#pragma once

#include <cudaTypedefs.h>

#include "pa_internal.cuh"

namespace pa_detail {
namespace mla {

using namespace pa;

constexpr int kLat = 512;                 // latent elements (the value part)
constexpr int kRope = 64;                 // rope elements
constexpr int kRow = kLat + kRope;        // 576 elements per cache row
constexpr int kRowBytes = kRow * 2;       // 1152 bytes
constexpr int kChunks = kRow / 64;        // nine 64-element (128-byte) chunks
constexpr float kRescaleLog2 = 8.0f;    // lazy-rescale threshold (base-2 units)
constexpr size_t kWorkspaceHeader = 256;

struct MlaParams {
  __nv_bfloat16* out;  // [B, H, 512]
  const __nv_bfloat16* q_latent;  // [B, H, 576]
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_lse;       // [B, H, splits]
  float* ws_o;         // [B, H, splits, 512]
  unsigned* counters;  // [B, H / HT]
  unsigned* err;
  int64_t num_blocks;
  int32_t num_heads;
  int32_t block_size;
  int32_t log2_bs;
  int32_t max_blocks_per_seq;
  int32_t num_splits;
  int32_t tokens_per_split;
  int32_t kv_evict_first;  // one head tile per sequence: nobody re-reads the rows
  int32_t num_seqs;
  int32_t num_slots;       // tcgen05 kernel: partial slots per head tile (2 per cluster)
  float scale_log2;
};

__device__ __forceinline__ int mla_effective_len(const MlaParams& p, int b, bool* clipped) {
  int L = __ldg(p.context_lens + b);
  L = L < 0 ? 0 : L;
  const int64_t cap = min(static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size,
                          static_cast<int64_t>(p.num_splits) * p.tokens_per_split);
  *clipped = static_cast<int64_t>(L) > cap;
  return *clipped ? static_cast<int>(cap) : L;
}

// swizzled address of 16-byte unit `unit` of row `row` in a [rows x 128 B] region
__device__ __forceinline__ uint32_t swz(uint32_t region, int row, int unit) {
  return region + static_cast<uint32_t>(row * 128 + ((unit ^ (row & 7)) << 4));
}

// Merge of one (sequence, head) row by one warp over n splits: weights
// 2^(lse_s - max), out = sum_s w_s o_s / sum_s w_s in bf16.  Lane owns
// elements 4*lane + 128*i, i = 0..3.
__device__ __forceinline__ void mla_merge_warp(const MlaParams& p, int64_t bh, int n, int lane) {
  const float* lse = p.ws_lse + bh * p.num_splits;
  const float* o = p.ws_o + bh * p.num_splits * kLat;
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, __ldcg(lse + s));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float4 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      const int my = s0 + lane;
      const float wl = my < n ? exp2f(__ldcg(lse + my) - M) : 0.f;
      const int cnt = min(32, n - s0);
      for (int k = 0; k < cnt; ++k) {
        const float w = __shfl_sync(0xffffffffu, wl, k);
        const float4* src = reinterpret_cast<const float4*>(o + static_cast<int64_t>(s0 + k) * kLat);
        W += w;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = __ldcg(src + lane + 32 * i);
          acc[i].x += w * v.x;
          acc[i].y += w * v.y;
          acc[i].z += w * v.z;
          acc[i].w += w * v.w;
        }
      }
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<uint2*>(p.out + bh * kLat + 4 * lane + 128 * i) =
        make_uint2(pack_bf16x2(acc[i].x * inv, acc[i].y * inv),
                   pack_bf16x2(acc[i].z * inv, acc[i].w * inv));
}

// Merge of `nheads` (sequence, head) rows bh0 .. bh0 + nheads - 1 over n
// splits by the whole CTA: weights w_s = 2^(lse_s - max) per head go to
// shared memory `wsm` (nheads * n floats) once, then every thread owns
// independent 4-element columns and sums its n partials with independent
// loads (a warp per head would walk the splits one L2 round trip at a
// time).  out = sum_s w_s o_s / sum_s w_s, in bf16.
__device__ __forceinline__ void mla_merge_cta(const MlaParams& p, int64_t bh0, int nheads, int n,
                                              float* wsm) {
  for (int h = threadIdx.x; h < nheads; h += blockDim.x) {
    const float* lse = p.ws_lse + (bh0 + h) * p.num_splits;
    float M = -INFINITY;
    for (int s = 0; s < n; ++s) M = fmaxf(M, __ldcg(lse + s));
    float W = 0.f;
    for (int s = 0; s < n; ++s) {
      const float w = M == -INFINITY ? 0.f : exp2f(__ldcg(lse + s) - M);
      wsm[h * n + s] = w;
      W += w;
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    for (int s = 0; s < n; ++s) wsm[h * n + s] *= inv;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nheads * (kLat / 4); idx += blockDim.x) {
    const int h = idx / (kLat / 4), e4 = idx % (kLat / 4);
    const float4* src =
        reinterpret_cast<const float4*>(p.ws_o + (bh0 + h) * p.num_splits * kLat) + e4;
    const float* w = wsm + h * n;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 4 <= n; s += 4) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = __ldcg(src + (s + u) * (kLat / 4));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float ww = w[s + u];
        acc.x += ww * x[u].x;
        acc.y += ww * x[u].y;
        acc.z += ww * x[u].z;
        acc.w += ww * x[u].w;
      }
    }
    for (; s < n; ++s) {
      const float4 x = __ldcg(src + s * (kLat / 4));
      const float ww = w[s];
      acc.x += ww * x.x;
      acc.y += ww * x.y;
      acc.z += ww * x.z;
      acc.w += ww * x.w;
    }
    *reinterpret_cast<uint2*>(p.out + (bh0 + h) * kLat + 4 * e4) =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

// Loads of one tile of `tile` tokens (called by one warp, all lanes): lane
// i < nbox looks up block piece i of the tile, the lanes agree on the tile's
// row mask, lane 0 posts it and the byte count on `full`, and each lane with
// a valid piece issues one TMA box per 64-element chunk into `stage`
// (chunk c at stage + c * chunk_bytes, rows of 128 bytes).
__device__ __forceinline__ void mla_issue_tile_at(const MlaParams& p, const CUtensorMap* tm_kv,
                                                  uint8_t* stage, int chunk_bytes, int tile,
                                                  uint64_t* full, uint64_t* mask_slot,
                                                  const int32_t* bt, int tok0, int tok_end,
                                                  uint64_t pol, int lane) {
  const int bs = p.block_size;
  const int rpb = bs < tile ? bs : tile;
  const int nbox = tile / rpb;
  const int nval = min(tile, tok_end - tok0);
  bool valid = false;
  int rows = 0, bid = -1, row0 = 0;
  if (lane < nbox) {
    const int first = tok0 + lane * rpb;
    rows = min(rpb, nval - lane * rpb);
    if (rows > 0) {
      row0 = first & (bs - 1);
      bid = __ldg(bt + (first >> p.log2_bs));
      valid = bid >= 0 && static_cast<int64_t>(bid) < p.num_blocks;
    }
  }
  uint64_t bits = 0;
  if (valid) bits = (rows >= 64 ? ~0ull : ((1ull << rows) - 1ull)) << (lane * rpb);
  const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits));
  const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits >> 32));
  const uint32_t vb = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) {
    *mask_slot = (static_cast<uint64_t>(hi) << 32) | lo;
    mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(vb) * rpb * kRowBytes));
  }
  __syncwarp();
  if (valid) {
    const int32_t row = bid * bs + row0;
    uint8_t* st = stage + lane * rpb * 128;
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c)
      tma_load_2d(st + c * chunk_bytes, tm_kv, 64 * c, row, full, pol);
  }
}

}  // namespace mla

// The tcgen05 kernel (mla_decode_tc.cu): 128-head tiles, each served by a
// cluster of two CTAs that own one half of the 512 output elements each,
// clusters spread over a token-balanced list of the sequences' tiles.
// grid = (2 * clusters, H / 128).  mrope maps the 32 rope elements of a row
// one CTA uses (64-byte boxes), mkv the latent chunks (128-byte boxes).
pa_status launch_mla_tc(const CUtensorMap& mrope, const CUtensorMap& mkv, const mla::MlaParams& p,
                        dim3 grid, cudaStream_t stream);
int mla_tc_tile();  // tokens per tile of the tcgen05 kernel

}  // namespace pa_detail
