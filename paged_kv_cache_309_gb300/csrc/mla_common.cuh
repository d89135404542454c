// mla_common.cuh -- pieces shared by the two MLA decode kernels (the
// mma.sync kernel in mla_decode.cu and the tcgen05 kernel in
// mla_decode_tc.cu): the latent row geometry, the kernel parameters and
// the tile loader.
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
  float* ws_lse;       // [H / HT, slots, HT] log2-sum-exp of the partial pieces
  float* ws_o;         // [H / HT, slots, HT, 512] (tcgen05: [.., slots, 2 halves, HT, 256])
  unsigned* counters;  // [B, H / HT] pieces counted (x 2 output halves for HT = 128)
  unsigned* err;
  int64_t num_blocks;
  int32_t num_heads;
  int32_t block_size;
  int32_t log2_bs;
  int32_t max_blocks_per_seq;
  int32_t num_splits;      // chunks (clusters) per head tile
  int32_t tokens_per_split;  // unused by the balanced schedules
  int32_t kv_evict_first;  // one head tile per sequence: nobody re-reads the rows
  int32_t num_seqs;
  int32_t num_slots;       // partial slots per head tile (2 per chunk)
  float scale_log2;
};

// swizzled address of 16-byte unit `unit` of row `row` in a [rows x 128 B] region
__device__ __forceinline__ uint32_t swz(uint32_t region, int row, int unit) {
  return region + static_cast<uint32_t>(row * 128 + ((unit ^ (row & 7)) << 4));
}

// Block id of piece `lane` of the tile starting at token tok0 (lane < nbox
// and inside the context), else -1: read ahead of the tile's issue so that
// the global-memory latency is not on the issuing warp's path.
__device__ __forceinline__ int mla_tile_bid(const MlaParams& p, const int32_t* bt, int tok0,
                                            int tok_end, int tile, int lane) {
  const int rpb = p.block_size < tile ? p.block_size : tile;
  const int first = tok0 + lane * rpb;
  return (lane < tile / rpb && first < tok_end) ? __ldg(bt + (first >> p.log2_bs)) : -1;
}

// Loads of one tile of `tile` tokens (called by one warp, all lanes): lane
// i < nbox holds the id of block piece i of the tile (mla_tile_bid), the
// lanes agree on the tile's row mask, lane 0 posts it and the byte count on
// `full`, and each lane with a valid piece loads its rows into `stage`
// (chunk c at stage + c * chunk_bytes, rows of 128 bytes).  When a block
// covers the whole tile (one piece), tm_kv is a 3-D map {64 elements, rows,
// 9 chunks} and one TMA instruction brings all nine chunks in that layout;
// otherwise tm_kv is 2-D and each piece takes one box per chunk.  (A TMA
// instruction costs its issuing warp ~180 cycles here, so nine per tile kept
// the issuing warp of the mma.sync kernel ~1.6 K cycles from its own work.)
__device__ __forceinline__ void mla_issue_tile_at(const MlaParams& p, const CUtensorMap* tm_kv,
                                                  uint8_t* stage, int chunk_bytes, int tile,
                                                  uint64_t* full, uint64_t* mask_slot,
                                                  int lane_bid, int tok0, int tok_end,
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
      bid = lane_bid;
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
    if (nbox == 1) {
      tma_load_3d(st, tm_kv, 0, row, 0, full, pol);
    } else {
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c)
        tma_load_2d(st + c * chunk_bytes, tm_kv, 64 * c, row, full, pol);
    }
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
