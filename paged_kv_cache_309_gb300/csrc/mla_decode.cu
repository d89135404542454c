// mla_decode.cu -- MLA decode attention over the paged latent cache.
//
// What is computed (PagedAttention-principle post, MLA section: a token's
// cache entry is its latent c_kv, K and V of head h are c_kv W_UK_h and
// c_kv W_UV_h, the rope part of K is carried beside the latent): with the
// two up-projections absorbed into the query and the output (done by
// mla_proj.cu), decode is one multi-query attention over the latent rows.
// For sequence b and head h:
//   s_j   = scale * q_lat[b, h, :] . row_j           (576 = 512 latent + 64 rope)
//   o_lat = sum_j softmax(s)_j * row_j[0:512]
// over the first context_lens[b] logical tokens, read through the block
// table (nano-vLLM walkthrough, section 2.6).  All heads read the same rows.
//
// Two kernels here (128-head tiles run on mla_decode_tc.cu): an mma.sync
// kernel for 64-head tiles and a tcgen05 kernel for 16-head tiles.  Both:
//  * grid = (head tile, chunk), one wave of resident CTAs per head tile.
//    Balanced schedule: the sequences' tiles laid end to end are cut into
//    one chunk of equal cost per CTA (each sequence start charged 2 tiles),
//    derived by every CTA from context_lens; a chunk that crosses sequences
//    runs as pieces (q_lat reloaded per piece, the pipeline's counters
//    running on across pieces).  Head tiles of one chunk are adjacent in the
//    launch order, so the second reads the latent rows from L2.
//  * rows come by TMA, 128-byte swizzled, in [rows x 128 B] chunk regions
//    (a 3-D box of several chunks when a block covers the tile, else one
//    box per block piece and chunk); a per-tile mask marks the rows that
//    exist, and rows that hold no token are zeroed before P . V reads them.
//  * epilogue per piece: a piece holding a whole sequence writes bf16 o_lat;
//    the others write fp32 partials + log2-sum-exp to the chunk's two slots
//    (a piece whose sequence began in an earlier chunk, one whose sequence
//    begins in this chunk) and count themselves per (sequence, head tile);
//    the CTA that completes a count merges that sequence after its own
//    pieces and zeroes the count.
// The mma.sync kernel (64 heads, 32-token tiles, three 72 KB stages, a
// ninth warp issuing the loads): eight warps compute S = Q . K^T
// (m16n8k16, heads on M, 16 heads x 16 tokens per warp) into a
// double-buffered fp32 score tile in shared memory, meet at one barrier,
// then each takes 16 heads x 256 output elements: an fp32 online softmax in
// base 2 with a lazy rescale (the running max moves only when a score beats
// it by more than 2^8) and O += P . V from the same stage.
// The tcgen05 kernel (16 heads, 64-token tiles) is described at its
// definition: tokens on M for both products, score units and value units
// in separate TMA rings.
//
// Every wait is bounded (2 s).  A timeout sets an error bit in the
// workspace's error word, drains the copies in flight and leaves.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>

#include "mla_common.cuh"
#include "tc_ops.cuh"

namespace pa_detail {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();  // decode.cu

namespace {

using namespace pa;
using namespace mla;

constexpr int kWarps = 8;                 // compute warps; warp kWarps issues the tile loads
constexpr int kComputeThreads = kWarps * 32;
constexpr int kThreads = kComputeThreads + 32;

// 64-head tiles (16-head tiles run on the tcgen05 kernel further down)
template <int HT>
struct MlaCfg {
  static_assert(HT == 64, "the mma.sync kernel serves 64-head tiles");
  static constexpr int kMB = HT / 16;                   // 16-head blocks
  static constexpr int kTile = 32;                      // tokens per stage
  static constexpr int kStages = 3;
  // registers per thread of the nine-warp block (measured on GB300: launches
  // at 168 and not at 200)
  static constexpr int kMaxRegs = 168;
  static constexpr int kWarpsPerMB = kWarps / kMB;      // 2
  // S: a 16-head block's warps split the tile's tokens into kTokGroups groups
  static constexpr int kTokGroups = kWarpsPerMB;
  static constexpr int kSTok = kTile / kTokGroups;      // tokens per warp in S: 16
  static constexpr int kDW = kLat / kWarpsPerMB;        // output elements per warp: 256
  static constexpr int kQBytes = kChunks * HT * 128;
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kStageBytes = kChunks * kChunkBytes;
  static constexpr int kSStride = kTile + 8;            // floats per score row
  static constexpr int kSBytes = HT * kSStride * 4;
  static constexpr int kStageOff = kQBytes;
  static constexpr int kSOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBarOff = kSOff + 2 * kSBytes;
  static constexpr int kBytes = kBarOff + (3 * kStages + 1) * 8 + 64;  // full, mask, q, empty, schedule
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory");
  static_assert(kSTok == 16, "S split");
};

template <int HT>
__device__ __forceinline__ void mla_issue_tile(const MlaParams& p, const CUtensorMap* tm_kv,
                                               uint8_t* smem, uint64_t* full, uint64_t* tile_mask,
                                               int lane_bid, int tok0, int tok_end, int stage,
                                               uint64_t pol, int lane) {
  using C = MlaCfg<HT>;
  mla_issue_tile_at(p, tm_kv, smem + C::kStageOff + stage * C::kStageBytes, C::kChunkBytes,
                    C::kTile, &full[stage], &tile_mask[stage], lane_bid, tok0, tok_end, pol,
                    lane);
}

// ------------------------------------------------------------- schedule --
// The work of one head tile is the sequences' kTile-token tiles laid end to
// end in sequence order (T tiles), cut into NC contiguous chunks, one per
// CTA (one wave of CTAs per head tile), of equal cost: tile t of sequence b
// sits at cost t + kPieceCost * (b + 1) (a piece's q_lat load and epilogue
// are charged to its sequence's start), the cost line of length T +
// kPieceCost * B is cut into min(NC, that) equal parts (each part spans a
// cost unit, so no chunk inside a sequence's span is empty), and a tile's
// chunk is floor(cost * parts / total) in closed form.  Where a chunk
// crosses a sequence boundary it splits into pieces.  A piece that covers
// its whole sequence writes bf16 output; the others write an fp32 partial
// to a slot: 2c for a piece whose sequence began in an earlier chunk, 2c + 1
// for one whose sequence begins in chunk c (at most one of each), and the
// CTA that completes a sequence's count merges it once its own work is
// done.  Every CTA derives the schedule from context_lens itself.
// kPC is the charge per sequence start in tiles: 2 (32-token tiles) for the
// mma.sync kernel, tok::kPieceCost (64-token tiles) for the tcgen05 kernel.
constexpr int kPieceCost = 2;  // tiles, the mma.sync kernel
template <int kPC>
__device__ __forceinline__ int bal_chunk(int64_t t, int b, int64_t total, int parts) {
  return static_cast<int>((t + static_cast<int64_t>(kPC) * (b + 1)) * parts / total);
}
__device__ __forceinline__ int bal_len(const MlaParams& p, int b, bool* clipped) {
  int L = __ldg(p.context_lens + b);
  L = L < 0 ? 0 : L;
  const int64_t cap = static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
  *clipped = static_cast<int64_t>(L) > cap;
  return *clipped ? static_cast<int>(cap) : L;
}
template <int kTile>
__device__ __forceinline__ int bal_tiles(const MlaParams& p, int b) {
  bool c;
  return (bal_len(p, b, &c) + kTile - 1) / kTile;
}
struct BalPiece {
  int b;       // sequence
  int tb, te;  // tile range [tb, te) of the sequence
  int pre;     // tiles of the sequences before b
  int n;       // tiles of the sequence
  bool first;  // the chunk's first piece
};
// Walks a chunk [g, g1) piece by piece.
template <int kTile>
struct BalIter {
  int b, pre, g, g1;
  bool started;
  __device__ __forceinline__ bool next(const MlaParams& p, BalPiece& pc) {
    if (g >= g1) return false;
    int n = bal_tiles<kTile>(p, b);
    while (pre + n <= g && b + 1 < p.num_seqs) {  // skips finished and empty sequences
      pre += n;
      ++b;
      n = bal_tiles<kTile>(p, b);
    }
    pc.b = b;
    pc.pre = pre;
    pc.n = n;
    pc.tb = g - pre;
    pc.te = min(n, g1 - pre);
    pc.first = !started;
    started = true;
    g = pre + pc.te;
    return true;
  }
};

// Merge of (sequence b, head tile ht) over its pieces by the whole CTA: the
// pieces are chunks c_first .. c_last, slot of the first 2 c_first + 1 (the
// sequence begins there), of the others 2c.  Per head, piece i
// gets weight 2^(lse_i - M) / sum_j 2^(lse_j - M); wsm holds HT * np
// weights.  The partials were written by other CTAs in this launch: read
// through L2 (__ldcg).
//
// kU 16-byte columns per thread and two pieces per round are in flight (the
// loads are L2 round trips; one column at a time left the merge latency-
// bound).  With kEarly, the first round's loads of the first two pieces go
// out before the weights are computed, so their latency overlaps the lse
// round (a block of 384 threads and kU = 6 covers 16 heads in one round).
template <int HT, int kPC, int kU = 4, bool kEarly = false>
__device__ __forceinline__ void merge_pieces_cta(const MlaParams& p, int b, int ht, int pre, int n,
                                                 int64_t total, int parts, float* wsm) {
  const int c_first = bal_chunk<kPC>(pre, b, total, parts);
  const int c_last = bal_chunk<kPC>(pre + n - 1, b, total, parts);
  const int np = c_last - c_first + 1;
  const int s0 = 2 * c_first + 1;
  auto slot = [&](int i) { return i == 0 ? s0 : 2 * (c_first + i); };
  const int64_t base = static_cast<int64_t>(ht) * p.num_slots;
  constexpr int kCols = HT * (kLat / 4);
  const int nthr = blockDim.x;
  auto part = [&](int i, int idx) {
    const int h = idx / (kLat / 4), e4 = idx % (kLat / 4);
    return __ldcg(reinterpret_cast<const float4*>(p.ws_o + ((base + slot(i)) * HT + h) * kLat) + e4);
  };
  // one or two pieces in one round: the loads go out first
  const bool early = kEarly && np <= 2 && kCols <= kU * nthr;
  float4 e0[kEarly ? kU : 1], e1[kEarly ? kU : 1];
  if (early) {
#pragma unroll
    for (int u = 0; u < (kEarly ? kU : 1); ++u) {
      const int idx = static_cast<int>(threadIdx.x) + u * nthr;
      e0[u] = e1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < kCols) {
        e0[u] = part(0, idx);
        if (np > 1) e1[u] = part(1, idx);
      }
    }
  }
  // every (head, piece) lse in one round of loads, then the weights per head
  for (int idx = threadIdx.x; idx < HT * np; idx += blockDim.x) {
    const int h = idx / np, i = idx - (idx / np) * np;
    wsm[idx] = __ldcg(p.ws_lse + (base + slot(i)) * HT + h);
  }
  __syncthreads();
  for (int h = threadIdx.x; h < HT; h += blockDim.x) {
    float* wh = wsm + h * np;
    float M = -INFINITY;
    for (int i = 0; i < np; ++i) M = fmaxf(M, wh[i]);
    float W = 0.f;
    for (int i = 0; i < np; ++i) {
      const float w = M == -INFINITY ? 0.f : exp2f(wh[i] - M);
      wh[i] = w;
      W += w;
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    for (int i = 0; i < np; ++i) wh[i] *= inv;
  }
  __syncthreads();
  const int64_t bh0 = static_cast<int64_t>(b) * p.num_heads + static_cast<int64_t>(ht) * HT;
  if (early) {
#pragma unroll
    for (int u = 0; u < (kEarly ? kU : 1); ++u) {
      const int idx = static_cast<int>(threadIdx.x) + u * nthr;
      if (idx < kCols) {
        const int h = idx / (kLat / 4), e4 = idx % (kLat / 4);
        const float w0 = wsm[h * np], w1 = np > 1 ? wsm[h * np + 1] : 0.f;
        *reinterpret_cast<uint2*>(p.out + (bh0 + h) * kLat + 4 * e4) =
            make_uint2(pack_bf16x2(w0 * e0[u].x + w1 * e1[u].x, w0 * e0[u].y + w1 * e1[u].y),
                       pack_bf16x2(w0 * e0[u].z + w1 * e1[u].z, w0 * e0[u].w + w1 * e1[u].w));
      }
    }
    __syncthreads();  // wsm is free again
    return;
  }
  for (int i0 = threadIdx.x; i0 < kCols; i0 += kU * nthr) {
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < np; i += 2) {
      const bool two = i + 1 < np;
      float4 x0[kU], x1[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = i0 + u * nthr;
        if (idx < kCols) {
          x0[u] = part(i, idx);
          x1[u] = two ? part(i + 1, idx) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int idx = i0 + u * nthr;
        if (idx < kCols) {
          const float* w = wsm + (idx / (kLat / 4)) * np;
          const float w0 = w[i], w1 = two ? w[i + 1] : 0.f;
          acc[u].x += w0 * x0[u].x + w1 * x1[u].x;
          acc[u].y += w0 * x0[u].y + w1 * x1[u].y;
          acc[u].z += w0 * x0[u].z + w1 * x1[u].z;
          acc[u].w += w0 * x0[u].w + w1 * x1[u].w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int idx = i0 + u * nthr;
      if (idx < kCols) {
        const int h = idx / (kLat / 4), e4 = idx % (kLat / 4);
        *reinterpret_cast<uint2*>(p.out + (bh0 + h) * kLat + 4 * e4) =
            make_uint2(pack_bf16x2(acc[u].x, acc[u].y), pack_bf16x2(acc[u].z, acc[u].w));
      }
    }
  }
  __syncthreads();  // wsm is free again
}

// Warp 0 of a CTA (all lanes): the schedule of chunk c of NC, written to
// sched[0] = T (the head tile's tiles), sched[2..3] = the chunk's tile range
// [g0, g1), sched[4..5] = the sequence of its first tile and the tiles before
// that sequence, sched[6] = 0 (merges recorded), sched[13] = 0 (abort flag).
template <int kTile, int kPC>
__device__ __forceinline__ void bal_schedule(const MlaParams& p, int c, int NC, bool report_clip,
                                             int* sched, int lane) {
  const int B = p.num_seqs;
  // tiles per sequence: up to 32 * kR sequences in registers (their loads
  // go out together, and the cuts below read no memory), more read again
  constexpr int kR = 4;
  const bool in_regs = B <= 32 * kR;
  int nreg[kR];
  int T = 0;
  bool any_clip = false;
  if (in_regs) {
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      nreg[r] = 0;
      if (32 * r + lane < B) {
        bool cl;
        nreg[r] = (bal_len(p, 32 * r + lane, &cl) + kTile - 1) / kTile;
        any_clip |= cl;
      }
    }
#pragma unroll
    for (int r = 0; r < kR; ++r)
      T += static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(nreg[r])));
  } else {
    for (int b0 = 0; b0 < B; b0 += 32) {
      int n = 0;
      if (b0 + lane < B) {
        bool cl;
        n = (bal_len(p, b0 + lane, &cl) + kTile - 1) / kTile;
        any_clip |= cl;
      }
      T += static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(n)));
    }
  }
  if (__any_sync(0xffffffffu, any_clip) && report_clip && lane == 0)
    atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
  // first tile of chunk k: the smallest t with cost(t) * parts >= k * total,
  // in the first non-empty sequence whose last tile reaches that cost (T
  // when none does); also that sequence and its first tile
  const int64_t total = static_cast<int64_t>(T) + static_cast<int64_t>(kPC) * B;
  const int parts = total < NC ? static_cast<int>(total) : NC;
  auto cut = [&](int k, int& bk, int& prek) -> int {
    if (k >= parts) return T;
    const int64_t x = (static_cast<int64_t>(k) * total + parts - 1) / parts;  // cost(t) >= x
    int pre = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int bb = b0 + lane;
      int n = 0;
      if (in_regs) {
#pragma unroll
        for (int r = 0; r < kR; ++r) n = 32 * r == b0 ? nreg[r] : n;  // selects, no local array
      } else {
        n = bb < B ? bal_tiles<kTile>(p, bb) : 0;
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int excl = incl - n;
      const int64_t last = static_cast<int64_t>(pre) + incl - 1 +
                           static_cast<int64_t>(kPC) * (bb + 1);
      const uint32_t hit = __ballot_sync(0xffffffffu, n > 0 && last >= x);
      if (hit) {
        const int l = __ffs(hit) - 1;
        bk = b0 + l;
        prek = pre + __shfl_sync(0xffffffffu, excl, l);
        const int64_t t = x - static_cast<int64_t>(kPC) * (bk + 1);
        return t > prek ? static_cast<int>(t) : prek;
      }
      pre += __shfl_sync(0xffffffffu, incl, 31);
    }
    return T;
  };
  int bfirst = 0, prefirst = 0, bnext = 0, prenext = 0;
  const int g0 = cut(c, bfirst, prefirst);
  const int g1 = cut(c + 1, bnext, prenext);
  if (lane == 0) {
    sched[0] = T;
    sched[1] = 0;
    sched[2] = g0;
    sched[3] = g1;
    sched[4] = bfirst;
    sched[5] = prefirst;
    sched[6] = 0;  // sequences this CTA merges
    sched[13] = 0;
  }
}

template <int HT>
__global__ void __maxnreg__(MlaCfg<HT>::kMaxRegs)
    mla_decode_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_kv, const MlaParams p) {
  using C = MlaCfg<HT>;
  constexpr int kTile = C::kTile;
  constexpr int kStages = C::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* tile_mask = full + kStages;
  uint64_t* qbar = tile_mask + kStages;
  uint64_t* empty = qbar + 1;                       // [kStages] every compute warp is done with a stage
  int* sched = reinterpret_cast<int*>(empty + kStages);  // [0..5] schedule, [6] merges, [7..12] their pieces, [13] abort
  volatile int* abort_flag = sched + 13;

  const int ht = blockIdx.x;
  const int c = blockIdx.y;    // chunk of the head tile's tile list
  const int NC = gridDim.y;    // chunks per head tile
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h0 = ht * HT;
  const int B = p.num_seqs;

  // ---- schedule (warp 0): total tiles, this CTA's chunk, its first sequence
  if (warp == 0) bal_schedule<kTile, kPieceCost>(p, c, NC, c == 0 && ht == 0, sched, lane);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init(qbar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const int g0 = sched[2], g1 = sched[3];
  const int64_t total = static_cast<int64_t>(sched[0]) + static_cast<int64_t>(kPieceCost) * B;
  const int parts = total < NC ? static_cast<int>(total) : NC;  // chunks with work
  const BalIter<kTile> it0{sched[4], sched[5], g0, g1, false};

  // sequences without tokens: zero output rows (chunk c takes b = c mod NC)
  for (int b = c; b < B; b += NC) {
    if (bal_tiles<kTile>(p, b) != 0) continue;
    for (int i = threadIdx.x; i < HT * (kLat / 8); i += blockDim.x) {
      const int h = i / (kLat / 8), e = i % (kLat / 8);
      reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * p.num_heads + h0 + h) *
                                           kLat)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (g0 >= g1) return;

  const uint32_t smem_base = smem_u32(smem);
  const uint64_t pol = p.kv_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
  const int ntotal = g1 - g0;  // tiles of this chunk

  // ---- the issuing side (warp kWarps): tile u of the chunk, across pieces,
  // into stage u % kStages once every compute warp has finished P.V of tile
  // u - kStages there (the stage's `empty` barrier).  The next tile is
  // prepared one issue ahead: its position, and its block ids read from the
  // table.  (Warp 0 used to issue between the CTA barrier and its own softmax,
  // ~1 K cycles per tile that every warp then waited for at the next barrier.)
  BalIter<kTile> iti = it0;
  BalPiece pci{};
  int tli = 0, Li = 0;
  const int32_t* bti = nullptr;
  int pre_tok0 = 0, pre_len = 0, pre_bid = -1;
  auto prepare_next = [&]() {  // issuing warp, all lanes
    if (tli >= pci.te || bti == nullptr) {
      if (!iti.next(p, pci)) return;
      tli = pci.tb;
      bool cl;
      Li = bal_len(p, pci.b, &cl);
      bti = p.block_tables + static_cast<int64_t>(pci.b) * p.max_blocks_per_seq;
    }
    pre_tok0 = tli * kTile;
    pre_len = Li;
    pre_bid = mla_tile_bid(p, bti, pre_tok0, Li, kTile, lane);
    ++tli;
  };
  auto issue_next = [&](int u) {  // issuing warp, all lanes: the prepared tile, then the next
    mla_issue_tile<HT>(p, &tm_kv, smem, full, tile_mask, pre_bid, pre_tok0, pre_len, u % kStages,
                       pol, lane);
    if (u + 1 < ntotal) prepare_next();
  };
  int issued = 0;
  if (warp == kWarps) {
    if (lane == 0) prefetch_tensormap(&tm_kv);
    prepare_next();
    bool pok = true;
    for (; issued < ntotal; ++issued) {
      if (issued >= kStages) {
        pok = __all_sync(0xffffffffu,
                         mbar_wait_bounded(&empty[issued % kStages],
                                           static_cast<uint32_t>(((issued / kStages) - 1) & 1),
                                           abort_flag));
        if (!pok) break;
      }
      issue_next(issued);
    }
    if (!pok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
  }

  const int gq = lane >> 2;  // mma groupID
  const int tq = lane & 3;   // thread in group
  const int mb = warp % C::kMB;  // this warp's 16-head block
  const int wi = warp / C::kMB;  // its index among that block's warps
  // lane-constant parts of the ldmatrix addresses
  const int qrow = 16 * mb + (lane & 15);  // Q: A operand rows
  const int qhalf = lane >> 4;             //    second 8 columns of a k-step
  const int tg = wi;  // S: token group
  const int krow = tg * 16 + (lane & 7) + ((lane >> 4) << 3);
  const int khalf = (lane >> 3) & 1;
  const int vrow_l = (lane & 7) + (((lane >> 3) & 1) << 3);  // V: token within the k-step
  const int vhalf = lane >> 4;                               //    second 8 elements
  float* s_tile = reinterpret_cast<float*>(smem + C::kSOff);

  bool ok = true;
  int u = 0;       // tiles of this chunk consumed
  int npiece = 0;  // pieces started (the parity of qbar)
  BalIter<kTile> itc = it0;
  BalPiece pc;
  while (warp < kWarps && itc.next(p, pc)) {  // the compute warps
    const int b = pc.b;
    const int64_t bh0 = static_cast<int64_t>(b) * p.num_heads + h0;
    const bool whole = pc.tb == 0 && pc.te == pc.n;
    const int slot = 2 * c + (pc.tb > 0 ? 0 : 1);
    float o[C::kDW / 8][4];
#pragma unroll
    for (int nt = 0; nt < C::kDW / 8; ++nt)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) o[nt][cc] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    if (ok) {
      // this piece's q_lat rows (every warp is done with the previous ones:
      // the last tile of a piece ends in a CTA barrier, the epilogue reads
      // registers only)
      if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(qbar, HT * kRowBytes);
        const uint64_t qpol = l2_policy_evict_normal();
        // one box: 9 chunks x HT rows x 128 bytes (chunk c at smem + c * HT * 128)
        tma_load_3d(smem, &tm_q, 0, b * p.num_heads + h0, 0, qbar, qpol);
      }
      // all warps agree on whether q_lat arrived (they meet at a barrier
      // every tile, so none may leave alone)
      ok = named_barrier_and(1, kComputeThreads, mbar_wait_bounded(qbar, npiece & 1, abort_flag));
    }
    ++npiece;
    for (int tl = pc.tb; tl < pc.te && ok; ++tl, ++u) {
      const int stage = u % kStages;
      const bool w_ok = mbar_wait_bounded(&full[stage], (u / kStages) & 1, abort_flag);
      const uint32_t st_base = smem_base + C::kStageOff + stage * C::kStageBytes;
      float* S = s_tile + (u & 1) * (HT * C::kSStride);
      uint64_t mask = 0;
      if (__all_sync(0xffffffffu, w_ok)) {
        mask = tile_mask[stage];
        // ---- S = Q . K^T for 16 heads x 16 tokens over the 576 elements
        constexpr int NTS = C::kSTok / 8;
        float sacc[NTS][4];
#pragma unroll
        for (int nt = 0; nt < NTS; ++nt)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) sacc[nt][cc] = 0.f;
        constexpr int kSteps = kChunks * 4;  // 16-wide k-steps
#pragma unroll 3
        for (int kc = 0; kc < kSteps; kc += 2) {
          const int ch = kc >> 2;
          const int j = kc & 3;  // k-steps j and j + 1 of chunk ch
          const uint32_t qreg = smem_base + ch * HT * 128;
          const uint32_t kreg = st_base + ch * C::kChunkBytes;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t a[4], bb[4];
            ldsm_x4(swz(qreg, qrow, 2 * (j + h2) + qhalf), a);
            ldsm_x4(swz(kreg, krow, 2 * (j + h2) + khalf), bb);
            mma_bf16_16816(sacc[0], a, bb[0], bb[1]);
            mma_bf16_16816(sacc[NTS - 1], a, bb[2], bb[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NTS; ++nt) {
          const int col = tg * C::kSTok + nt * 8 + 2 * tq;
          float* r0 = S + (16 * mb + gq) * C::kSStride + col;
          float* r1 = r0 + 8 * C::kSStride;
          *reinterpret_cast<float2*>(r0) = make_float2(sacc[nt][0], sacc[nt][1]);
          *reinterpret_cast<float2*>(r1) = make_float2(sacc[nt][2], sacc[nt][3]);
        }
        // rows of this warp's tokens that hold no token: zero their value
        // part (0 x NaN would poison P . V); their scores are masked below
        const uint32_t my_mask = static_cast<uint32_t>(mask >> (tg * C::kSTok)) &
                                 ((1u << C::kSTok) - 1u);
        if (my_mask != (1u << C::kSTok) - 1u) {
          uint8_t* st = smem + C::kStageOff + stage * C::kStageBytes;
          for (int idx = lane; idx < C::kSTok * 64; idx += 32) {
            const int rr = idx >> 6, unit = idx & 63;  // 64 units of 16 B = 512 elements
            if (!((my_mask >> rr) & 1u))
              *reinterpret_cast<uint4*>(st + (unit >> 3) * C::kChunkBytes +
                                        (tg * C::kSTok + rr) * 128 + ((unit & 7) << 4)) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // generic writes before the stage's next TMA fill
        }
      }
      // every warp's scores (and zeroed rows) are in place, and every warp
      // is done with tile u - 1: its stage takes tile u - 1 + kStages
      if (!named_barrier_and(1, kComputeThreads, w_ok)) {
        ok = false;
        break;
      }
      // ---- softmax over this warp's 16 heads, then O += P . V.  The score
      // tile is read twice (max, then weights) rather than held in registers.
      constexpr int KS = kTile / 16;
      // scaled, masked scores at the A-fragment positions of k-step kk:
      // rows gq (r = 0) and gq + 8 (r = 1), columns 2tq, 2tq+1, 2tq+8, 2tq+9
      auto load_scores = [&](int kk, int r, float (&x)[4]) {
        const float* row = S + (16 * mb + gq + 8 * r) * C::kSStride + 16 * kk + 2 * tq;
        const float2 x0 = *reinterpret_cast<const float2*>(row);
        const float2 x1 = *reinterpret_cast<const float2*>(row + 8);
        const uint32_t bits = static_cast<uint32_t>(mask >> (16 * kk + 2 * tq));
        x[0] = (bits & 1u) ? x0.x * p.scale_log2 : -INFINITY;
        x[1] = (bits & 2u) ? x0.y * p.scale_log2 : -INFINITY;
        x[2] = (bits & 0x100u) ? x1.x * p.scale_log2 : -INFINITY;
        x[3] = (bits & 0x200u) ? x1.y * p.scale_log2 : -INFINITY;
      };
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float x[4];
          load_scores(kk, r, x);
          mx[r] = fmaxf(mx[r], fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        if (mx[r] > m_run[r] + kRescaleLog2) {  // new running max (always on the first)
          const float corr = exp2f(m_run[r] - mx[r]);
          l_run[r] *= corr;
#pragma unroll
          for (int nt = 0; nt < C::kDW / 8; ++nt) {
            o[nt][2 * r] *= corr;
            o[nt][2 * r + 1] *= corr;
          }
          m_run[r] = mx[r];
        }
      }
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        float pv[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          load_scores(kk, r, pv[r]);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            // a masked score is -inf and m_run is finite once a token was seen
            pv[r][cc] = pv[r][cc] == -INFINITY ? 0.f : exp2f(pv[r][cc] - m_run[r]);
            l_run[r] += pv[r][cc];
          }
        }
        const uint32_t a[4] = {pack_bf16x2(pv[0][0], pv[0][1]), pack_bf16x2(pv[1][0], pv[1][1]),
                               pack_bf16x2(pv[0][2], pv[0][3]), pack_bf16x2(pv[1][2], pv[1][3])};
        const int vrow = 16 * kk + vrow_l;
#pragma unroll
        for (int np = 0; np < C::kDW / 16; ++np) {
          const int d = wi * C::kDW + 16 * np + 8 * vhalf;  // first element of this lane's unit
          uint32_t bv[4];
          ldsm_x4_trans(swz(st_base + (d >> 6) * C::kChunkBytes, vrow, (d & 63) >> 3), bv);
          mma_bf16_16816(o[2 * np], a, bv[0], bv[1]);
          mma_bf16_16816(o[2 * np + 1], a, bv[2], bv[3]);
        }
      }
      // this warp is done with the stage (its scores were read into
      // registers before the barrier's other side could rewrite them)
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }

    // ---- epilogue of the piece: rows 16mb + gq (+8), elements wi*kDW + 8nt + 2tq (+1)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int hh = 16 * mb + gq + 8 * r;
      // after a timeout the piece is empty: weight 0 in the merge, zero row if whole
      const float inv = ok && l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
      if (whole) {
        __nv_bfloat16* dst = p.out + (bh0 + hh) * kLat + wi * C::kDW + 2 * tq;
#pragma unroll
        for (int nt = 0; nt < C::kDW / 8; ++nt)
          *reinterpret_cast<uint32_t*>(dst + 8 * nt) =
              pack_bf16x2(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
      } else {
        const int64_t srow = (static_cast<int64_t>(ht) * p.num_slots + slot) * HT + hh;
        float* dst = p.ws_o + srow * kLat + wi * C::kDW + 2 * tq;
#pragma unroll
        for (int nt = 0; nt < C::kDW / 8; ++nt)
          *reinterpret_cast<float2*>(dst + 8 * nt) =
              make_float2(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
        if (wi == 0 && tq == 0)
          p.ws_lse[srow] = ok && l_run[r] > 0.f ? m_run[r] + log2f(l_run[r]) : -INFINITY;
      }
    }
    if (!whole) {
      // count the piece; the CTA that completes the sequence's count merges
      // it after its own work and returns the counter to zero
      named_barrier_and(1, kComputeThreads, true);  // every partial of this piece is written
      if (threadIdx.x == 0) {
        __threadfence();
        const int c_first = bal_chunk<kPieceCost>(pc.pre, b, total, parts);
        const int c_last = bal_chunk<kPieceCost>(pc.pre + pc.n - 1, b, total, parts);
        unsigned* ctr = p.counters + static_cast<int64_t>(b) * (p.num_heads / HT) + ht;
        const unsigned prev = atomicAdd(ctr, 1u);
        if (prev + 1u == static_cast<unsigned>(c_last - c_first + 1)) {
          atomicExch(ctr, 0u);
          __threadfence();
          const int k = sched[6]++;
          sched[7 + 3 * k] = b;
          sched[8 + 3 * k] = pc.pre;
          sched[9 + 3 * k] = pc.n;
        }
      }
    }
  }

  if (!ok && threadIdx.x == 0) {
    // stop the issuing warp, and wait (bounded) for the q_lat copy in flight
    *abort_flag = 1;
    atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    mbar_wait_bounded(qbar, (npiece - 1) & 1, nullptr);
  }
  __syncthreads();
  if (*abort_flag) {
    // the tiles issued but not consumed (at most the last kStages) land
    // before the shared memory is reused or released
    if (warp == kWarps && lane == 0)
      for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
        mbar_wait_bounded(&full[t % kStages], (t / kStages) & 1, nullptr);
    __syncthreads();
  }
  // ---- merges this CTA completed (at most its first and last piece); the
  // pipeline's shared memory is free now and holds the merge weights
  const int nmerge = sched[6];
  for (int k = 0; k < nmerge; ++k)
    merge_pieces_cta<HT, kPieceCost>(p, sched[7 + 3 * k], ht, sched[8 + 3 * k], sched[9 + 3 * k], total, parts,
                         reinterpret_cast<float*>(smem + C::kStageOff));
}

// ------------------------------------------------------------------------
// Tokens-on-M tcgen05 kernel for 16-head tiles.  With 16 heads, heads on M
// cannot feed the 5th-generation tensor cores (M is 64 or 128), so both
// products put the 64 tokens of a tile (or 128 latent elements) on M and the
// 16 heads on N:
//   S^T(t)  = K(t) . Q^T      M = 64 tokens, N = 16, K = 576: 36 tcgen05.mma,
//                             A = the tile's rows (K-major, 128-byte swizzle),
//                             B = the piece's q_lat rows; into TMEM, where row r
//                             sits in lane 32 (r / 16) + r % 16
//   O^T    += V(t)^T . P^T    M = 128 latent elements (four blocks), N = 16,
//                             K = 64 tokens: 16 tcgen05.mma, A = the value
//                             part of the tile's rows read MN-major (its 64
//                             elements of a chunk are contiguous), B = the
//                             bf16 weights written by the softmax warps
//                             (K-major, [16 heads][64 tokens])
// A narrow tcgen05.mma costs ~58-60 issue cycles on this part however small
// it is (measured for M = 64 and 128, N = 16 to 64), so a tile is ~3.1 K
// cycles of products, about what one SM's share of HBM needs to bring the
// tile's 72 KB.  Holding a tile from its load to its P . V left two 72 KB
// stages in shared memory and one chain (load, scores, softmax, P . V) per
// stage.  Instead the rows come twice: score units of three chunks stream
// through a five-slot ring and are released as soon as their score
// products are done; the value part (chunks 0-7) is read again, from L2,
// into a four-slot ring of two-chunk units, one per output block, for the
// output products.  HBM reads stay at the rows' bytes (measured 1.02x); L2
// to SM traffic doubles.  Eight softmax warps, two per TMEM lane quadrant,
// eight heads each.  One CTA per SM.
namespace tok {
constexpr int HT = 16;
constexpr int kTile = 64;                           // tokens per tile
// charge per sequence start, in tiles, of the balanced cut (launch, back to
// back: 53.9 / 53.1 / 52.0 / 53.8 / 54.1 us with 1 / 2 / 3 / 4 / 5)
constexpr int kPieceCost = 3;
constexpr int kChunkBytes = kTile * 128;            // one 64-element chunk of the tile's rows
// chunks per score unit: one TMA box each, whose issue costs the loading
// warp ~180 cycles, so units of one chunk (nine boxes a tile) made that warp
// the bottleneck (88.8 against 53.0 us)
constexpr int kSChunks = 3;
constexpr int kSUnitBytes = kSChunks * kChunkBytes; // 24 KB
constexpr int kSUnits = 5;                          // score-unit ring
constexpr int kSPerTile = kChunks / kSChunks;       // score units per tile
constexpr int kVUnitBytes = 2 * kChunkBytes;        // 16 KB: the 128 latent elements of one output block
constexpr int kVUnits = 4;                          // value-unit ring
constexpr int kMasks = 4;                           // row-mask ring (tiles)
constexpr int kQBytes = kChunks * HT * 128;         // 18 KB: q_lat rows, nine [16 x 128 B] chunks
constexpr int kPBytes = HT * 128;                   // 2 KB: weights, [16 heads x 64 tokens] bf16
constexpr int kQOff = 0;                            // two q_lat buffers (pieces alternate)
constexpr int kPOff = kQOff + 2 * kQBytes;          // two weight buffers (tiles alternate)
constexpr int kSUOff = kPOff + 2 * kPBytes;
constexpr int kVUOff = kSUOff + kSUnits * kSUnitBytes;
constexpr int kScrOff = kVUOff + kVUnits * kVUnitBytes;
constexpr int kScrBytes = (2 * 4 * HT + 4 * HT) * 4;  // per-quadrant maxima (x 2 tiles), row sums
constexpr int kBarOff = kScrOff + kScrBytes;
// su_full, su_empty, vu_full, vu_empty, mask_full, tile_mask, then q_full,
// q_empty, s_full, s_free, p_full, pv_done, drain (2 each), o_full, o_free
constexpr int kNumBars = 2 * kSUnits + 2 * kVUnits + 2 * kMasks + 7 * 2 + 2;
constexpr int kBytes = kBarOff + kNumBars * 8 + 16 + 16 * 4;  // barriers, TMEM slot, schedule
constexpr int kAlloc = kBytes + 1024;
static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0 && kSUOff % 1024 == 0 &&
                  kVUOff % 1024 == 0 && kQBytes % 1024 == 0 && kSUnitBytes % 1024 == 0 &&
                  kVUnitBytes % 1024 == 0,
              "128-byte swizzled operands start on 1 KB boundaries");
static_assert(kAlloc <= 227 * 1024, "shared memory");
static_assert(kChunks % kSChunks == 0, "whole score units per tile");
// a tile whose rows are not all tokens waits, in the softmax, for its own
// value units before P.V(u) can free any slot: the ring must hold one tile
static_assert(kVUnits >= 4, "value ring of at least one tile");
// warps: 0 score-unit loads, 1 score products (+ TMEM), 2 output products,
// 3 value-unit loads, 4-11 softmax
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kSW0 = 4;     // first softmax warp; warp w reads TMEM lane quadrant w % 4
constexpr int kSWarps = 8;  // softmax warps: two per lane quadrant, eight heads each
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kSCol = 0;   // two 16-column score buffers
constexpr uint32_t kOCol = 32;  // O^T: four 16-column blocks (latent elements 128 j ..)
constexpr uint32_t kIdescS = tc::instr_desc(64, HT, false);
constexpr uint32_t kIdescPV = tc::instr_desc(128, HT, false, true);

// Loads chunks [c0, c0 + nc) of the rows of one tile (tokens tok0 .. of a
// sequence of tok_end tokens) into dst, chunk c at dst + (c - c0) *
// kChunkBytes as [64 rows x 128 B], 128-byte swizzled; called by one warp,
// all lanes.  Lane i < nbox holds the block id of block piece i of the tile
// (mla_tile_bid).  A block that covers the tile is one 3-D box of nc chunks
// (tm3, whose box depth is nc), smaller blocks take one 2-D box (tm2) per
// piece and chunk.  Rows of invalid or missing pieces are not loaded.  When
// mask is not null, lane 0 stores there the tile's row mask.
__device__ __forceinline__ void issue_chunks(const MlaParams& p, const CUtensorMap* tm3,
                                             const CUtensorMap* tm2, uint8_t* dst, int c0, int nc,
                                             uint64_t* full, int lane_bid, int tok0, int tok_end,
                                             uint64_t pol, int lane, uint64_t* mask) {
  const int bs = p.block_size;
  const int rpb = bs < kTile ? bs : kTile;
  const int nbox = kTile / rpb;
  const int nval = min(kTile, tok_end - tok0);
  bool valid = false;
  int rows = 0, row0 = 0;
  if (lane < nbox) {
    rows = min(rpb, nval - lane * rpb);
    if (rows > 0) {
      row0 = (tok0 + lane * rpb) & (bs - 1);
      valid = lane_bid >= 0 && static_cast<int64_t>(lane_bid) < p.num_blocks;
    }
  }
  if (mask != nullptr) {
    uint64_t bits = 0;
    if (valid) bits = (rows >= 64 ? ~0ull : ((1ull << rows) - 1ull)) << (lane * rpb);
    const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits));
    const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits >> 32));
    if (lane == 0) *mask = (static_cast<uint64_t>(hi) << 32) | lo;
  }
  const uint32_t vb = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(vb) * rpb * nc * 128));
  __syncwarp();
  if (valid) {
    const int32_t row = lane_bid * bs + row0;
    uint8_t* st = dst + lane * rpb * 128;
    if (nbox == 1 && nc > 1) {
      tma_load_3d(st, tm3, 0, row, c0, full, pol);
    } else {
#pragma unroll 1
      for (int c = 0; c < nc; ++c)
        tma_load_2d(st + c * kChunkBytes, tm2, 64 * (c0 + c), row, full, pol);
    }
  }
}

// The tile positions of a chunk in order, with the block id of the current
// tile read one tile ahead (the issuing warps' walk; all lanes).
struct TileWalk {
  BalIter<kTile> it;
  BalPiece pc;
  int tl, L, bid;
  const int32_t* bt;
  bool have, first;  // a current tile; it starts a piece
  __device__ __forceinline__ bool advance(const MlaParams& p) {
    first = false;
    if (bt == nullptr || tl >= pc.te) {
      if (!it.next(p, pc)) return false;
      tl = pc.tb;
      bool cl;
      L = bal_len(p, pc.b, &cl);
      bt = p.block_tables + static_cast<int64_t>(pc.b) * p.max_blocks_per_seq;
      first = true;
    }
    return true;
  }
  __device__ __forceinline__ void start(const MlaParams& p, const BalIter<kTile>& it0, int lane) {
    it = it0;
    bt = nullptr;
    tl = 0;
    have = advance(p);
    bid = have ? mla_tile_bid(p, bt, tl * kTile, L, kTile, lane) : -1;
  }
};
}  // namespace tok

__global__ void __launch_bounds__(tok::kThreads, 1)
    mla_decode_tok_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_s3,
                          const __grid_constant__ CUtensorMap tm_v2,
                          const __grid_constant__ CUtensorMap tm_kv, const MlaParams p) {
  using namespace tok;
  using namespace tc;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* su_full = bars;                      // [kSUnits] a score unit landed
  uint64_t* su_empty = su_full + kSUnits;        // [kSUnits] its score products are done
  uint64_t* vu_full = su_empty + kSUnits;        // [kVUnits] a value unit landed
  uint64_t* vu_empty = vu_full + kVUnits;        // [kVUnits] its output products are done
  uint64_t* mask_full = vu_empty + kVUnits;      // [kMasks] a tile's row mask is written
  uint64_t* tile_mask = mask_full + kMasks;      // [kMasks] rows of the tile that exist
  uint64_t* q_full = tile_mask + kMasks;         // [2] a piece's q_lat landed
  uint64_t* q_empty = q_full + 2;                // [2] that piece's score products are done
  uint64_t* s_full = q_empty + 2;                // [2] scores of a tile in TMEM
  uint64_t* s_free = s_full + 2;                 // [2] the softmax warps have read them
  uint64_t* p_full = s_free + 2;                 // [2] weights of a tile written
  uint64_t* pv_done = p_full + 2;                // [2] its output products are done
  uint64_t* drain = pv_done + 2;                 // [2] every product of an issuing thread is done
  uint64_t* o_full = drain + 2;                  // a piece's output is complete in TMEM
  uint64_t* o_free = o_full + 1;                 // the epilogue has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  int* sched = reinterpret_cast<int*>(smem + kBarOff + kNumBars * 8 + 16);
  volatile int* abort_flag = sched + 13;
  float* wmax = reinterpret_cast<float*>(smem + kScrOff);  // [2 tiles][4 quadrants][16 heads]
  float* lsum = wmax + 2 * 4 * HT;                          // [4 quadrants][16 heads]

  const int ht = blockIdx.x;
  const int c = blockIdx.y;
  const int NC = gridDim.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h0 = ht * HT;
  const int B = p.num_seqs;

  if (warp == 0) bal_schedule<kTile, tok::kPieceCost>(p, c, NC, c == 0 && ht == 0, sched, lane);
  if (threadIdx.x == 64) {  // not warp 1, which allocates the tensor memory meanwhile
    for (int s = 0; s < kSUnits; ++s) {
      mbar_init(&su_full[s], 1);
      mbar_init(&su_empty[s], 1);
    }
    for (int s = 0; s < kVUnits; ++s) {
      mbar_init(&vu_full[s], 1);
      mbar_init(&vu_empty[s], 1);
    }
    for (int s = 0; s < kMasks; ++s) mbar_init(&mask_full[s], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kSWarps);
      mbar_init(&p_full[s], kSWarps);
      mbar_init(&pv_done[s], 1);
      mbar_init(&drain[s], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, kSWarps);
    mbar_init_fence();
  }
  if (warp == 1) {  // this warp owns the CTA's tensor memory
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int g0 = sched[2], g1 = sched[3];
  const int64_t total = static_cast<int64_t>(sched[0]) + static_cast<int64_t>(tok::kPieceCost) * B;
  const int parts = total < NC ? static_cast<int>(total) : NC;  // chunks with work
  const BalIter<kTile> it0{sched[4], sched[5], g0, g1, false};
  const bool has_work = g0 < g1;

  // sequences without tokens: zero output rows (chunk c takes b = c mod NC)
  for (int b = c; b < B; b += NC) {
    if (bal_tiles<kTile>(p, b) != 0) continue;
    for (int i = threadIdx.x; i < HT * (kLat / 8); i += tok::kThreads) {
      const int h = i / (kLat / 8), e = i % (kLat / 8);
      reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * p.num_heads + h0 + h) *
                                           kLat)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  int issued = 0, nq = 0;  // units and q_lat rows whose loads this warp issued
  if ((warp == 0 || warp == 3) && has_work) {
    // ------------------------------------------------------------ TMA loads
    // Warp 0: the three score units of each tile (chunks 0-2, 3-5, 6-8; unit
    // n into ring slot n % kSUnits once the score products of unit n -
    // kSUnits are done), the tile's row mask with its first unit, and each
    // piece's q_lat (buffer piece & 1, once the score products of the piece
    // two before are done).  Warp 3: the four value units of each tile
    // (chunks 2j, 2j + 1: the 128 latent elements of output block j), read
    // again from L2 for the output products, unit n into slot n % kVUnits
    // once the output products of unit n - kVUnits are done.  The block id
    // of the next tile is read before the waits.
    const bool is_s = warp == 0;
    const uint64_t pol = is_s ? l2_policy_evict_normal()
                              : (p.kv_evict_first ? l2_policy_evict_first() : l2_policy_evict_normal());
    const uint64_t qpol = l2_policy_evict_normal();
    if (lane == 0) {
      prefetch_tensormap(is_s ? &tm_s3 : &tm_v2);
      prefetch_tensormap(&tm_kv);
      if (is_s) prefetch_tensormap(&tm_q);
    }
    TileWalk w;
    w.start(p, it0, lane);
    const int nunits = is_s ? kSPerTile : 4;
    const int ring = is_s ? kSUnits : kVUnits;
    uint64_t* full = is_s ? su_full : vu_full;
    uint64_t* empty = is_s ? su_empty : vu_empty;
    bool ok = true;
    int u = 0;
    while (ok && w.have) {
      const int b_cur = w.pc.b, tok0 = w.tl * kTile, L_cur = w.L, bid_cur = w.bid;
      const bool first = w.first;
      ++w.tl;
      w.have = w.advance(p);
      w.bid = w.have ? mla_tile_bid(p, w.bt, w.tl * kTile, w.L, kTile, lane) : -1;
      if (is_s && first) {
        if (nq >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&q_empty[nq & 1], ((nq - 2) >> 1) & 1,
                                                         abort_flag));
          if (!ok) break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[nq & 1], HT * kRowBytes);
          // one box: 9 chunks x 16 rows x 128 bytes
          tma_load_3d(smem + kQOff + (nq & 1) * kQBytes, &tm_q, 0, b_cur * p.num_heads + h0, 0,
                      &q_full[nq & 1], qpol);
        }
        ++nq;
      }
      for (int i = 0; i < nunits && ok; ++i) {
        const int slot = issued % ring;
        if (issued >= ring) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[slot], ((issued / ring) - 1) & 1,
                                                         abort_flag));
          if (!ok) break;
        }
        uint8_t* dst = smem + (is_s ? kSUOff + slot * kSUnitBytes : kVUOff + slot * kVUnitBytes);
        uint64_t* msk = (is_s && i == 0) ? &tile_mask[u % kMasks] : nullptr;
        issue_chunks(p, is_s ? &tm_s3 : &tm_v2, &tm_kv, dst, is_s ? kSChunks * i : 2 * i,
                     is_s ? kSChunks : 2, &full[slot], bid_cur, tok0, L_cur, pol, lane, msk);
        if (msk != nullptr && lane == 0) mbar_arrive(&mask_full[u % kMasks]);  // after the mask store
        ++issued;
      }
      ++u;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------ MMA issuers
    // One thread of warp 1 issues the score products, one of warp 2 the
    // output products; each commits its own (a commit tracks the issuing
    // thread's products).
    if (lane == 0 && has_work) {
      const bool is_s = warp == 1;
      const uint32_t su0 = smem_u32(smem + kSUOff);
      const uint32_t vu0 = smem_u32(smem + kVUOff);
      const uint32_t q0 = smem_u32(smem + kQOff);
      const uint32_t p0 = smem_u32(smem + kPOff);
      BalIter<kTile> it = it0;
      BalPiece pc;
      bool ok = true;
      int u = 0, kp = 0, n = 0;  // tile, piece, unit
      while (ok && it.next(p, pc)) {
        if (is_s) {
          // S^T(u) over the 576 elements, unit by unit: 4 k-steps of 16 per
          // 64-element chunk (a k-step advances the start by 32 bytes inside
          // the 128-byte swizzled rows), into score buffer u & 1 once the
          // softmax has read S^T(u - 2) from it; each unit's slot is released
          // when its products are done
          const uint32_t qb = q0 + (kp & 1) * kQBytes;
          ok = mbar_wait_bounded_long(&q_full[kp & 1], (kp >> 1) & 1, abort_flag);
          for (int tl = pc.tb; tl < pc.te && ok; ++tl, ++u) {
            ok = u < 2 || mbar_wait_bounded_long(&s_free[u & 1], ((u - 2) >> 1) & 1, abort_flag);
            const uint32_t d = tmem + kSCol + HT * (u & 1);
            for (int i = 0; i < kSPerTile && ok; ++i, ++n) {
              const int slot = n % kSUnits;
              ok = mbar_wait_bounded_long(&su_full[slot], (n / kSUnits) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint32_t kb = su0 + slot * kSUnitBytes;
#pragma unroll
              for (int j = 0; j < kSChunks * 4; ++j) {
                const int ch = kSChunks * i + (j >> 2);
                tc_mma_ss(d, smem_desc(kb + (j >> 2) * kChunkBytes + 32 * (j & 3), 16, 1024),
                          smem_desc(qb + ch * (HT * 128) + 32 * (j & 3), 16, 1024), kIdescS,
                          (i > 0 || j > 0) ? 1u : 0u);
              }
              tc_commit(&su_empty[slot]);
            }
            if (ok) tc_commit(&s_full[u & 1]);
          }
          if (ok) tc_commit(&q_empty[kp & 1]);  // this piece's q_lat is no longer read
        } else {
          // O^T += V(u)^T . P^T(u): block j (latent elements 128 j ..) reads
          // value unit 4u + j MN-major (leading offset: the next 64 elements
          // = the next chunk; stride offset: the next 8 tokens = 1 KB; a
          // k-step of 16 tokens advances 2 KB).  A piece's first tile starts
          // the output afresh once the previous piece's epilogue has read it.
          for (int tl = pc.tb; tl < pc.te && ok; ++tl, ++u) {
            const bool fresh = tl == pc.tb;
            ok = mbar_wait_bounded_long(&p_full[u & 1], (u >> 1) & 1, abort_flag) &&
                 (!fresh || kp == 0 || mbar_wait_bounded_long(o_free, (kp - 1) & 1, abort_flag));
            const uint32_t pb = p0 + (u & 1) * kPBytes;
            for (int j = 0; j < kLat / 128 && ok; ++j, ++n) {
              const int slot = n % kVUnits;
              ok = mbar_wait_bounded_long(&vu_full[slot], (n / kVUnits) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint32_t vb = vu0 + slot * kVUnitBytes;
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                tc_mma_ss(tmem + kOCol + HT * j, smem_desc(vb + kk * 2048, kChunkBytes, 1024),
                          smem_desc(pb + 32 * kk, 16, 1024), kIdescPV,
                          (!fresh || kk > 0) ? 1u : 0u);
              tc_commit(&vu_empty[slot]);
            }
            if (!ok) break;
            tc_commit(&pv_done[u & 1]);
            if (tl + 1 == pc.te) tc_commit(o_full);
          }
        }
        ++kp;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
      }
      // every product issued completes before tensor memory is freed
      tc_commit(&drain[is_s ? 0 : 1]);
      mbar_wait_bounded(&drain[is_s ? 0 : 1], 0, nullptr);
    }
    __syncwarp();
  } else if (warp >= kSW0 && has_work) {
    // ------------------------------------------------------------ softmax
    // Eight warps: warp w reads TMEM lane quadrant q = w % 4 and takes heads
    // hs .. hs + 7, hs = 8 ((w - 3) / 4).  For the scores lanes 0-15 of a
    // quadrant hold tokens 16 q .. 16 q + 15 of the tile; for the output
    // every lane holds latent element 128 j + 32 q + lane of block j.  Per
    // tile: the per-head maximum over the tile's tokens (16-lane shuffles,
    // then the four quadrants' maxima through shared memory and one named
    // barrier), the lazy rescale of the running maximum (it moves only when
    // a score beats it by more than 2^8; O^T is then scaled in TMEM once the
    // previous tile's products are done), the bf16 weights into weight
    // buffer u & 1, and per-lane partial row sums.  Every named barrier
    // carries the waits' results, so the eight warps leave together.
    constexpr int kHW = 8;  // heads per softmax warp
    const int q = warp & 3;
    const int hs = kHW * ((warp - kSW0) / 4);
    const int tok = 16 * q + lane;  // the token whose scores this lane reads (lanes 0-15)
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    bool ok = true, fail = false;
    BalIter<kTile> it = it0;
    BalPiece pc;
    int u = 0, kp = 0;
    while (ok && it.next(p, pc)) {
      const int b = pc.b;
      const bool whole = pc.tb == 0 && pc.te == pc.n;
      float m_run[kHW], l_part[kHW];
#pragma unroll
      for (int h = 0; h < kHW; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
      }
      for (int tl = pc.tb; tl < pc.te; ++tl, ++u) {
        const int k = u & 1;
        const bool w_ok = __all_sync(
            0xffffffffu,
            mbar_wait_bounded_long(&s_full[k], (u >> 1) & 1, abort_flag) &&
                mbar_wait_bounded(&mask_full[u % kMasks], (u / kMasks) & 1, abort_flag));
        float x[kHW];
        uint64_t mask = 0;
        if (w_ok) {
          tc_fence_after();
          tc_ld8_nowait(tmem + lane_base + kSCol + HT * k + hs, x);
          tc_wait_ld();
          mask = tile_mask[u % kMasks];  // read before s_free: the slot is reused 4 tiles on
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[k]);  // the score products of tile u + 2 may go
        }
        const bool valid = w_ok && lane < 16 && ((mask >> tok) & 1ull);
        float mx[kHW];
#pragma unroll
        for (int h = 0; h < kHW; ++h) {
          x[h] = valid ? x[h] * p.scale_log2 : -INFINITY;
          mx[h] = x[h];
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
#pragma unroll
          for (int h = 0; h < kHW; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
        if (lane == 0) {
          float4* wm = reinterpret_cast<float4*>(wmax + (k * 4 + q) * HT + hs);
          wm[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
          wm[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
        }
        if (!named_barrier_and(1, kSWarps * 32, w_ok && !fail)) {
          ok = false;
          break;
        }
        float tmax[kHW];
#pragma unroll
        for (int h = 0; h < kHW; ++h) tmax[h] = -INFINITY;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const float4* wa = reinterpret_cast<const float4*>(wmax + (k * 4 + qq) * HT + hs);
          const float4 v0 = wa[0], v1 = wa[1];
          tmax[0] = fmaxf(tmax[0], v0.x);
          tmax[1] = fmaxf(tmax[1], v0.y);
          tmax[2] = fmaxf(tmax[2], v0.z);
          tmax[3] = fmaxf(tmax[3], v0.w);
          tmax[4] = fmaxf(tmax[4], v1.x);
          tmax[5] = fmaxf(tmax[5], v1.y);
          tmax[6] = fmaxf(tmax[6], v1.z);
          tmax[7] = fmaxf(tmax[7], v1.w);
        }
        bool resc = false;
        float corr[kHW];
#pragma unroll
        for (int h = 0; h < kHW; ++h) {
          corr[h] = 1.f;
          if (tmax[h] > m_run[h] + kRescaleLog2) {  // always on a piece's first tile
            corr[h] = exp2f(m_run[h] - tmax[h]);     // 0 while m_run is -inf
            m_run[h] = tmax[h];
            resc = true;
          }
        }
        bool t_ok = true;
        if (resc) {  // the same on every thread of the warp: the maxima are shared
#pragma unroll
          for (int h = 0; h < kHW; ++h) l_part[h] *= corr[h];
          if (tl != pc.tb) {
            t_ok = __all_sync(0xffffffffu,
                              mbar_wait_bounded_long(&pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1,
                                                     abort_flag));
            if (t_ok) {
              tc_fence_after();
#pragma unroll
              for (int j = 0; j < kLat / 128; ++j) {
                float o[kHW];
                tc_ld8_nowait(tmem + lane_base + kOCol + HT * j + hs, o);
                tc_wait_ld();
#pragma unroll
                for (int h = 0; h < kHW; ++h) o[h] *= corr[h];
                tc_st8_nowait(tmem + lane_base + kOCol + HT * j + hs, o);
              }
              tc_wait_st();
            }
          }
        }
        float pw[kHW];
#pragma unroll
        for (int h = 0; h < kHW; ++h) {
          // a masked score is -inf and m_run is finite once a token was seen
          pw[h] = x[h] == -INFINITY ? 0.f : exp2f(x[h] - m_run[h]);
          l_part[h] += pw[h];
        }
        // weight buffer k is free once P.V(u - 2) has read it.  A tile with
        // rows that hold no token waits for this warp's two value units:
        // first for P.V(u - 1), which releases the ring's slots to this
        // tile (until then a unit's barrier may still be a phase behind,
        // and its parity would read as this tile's), then for the units.
        const bool partial = mask != ~0ull;  // the same on every lane
        const int n0 = 4 * u + 2 * (hs / kHW);  // value units of this warp's chunks
        t_ok = __all_sync(
            0xffffffffu,
            t_ok &&
                (u < 2 ||
                 mbar_wait_bounded_long(&pv_done[k], ((u - 2) >> 1) & 1, abort_flag)) &&
                (!partial ||
                 ((u < 1 || mbar_wait_bounded_long(&pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1,
                                                   abort_flag)) &&
                  mbar_wait_bounded_long(&vu_full[n0 % kVUnits], (n0 / kVUnits) & 1, abort_flag) &&
                  mbar_wait_bounded_long(&vu_full[(n0 + 1) % kVUnits], ((n0 + 1) / kVUnits) & 1,
                                         abort_flag))));
        if (t_ok) {
          if (lane < 16) {
            // element (head h, token tok) of the K-major 128-byte swizzled
            // [16 x 128 B] weight tile
            uint8_t* pb = smem + kPOff + k * kPBytes;
            const uint32_t unit = static_cast<uint32_t>(tok >> 3);
            const uint32_t sub = static_cast<uint32_t>(tok & 7) << 1;
#pragma unroll
            for (int h = 0; h < kHW; ++h)
              *reinterpret_cast<__nv_bfloat16*>(pb + (hs + h) * 128 +
                                                (((unit ^ ((hs + h) & 7)) << 4) | sub)) =
                  __float2bfloat16_rn(pw[h]);
            if (!valid) {
              // a row that holds no token: zero its value part (0 x NaN
              // would poison the output products); the two warps of a
              // quadrant take two value units (four chunks) each
#pragma unroll 1
              for (int i = 0; i < 2; ++i) {
                uint8_t* row = smem + kVUOff + ((n0 + i) % kVUnits) * kVUnitBytes + tok * 128;
                for (int e = 0; e < 16; ++e)
                  *reinterpret_cast<uint4*>(row + (e >> 3) * kChunkBytes + ((e & 7) << 4)) =
                      make_uint4(0u, 0u, 0u, 0u);
              }
            }
          }
          fence_proxy_async_smem();  // generic writes before the tensor cores read them
          tc_fence_before();         // and the rescale's TMEM stores
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[k]);
        } else {
          fail = true;  // the next named barrier takes all eight warps out
          if (lane == 0) *abort_flag = 1;
        }
      }
      if (!ok) break;

      // ---- epilogue of the piece: 1 / l per head, then O^T from TMEM
      const bool e_ok = !fail && __all_sync(0xffffffffu,
                                            mbar_wait_bounded_long(o_full, kp & 1, abort_flag));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1)
#pragma unroll
        for (int h = 0; h < kHW; ++h) l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], off);
      if (lane == 0) {
        float4* ls = reinterpret_cast<float4*>(lsum + q * HT + hs);
        ls[0] = make_float4(l_part[0], l_part[1], l_part[2], l_part[3]);
        ls[1] = make_float4(l_part[4], l_part[5], l_part[6], l_part[7]);
      }
      if (!named_barrier_and(1, kSWarps * 32, e_ok)) {
        ok = false;
        break;
      }
      float lrow[kHW], inv[kHW];
#pragma unroll
      for (int h = 0; h < kHW; ++h) {
        lrow[h] = lsum[hs + h] + lsum[HT + hs + h] + lsum[2 * HT + hs + h] + lsum[3 * HT + hs + h];
        inv[h] = lrow[h] > 0.f ? 1.f / lrow[h] : 0.f;
      }
      tc_fence_after();
      const int64_t bh0 = static_cast<int64_t>(b) * p.num_heads + h0 + hs;
      const int slot = 2 * c + (pc.tb > 0 ? 0 : 1);
      const int64_t srow0 = (static_cast<int64_t>(ht) * p.num_slots + slot) * HT + hs;
#pragma unroll
      for (int j = 0; j < kLat / 128; ++j) {
        float o[kHW];
        tc_ld8_nowait(tmem + lane_base + kOCol + HT * j + hs, o);
        tc_wait_ld();
        const int col = 128 * j + 32 * q + lane;
        if (whole) {
#pragma unroll
          for (int h = 0; h < kHW; ++h)
            p.out[(bh0 + h) * kLat + col] = __float2bfloat16_rn(o[h] * inv[h]);
        } else {
#pragma unroll
          for (int h = 0; h < kHW; ++h) p.ws_o[(srow0 + h) * kLat + col] = o[h] * inv[h];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);  // the next piece's products may overwrite O^T
      if (!whole) {
        if (q == 0) {
#pragma unroll
          for (int h = 0; h < kHW; ++h)
            if (lane == h)
              p.ws_lse[srow0 + h] = lrow[h] > 0.f ? m_run[h] + log2f(lrow[h]) : -INFINITY;
        }
        // count the piece; the CTA that completes the sequence's count merges
        // it after its own work and returns the counter to zero
        named_barrier_and(1, kSWarps * 32, true);  // every partial of this piece is written
        if (threadIdx.x == kSW0 * 32) {
          __threadfence();
          const int c_first = bal_chunk<tok::kPieceCost>(pc.pre, b, total, parts);
          const int c_last = bal_chunk<tok::kPieceCost>(pc.pre + pc.n - 1, b, total, parts);
          unsigned* ctr = p.counters + static_cast<int64_t>(b) * (p.num_heads / HT) + ht;
          const unsigned prev = atomicAdd(ctr, 1u);
          if (prev + 1u == static_cast<unsigned>(c_last - c_first + 1)) {
            atomicExch(ctr, 0u);
            __threadfence();
            const int m = sched[6]++;
            sched[7 + 3 * m] = b;
            sched[8 + 3 * m] = pc.pre;
            sched[9 + 3 * m] = pc.n;
          }
        }
      }
      ++kp;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  }

  // ---- teardown: every role is done and the issuing threads drained their
  // products; after a timeout the loads in flight land first
  __syncthreads();
  if (*abort_flag) {
    if ((warp == 0 || warp == 3) && lane == 0) {
      const int ring = warp == 0 ? kSUnits : kVUnits;
      uint64_t* full = warp == 0 ? su_full : vu_full;
      for (int t = issued > ring ? issued - ring : 0; t < issued; ++t)
        mbar_wait_bounded(&full[t % ring], (t / ring) & 1, nullptr);
      for (int k2 = nq > 2 ? nq - 2 : 0; k2 < nq; ++k2)
        mbar_wait_bounded(&q_full[k2 & 1], (k2 >> 1) & 1, nullptr);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  // ---- merges this CTA completed; the rings' shared memory holds the weights
  const int nmerge = sched[6];
  for (int k = 0; k < nmerge; ++k)
    merge_pieces_cta<HT, tok::kPieceCost, 6, true>(p, sched[7 + 3 * k], ht, sched[8 + 3 * k], sched[9 + 3 * k],
                                  total, parts, reinterpret_cast<float*>(smem + kSUOff));
}

pa_status launch_mla_tok(const CUtensorMap& mq, const CUtensorMap& ms3, const CUtensorMap& mv2,
                         const CUtensorMap& mkv, const MlaParams& p, dim3 grid,
                         cudaStream_t stream) {
  static std::atomic<uint64_t> smem_raised{0};
  auto kern = mla_decode_tok_kernel;
  if (!ensure_smem_limit(kern, tok::kAlloc, smem_raised)) return PA_ERR_CUDA;
  kern<<<grid, tok::kThreads, tok::kAlloc, stream>>>(mq, ms3, mv2, mkv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <int HT>
pa_status launch_mla_split(const CUtensorMap& mq, const CUtensorMap& mkv, const MlaParams& p,
                           dim3 grid, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_raised{0};
  auto kern = mla_decode_split_kernel<HT>;
  constexpr int kSmem = MlaCfg<HT>::kAlloc;
  if (!ensure_smem_limit(kern, kSmem, smem_raised)) return PA_ERR_CUDA;
  kern<<<grid, kThreads, kSmem, stream>>>(mq, mkv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// 2-D bf16 map over [rows, 576] with a 1152-byte row stride; box = 64
// elements (128 bytes) x box_rows, 128-byte swizzled.
bool make_row576_map(CUtensorMap* map, const void* base, int64_t rows, int32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over the same [rows, 576] rows as {64 elements, rows, 9
// chunks} (strides 1152 and 128 bytes): a box {64, box_rows, box_chunks}
// lands as box_chunks [box_rows x 128 B] chunk regions one after another,
// 128-byte swizzled, the layout the 2-D boxes build one chunk at a time.
bool make_row576_chunked_map(CUtensorMap* map, const void* base, int64_t rows,
                             int32_t box_rows, int32_t box_chunks = kChunks) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(kChunks)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes), 128u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_chunks)};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The rope half of one CTA of the tcgen05 kernel: 32 elements (64 bytes) of
// each row, 64-byte swizzled.
bool make_rope32_map(CUtensorMap* map, const void* base, int64_t rows, int32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
  const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

// 128: the tcgen05 kernel (mla_decode_tc.cu); 64 / 16: the mma.sync kernel
int mla_head_tile(int32_t num_heads) {
  return num_heads % 128 == 0 ? 128 : num_heads % 64 == 0 ? 64 : 16;
}

DecodePlan make_mla_plan(int32_t num_seqs, int32_t num_heads, int32_t max_context_len,
                         int32_t num_sms) {
  if (num_sms <= 0) num_sms = 148;
  const int ht = mla_head_tile(num_heads);
  if (max_context_len <= 0 || num_seqs <= 0 || num_heads <= 0) return {1, 0};
  // One wave per head tile: 2-CTA clusters for the tcgen05 kernel, resident
  // CTAs for the mma.sync kernel, each taking an equal share of the tile's
  // token tiles (the kernels derive their chunk from context_lens);
  // num_splits = chunks (clusters) per head tile
  const int64_t per_tile = ht == 128 ? (num_sms / 2) / (num_heads / 128)
                                     : static_cast<int64_t>(num_sms) / (num_heads / ht);
  return {static_cast<int32_t>(per_tile < 1 ? 1 : per_tile), 0};
}

// [error word | pad] [counters B * H/HT (x 2 output halves for HT = 128)]
// [lse H/HT * 2C * HT] [o H/HT * 2C * HT * 512], C = plan.num_splits chunks
// (clusters) per head tile, two partial slots each.
size_t mla_workspace_bytes(int32_t num_seqs, int32_t num_heads, const DecodePlan& plan) {
  const int ht = mla_head_tile(num_heads);
  size_t bytes = kWorkspaceHeader;
  const size_t rows = static_cast<size_t>(num_heads) * 2 * plan.num_splits;  // slots x heads
  bytes += align256(static_cast<size_t>(num_seqs) * (num_heads / ht) * (ht == 128 ? 2 : 1) * 4);
  bytes += align256(rows * sizeof(float));
  bytes += rows * kLat * sizeof(float);
  return bytes;
}

pa_status launch_mla_decode(const MlaDecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return PA_OK;
  const int ht = mla_head_tile(a.num_heads);
  const int tile = ht == 128 ? mla_tc_tile() : ht == 64 ? MlaCfg<64>::kTile : tok::kTile;
  const int32_t box_rows = a.block_size < tile ? a.block_size : tile;
  CUtensorMap mq, mkv;
  // mma.sync kernel: q_lat rows and, when a block covers a whole tile, the
  // latent tiles come as one 3-D box each (all nine 64-element chunks)
  const bool chunked_kv = ht == 64 && box_rows == tile;
  const int64_t cache_rows = a.num_blocks * a.block_size;
  if (!(ht == 128 ? make_row576_map(&mq, a.q_latent, static_cast<int64_t>(a.num_seqs) * a.num_heads, ht)
                  : make_row576_chunked_map(&mq, a.q_latent,
                                            static_cast<int64_t>(a.num_seqs) * a.num_heads, ht)) ||
      !(chunked_kv ? make_row576_chunked_map(&mkv, a.latent_cache, cache_rows, box_rows)
                   : make_row576_map(&mkv, a.latent_cache, cache_rows, box_rows)))
    return PA_ERR_CUDA;
  MlaParams p;
  p.num_seqs = a.num_seqs;
  p.num_slots = 2 * a.plan.num_splits;
  p.out = static_cast<__nv_bfloat16*>(a.out_latent);
  p.q_latent = static_cast<const __nv_bfloat16*>(a.q_latent);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.err = reinterpret_cast<unsigned*>(ws);
  const size_t nrows = static_cast<size_t>(a.num_heads) * 2 * a.plan.num_splits;
  const size_t ctr_bytes =
      align256(static_cast<size_t>(a.num_seqs) * (a.num_heads / ht) * (ht == 128 ? 2 : 1) * 4);
  p.counters = reinterpret_cast<unsigned*>(ws + kWorkspaceHeader);
  p.ws_lse = reinterpret_cast<float*>(ws + kWorkspaceHeader + ctr_bytes);
  p.ws_o = reinterpret_cast<float*>(ws + kWorkspaceHeader + ctr_bytes + align256(nrows * 4));
  p.num_blocks = a.num_blocks;
  p.num_heads = a.num_heads;
  p.block_size = a.block_size;
  int lg = 0;
  while ((1 << lg) < a.block_size) ++lg;
  p.log2_bs = lg;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_splits = a.plan.num_splits;
  p.tokens_per_split = a.plan.tokens_per_split;
  p.kv_evict_first = (a.num_heads == ht && ht != 128) ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)
  if (ht == 128) {
    CUtensorMap mrope;
    if (!make_rope32_map(&mrope, a.latent_cache, a.num_blocks * a.block_size, box_rows))
      return PA_ERR_CUDA;
    const dim3 grid(static_cast<unsigned>(2 * a.plan.num_splits),
                    static_cast<unsigned>(a.num_heads / ht), 1u);
    return launch_mla_tc(mrope, mkv, p, grid, stream);
  }
  const dim3 grid(static_cast<unsigned>(a.num_heads / ht), static_cast<unsigned>(a.plan.num_splits),
                  1u);
  if (ht == 64) return launch_mla_split<64>(mq, mkv, p, grid, stream);
  // 16-head tiles: score units of three chunks and value units of two, as
  // 3-D boxes when a block covers a tile (else mkv's 2-D boxes)
  CUtensorMap ms3 = mkv, mv2 = mkv;
  if (box_rows == tok::kTile &&
      (!make_row576_chunked_map(&ms3, a.latent_cache, cache_rows, box_rows, tok::kSChunks) ||
       !make_row576_chunked_map(&mv2, a.latent_cache, cache_rows, box_rows, 2)))
    return PA_ERR_CUDA;
  return launch_mla_tok(mq, ms3, mv2, mkv, p, grid, stream);
}

}  // namespace pa_detail
