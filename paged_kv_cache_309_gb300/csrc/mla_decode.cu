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
// How (sm_103a):
//  * grid = (head tile, chunk); a head tile is 64 heads (16 when the head
//    count is not a multiple of 64), one wave of resident CTAs per head
//    tile.  Balanced schedule: the sequences' 32-token tiles laid end to
//    end are cut into one chunk of equal cost per CTA (each sequence start
//    charged 2 tiles), derived by every CTA from context_lens; a chunk that
//    crosses sequences runs as pieces (q_lat reloaded per piece, the
//    pipeline's stage and phase counters running on across pieces).  Head tiles of one chunk are adjacent in the launch
//    order, so the second reads the latent rows from L2.
//  * the split's tokens stream in tiles of 32 through a TMA ring (3 stages
//    for 64 heads; for 16 heads 2 stages and two CTAs per SM), 128-byte
//    swizzled, completion on an mbarrier; a per-tile mask marks the rows
//    that exist.  When a block covers the tile it is one 3-D box (all nine
//    64-element chunks), else one [rows x 128 B] box per (block piece,
//    chunk).  A ninth warp issues the loads: it refills a stage once all
//    eight compute warps have arrived on the stage's `empty` barrier after
//    their P . V of the tile there (warp 0 issued them before, between the
//    CTA barrier and its own softmax, which every warp then waited for).
//    Compute warp 0 loads each piece's q_lat (one 3-D box).
//  * eight warps per tile: (1) S = Q . K^T on the tensor cores
//    (mma.sync m16n8k16, bf16 in, fp32 accumulate; heads on M, each warp a
//    16-head x 16-token block over all 576 elements, or for 16 heads a
//    16 x 8 block over half of them) written to a double-buffered fp32
//    score tile in shared memory; (2) one barrier;
//    (3) each warp takes 16 heads x (512 / warps per head block) output
//    elements: reads its heads' scores straight into the A-fragment
//    positions, runs an fp32 online softmax in base 2 with a lazy rescale
//    (the running max moves only when a score beats it by more than 2^8),
//    rounds the weights to bf16 and accumulates O += P . V from the same
//    shared-memory tile (V = the first 512 elements of each row).
//  * epilogue per piece: a piece holding a whole sequence writes bf16 o_lat;
//    the others write fp32 partials + log2-sum-exp to the chunk's two slots
//    (a piece whose sequence began in an earlier chunk, one whose sequence
//    begins in this chunk) and count themselves per (sequence,
//    head tile); the CTA that completes a count merges that sequence after
//    its own pieces and zeroes the count.
//
// Every wait is bounded (2 s).  A timeout sets an error bit in the
// workspace's error word, drains the copies in flight and leaves.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>

#include "mla_common.cuh"

namespace pa_detail {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();  // decode.cu

namespace {

using namespace pa;
using namespace mla;

constexpr int kWarps = 8;                 // compute warps; warp kWarps issues the tile loads
constexpr int kComputeThreads = kWarps * 32;
constexpr int kThreads = kComputeThreads + 32;

template <int HT>
struct MlaCfg {
  static constexpr int kMB = HT / 16;                   // 16-head blocks
  static constexpr int kTile = 32;                      // tokens per stage
  static constexpr int kStages = HT == 64 ? 3 : 2;
  static constexpr int kCtasPerSm = HT == 64 ? 1 : 2;  // 16 heads: two CTAs hide each other's barriers
  // registers per thread of the nine-warp block (measured on GB300: 16 heads
  // at 96 keep two CTAs per SM, by ncu's occupancy section, without the
  // spills of 80; 64 heads launch at 168 and not at 200)
  static constexpr int kMaxRegs = HT == 64 ? 168 : 96;
  static constexpr int kWarpsPerMB = kWarps / kMB;      // 2 or 8
  // S: a 16-head block's warps split the tile's tokens into kTokGroups
  // groups and, for 16 heads, the 576-element reduction into two halves
  static constexpr int kKSplit = HT == 64 ? 1 : 2;
  static constexpr int kTokGroups = kWarpsPerMB / kKSplit;  // 2 or 4
  static constexpr int kSTok = kTile / kTokGroups;      // tokens per warp in S: 16 or 8
  static constexpr int kDW = kLat / kWarpsPerMB;        // output elements per warp: 256 or 64
  static constexpr int kQBytes = kChunks * HT * 128;
  static constexpr int kChunkBytes = kTile * 128;
  static constexpr int kStageBytes = kChunks * kChunkBytes;
  static constexpr int kSStride = kTile + 8;            // floats per score row
  static constexpr int kSBytes = kKSplit * HT * kSStride * 4;  // one partial per k-half
  static constexpr int kStageOff = kQBytes;
  static constexpr int kSOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBarOff = kSOff + 2 * kSBytes;
  static constexpr int kBytes = kBarOff + (3 * kStages + 1) * 8 + 64;  // full, mask, q, empty, schedule
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc * kCtasPerSm <= 227 * 1024, "shared memory");
  static_assert(kSTok == 16 || kSTok == 8, "S split");
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
constexpr int kPieceCost = 2;  // tiles
__device__ __forceinline__ int bal_chunk(int64_t t, int b, int64_t total, int parts) {
  return static_cast<int>((t + static_cast<int64_t>(kPieceCost) * (b + 1)) * parts / total);
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
template <int HT>
__device__ __forceinline__ void merge_pieces_cta(const MlaParams& p, int b, int ht, int pre, int n,
                                                 int64_t total, int parts, float* wsm) {
  const int c_first = bal_chunk(pre, b, total, parts);
  const int c_last = bal_chunk(pre + n - 1, b, total, parts);
  const int np = c_last - c_first + 1;
  const int s0 = 2 * c_first + 1;
  auto slot = [&](int i) { return i == 0 ? s0 : 2 * (c_first + i); };
  const int64_t base = static_cast<int64_t>(ht) * p.num_slots;
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
  // kU 16-byte columns per thread and two pieces per round in flight (the
  // loads are L2 round trips; one column at a time left the merge latency-bound)
  constexpr int kCols = HT * (kLat / 4);
  constexpr int kU = 4;
  const int nthr = blockDim.x;
  auto part = [&](int i, int idx) {
    const int h = idx / (kLat / 4), e4 = idx % (kLat / 4);
    return __ldcg(reinterpret_cast<const float4*>(p.ws_o + ((base + slot(i)) * HT + h) * kLat) + e4);
  };
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
  if (warp == 0) {
    int T = 0;
    bool any_clip = false;
    for (int b0 = 0; b0 < B; b0 += 32) {
      int n = 0;
      if (b0 + lane < B) {
        bool cl;
        n = (bal_len(p, b0 + lane, &cl) + kTile - 1) / kTile;
        any_clip |= cl;
      }
      T += static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(n)));
    }
    if (__any_sync(0xffffffffu, any_clip) && c == 0 && ht == 0 && lane == 0)
      atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
    // first tile of chunk k: the smallest t with cost(t) * parts >= k * total,
    // in the first non-empty sequence whose last tile reaches that cost (T
    // when none does); also that sequence and its first tile
    const int64_t total = static_cast<int64_t>(T) + static_cast<int64_t>(kPieceCost) * B;
    const int parts = total < NC ? static_cast<int>(total) : NC;
    auto cut = [&](int k, int& bk, int& prek) -> int {
      if (k >= parts) return T;
      const int64_t x = (static_cast<int64_t>(k) * total + parts - 1) / parts;  // cost(t) >= x
      int pre = 0;
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int bb = b0 + lane;
        const int n = bb < B ? bal_tiles<kTile>(p, bb) : 0;
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        const int excl = incl - n;
        const int64_t last = static_cast<int64_t>(pre) + incl - 1 +
                             static_cast<int64_t>(kPieceCost) * (bb + 1);
        const uint32_t hit = __ballot_sync(0xffffffffu, n > 0 && last >= x);
        if (hit) {
          const int l = __ffs(hit) - 1;
          bk = b0 + l;
          prek = pre + __shfl_sync(0xffffffffu, excl, l);
          const int64_t t = x - static_cast<int64_t>(kPieceCost) * (bk + 1);
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
  const int tg = wi % C::kTokGroups;  // S: token group
  const int kh = wi / C::kTokGroups;  // S: half of the 576-element reduction
  const int krow = C::kSTok == 16 ? tg * 16 + (lane & 7) + ((lane >> 4) << 3)
                                  : tg * 8 + (lane & 7);
  const int khalf = C::kSTok == 16 ? ((lane >> 3) & 1) : (lane >> 3);
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
      float* S = s_tile + (u & 1) * (C::kKSplit * HT * C::kSStride);
      uint64_t mask = 0;
      if (__all_sync(0xffffffffu, w_ok)) {
        mask = tile_mask[stage];
        // ---- S = Q . K^T for 16 heads x kSTok tokens over the 576 elements
        constexpr int NTS = C::kSTok / 8;
        float sacc[NTS][4], sacc2[1][4];  // sacc2: a second chain for 8-token blocks
#pragma unroll
        for (int nt = 0; nt < NTS; ++nt)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) sacc[nt][cc] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) sacc2[0][cc] = 0.f;
        constexpr int kSteps = kChunks * 4 / C::kKSplit;  // 16-wide k-steps per warp
#pragma unroll 3
        for (int kc = kh * kSteps; kc < (kh + 1) * kSteps; kc += 2) {
          const int ch = kc >> 2;
          const int j = kc & 3;  // k-steps j and j + 1 of chunk ch
          const uint32_t qreg = smem_base + ch * HT * 128;
          const uint32_t kreg = st_base + ch * C::kChunkBytes;
          if constexpr (C::kSTok == 16) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t a[4], bb[4];
              ldsm_x4(swz(qreg, qrow, 2 * (j + h2) + qhalf), a);
              ldsm_x4(swz(kreg, krow, 2 * (j + h2) + khalf), bb);
              mma_bf16_16816(sacc[0], a, bb[0], bb[1]);
              mma_bf16_16816(sacc[NTS - 1], a, bb[2], bb[3]);
            }
          } else {
            uint32_t a0[4], a1[4], bb[4];
            ldsm_x4(swz(qreg, qrow, 2 * j + qhalf), a0);
            ldsm_x4(swz(qreg, qrow, 2 * j + 2 + qhalf), a1);
            ldsm_x4(swz(kreg, krow, 2 * j + khalf), bb);
            mma_bf16_16816(sacc[0], a0, bb[0], bb[1]);
            mma_bf16_16816(sacc2[0], a1, bb[2], bb[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NTS; ++nt) {
          const int col = tg * C::kSTok + nt * 8 + 2 * tq;
          float* r0 = S + (kh * HT + 16 * mb + gq) * C::kSStride + col;
          float* r1 = r0 + 8 * C::kSStride;
          if constexpr (NTS == 1) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) sacc[nt][cc] += sacc2[0][cc];
          }
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
        float2 x0 = *reinterpret_cast<const float2*>(row);
        float2 x1 = *reinterpret_cast<const float2*>(row + 8);
        if constexpr (C::kKSplit == 2) {  // the other half of the reduction
          const float2 y0 = *reinterpret_cast<const float2*>(row + HT * C::kSStride);
          const float2 y1 = *reinterpret_cast<const float2*>(row + HT * C::kSStride + 8);
          x0 = make_float2(x0.x + y0.x, x0.y + y0.y);
          x1 = make_float2(x1.x + y1.x, x1.y + y1.y);
        }
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
        const int c_first = bal_chunk(pc.pre, b, total, parts);
        const int c_last = bal_chunk(pc.pre + pc.n - 1, b, total, parts);
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
    merge_pieces_cta<HT>(p, sched[7 + 3 * k], ht, sched[8 + 3 * k], sched[9 + 3 * k], total, parts,
                         reinterpret_cast<float*>(smem + C::kStageOff));
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
// chunks} (strides 1152 and 128 bytes): a box {64, box_rows, 9} lands as
// nine [box_rows x 128 B] chunk regions one after another, 128-byte
// swizzled, the layout the 2-D boxes build one chunk at a time.
bool make_row576_chunked_map(CUtensorMap* map, const void* base, int64_t rows,
                             int32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(kChunks)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes), 128u};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(kChunks)};
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
                                     : static_cast<int64_t>(ht == 16 ? MlaCfg<16>::kCtasPerSm : 1) *
                                           num_sms / (num_heads / ht);
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
  const int tile = ht == 128 ? mla_tc_tile() : ht == 64 ? MlaCfg<64>::kTile : MlaCfg<16>::kTile;
  const int32_t box_rows = a.block_size < tile ? a.block_size : tile;
  CUtensorMap mq, mkv;
  // mma.sync kernel: q_lat rows and, when a block covers a whole tile, the
  // latent tiles come as one 3-D box each (all nine 64-element chunks)
  const bool chunked_kv = ht != 128 && box_rows == tile;
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
  return ht == 64 ? launch_mla_split<64>(mq, mkv, p, grid, stream)
                  : launch_mla_split<16>(mq, mkv, p, grid, stream);
}

}  // namespace pa_detail
