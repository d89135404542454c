// mla_decode_tc.cu -- MLA decode attention over the paged latent cache on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Same computation as mla_decode.cu (PagedAttention-principle post, MLA
// section; absorbed form): for sequence b and head h
//   s_j = scale * q_lat[b, h, :] . row_j (576 elements),
//   o_lat[b, h, :] = sum_j softmax(s)_j row_j[0:512],
// for head counts that are a multiple of 128.  With 128 heads per token the
// two products cost ~242 flops per byte of cache, about the GB300's
// flop/byte balance, so they belong on tcgen05 rather than mma.sync.
//
// Layout of the work (sm_103a):
//  * 128 heads are the M dimension of every product (one TMEM lane per
//    head).  The fp32 output of 128 heads x 512 elements would fill all 512
//    TMEM columns, so a CLUSTER of two CTAs serves each 128-head tile, and
//    CTA v (its rank in the cluster) owns one half of the row: latent
//    elements 256v .. 256v + 255 (its half of the output) and rope elements
//    32v .. 32v + 31.
//  * schedule: the sequences' 64-token tiles, laid end to end, are cut into
//    one contiguous chunk of equal cost per cluster (one wave of clusters;
//    each sequence start is charged 4 tiles); a chunk that crosses sequence
//    boundaries is worked piece by piece, a piece that is not a whole
//    sequence writes an fp32 partial, and the CTA completing a sequence's
//    pieces merges them after its own work.
//  * CTA v loads only its slice of every latent row (4 latent chunks of 128
//    bytes, 128-byte swizzled, and its 64 rope bytes, 64-byte swizzled: 576
//    of the row's 1152 bytes) through a 3-stage TMA ring of 36 KB.  Its
//    slice of q_lat sits in TMEM (latent part, bf16 pairs) and in shared
//    memory (rope part).
//  * partial S[128 x 64] over the CTA's 288 elements: 18 tcgen05.mma
//    (M=128, N=64, K=16).  The exchange threads (thread = head row) read
//    the 64 partial scores (tcgen05.ld), send them to the other CTA's
//    exchange buffer through distributed shared memory (st.async, counted
//    in bytes on the other CTA's mbarrier), add the other CTA's partials
//    and write the full scores back: both CTAs add the same two numbers, so
//    both run the identical softmax.  The softmax threads write the weights
//    (bf16) over the score buffer in TMEM.
//  * O[128 x 256] += P . V: 4 tcgen05.mma (N=256, K=16) with P from TMEM
//    and V = the CTA's latent chunks read in place as an MN-major operand.
//  * warp roles: warp 0 issues the TMA loads; one thread of warp 1 (the TMEM
//    owner) issues the score products and one thread of warp 6 the output
//    products, each blocking in bounded waits; warps 7-10 trade the partial
//    scores with the other CTA; warps 2-5 load q_lat and run the softmax:
//    fp32, base 2, lazy rescale (the running max moves only when a score
//    beats it by more than 2^8; the rescale reads, scales and writes back
//    the TMEM output row).
//  * epilogue of a piece: the softmax threads read their output row from
//    TMEM and write bf16 (whole sequence) or an fp32 partial + log2-sum-exp
//    (column-quad-major, so a warp's stores are 512 contiguous bytes).  The
//    next piece's q_lat is loaded before that epilogue, as soon as this
//    piece's last scores were read, so its score products overlap it.
//
// Every wait is bounded (2 s); a timeout sets an error bit, the roles leave
// their loops, the MMAs and copies already issued are drained, TMEM is
// freed, and the two CTAs meet at a cluster barrier before either exits.
#include <atomic>
#include <cmath>

#include "mla_common.cuh"
#include "tc_ops.cuh"

namespace pa_detail {
namespace {

using namespace pa;
using namespace mla;
using namespace tc;

constexpr int kHT = 128;               // heads per CTA (M)
constexpr int kTile = 64;              // tokens per tile (N of S, K of P.V)
constexpr int kHalf = kLat / 2;        // output (and latent) elements per CTA
constexpr int kRopeHalf = kRope / 2;   // rope elements per CTA
constexpr int kThreads = 11 * 32;
constexpr int kPVWarp = 6;   // P.V products (warp 1: score products, TMEM owner)
constexpr int kXWarp0 = 7;   // warps 7-10: score exchange with the other CTA
constexpr int kChunkBytes = kTile * 128;             // one 64-element chunk of a tile: 8 KB
constexpr int kLatChunks = kHalf / 64;               // 4 latent chunks per CTA
constexpr int kRopeTileBytes = kTile * kRopeHalf * 2;  // this CTA's 32 rope elements: 4 KB
constexpr int kStageBytes = kLatChunks * kChunkBytes + kRopeTileBytes;  // 36 KB
constexpr int kStages = 3;
constexpr int kRecvBytes = kTile * kHT * 4;          // one tile of the peer's partial scores
constexpr int kQRopeBytes = kHT * kRopeHalf * 2;     // this CTA's rope part of q_lat (64-byte rows)
constexpr int kStageOff = 0;
constexpr int kRecvOff = kStageOff + kStages * kStageBytes;
constexpr int kQRopeOff = kRecvOff + 2 * kRecvBytes;
constexpr int kBarOff = kQRopeOff + kQRopeBytes;
// barriers: q_full, kv_full[kStages], kv_empty[kStages], s_full[2],
// p_full[2], pv_done[2], recv_full[2], sent_free[2], o_done, drain[2],
// part_done, sum_full[2], mrg_full[kMrgBufs]; then tile masks, the TMEM
// slot and flags, the schedule
constexpr int kMrgBufs = 3;
constexpr int kNumBars = 17 + kMrgBufs + 2 * kStages;
constexpr int kMaskOff = kBarOff + kNumBars * 8;
constexpr int kMiscOff = kMaskOff + kStages * 8;
constexpr int kSchedOff = kMiscOff + 32;             // schedule words and the merge list
constexpr int kMaxMerges = 32;
constexpr int kBytes = kSchedOff + (8 + 3 * kMaxMerges) * 4;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "shared memory");

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;      // [0, 256): this CTA's half of the output
constexpr uint32_t kQCol = 256;    // [256, 384): this CTA's latent part of q_lat (bf16 pairs)
constexpr uint32_t kSCol = 384;    // [384, 512): two 64-column partial-score tiles

constexpr uint32_t kIdescS = instr_desc(kHT, kTile, false);
constexpr uint32_t kIdescPV = instr_desc(kHT, kHalf, true);

// ---------------------------------------------------------- cluster ops --
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// asynchronous 16-byte store into the other CTA's shared memory; its
// completion is counted (16 bytes) on that CTA's mbarrier `bar`
__device__ __forceinline__ void st_async_peer(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
      ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}
// arrival on the other CTA's barrier without release ordering: used where
// the only prior accesses to order are loads whose values are already in use
__device__ __forceinline__ void arrive_peer_relaxed(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait (2 s, or earlier once *abort_flag is set) for a phase whose
// arrivals come from the other CTA of the cluster
__device__ __forceinline__ bool wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                     volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
    }
  }
}
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Loads of one tile (one warp, all lanes): like mla_issue_tile_at, but only
// this CTA's slice: latent chunks 4v .. 4v + 3 into slots 0..3 of the stage
// (128-byte rows) and rope elements 32v .. 32v + 31 behind them (64-byte
// rows, 64-byte swizzle).
__device__ __forceinline__ void issue_half_tile(const MlaParams& p, const CUtensorMap* tm_kv,
                                                const CUtensorMap* tm_rope,
                                                uint8_t* stage, uint64_t* full,
                                                uint64_t* mask_slot, const int32_t* bt, int tok0,
                                                int tok_end, int v, uint64_t pol, int lane) {
  const int bs = p.block_size;
  const int rpb = bs < kTile ? bs : kTile;
  const int nbox = kTile / rpb;
  const int nval = min(kTile, tok_end - tok0);
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
    mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(vb) * rpb *
                                                      (kLatChunks * 128 + kRopeHalf * 2)));
  }
  __syncwarp();
  if (valid) {
    const int32_t row = bid * bs + row0;
    uint8_t* st = stage + lane * rpb * 128;
#pragma unroll 1
    for (int c = 0; c < kLatChunks; ++c)
      tma_load_2d(st + c * kChunkBytes, tm_kv, 64 * (kLatChunks * v + c), row, full, pol);
    tma_load_2d(stage + kLatChunks * kChunkBytes + lane * rpb * (kRopeHalf * 2), tm_rope,
                kLat + kRopeHalf * v, row, full, pol);
  }
}

// ------------------------------------------------------------- schedule --
// The work of one 128-head tile is the sequences' 64-token tiles laid end
// to end in sequence order (T tiles), cut into C contiguous chunks, one per
// cluster, of equal COST: tile t of sequence b sits at cost t + kPieceCost
// * (b + 1) (every sequence start is charged kPieceCost tiles: a cluster
// pays for each piece it starts a q_lat load, a pipeline drain and an
// epilogue), the cost line of length T + kPieceCost * B is cut into C equal
// parts (min(C, total) parts, so that each part spans at least one cost
// unit and no cluster inside a sequence's span is empty; the clusters past
// them get no work), and cluster(t) = floor(cost(t) * C / total) in closed
// form.  Where
// a chunk crosses a sequence boundary it splits into pieces.  A piece that
// covers its whole sequence writes bf16 output; the others write an fp32
// partial to a slot: 2c for a piece whose sequence began in an earlier
// cluster, 2c + 1 for one whose sequence begins in cluster c (a cluster has
// at most one of each), and the CTA that completes a sequence's count
// merges it.  Every CTA derives the schedule from context_lens itself.
constexpr int kPieceCost = 4;  // tiles
__device__ __forceinline__ int bal_cluster(int64_t t, int b, int64_t total, int C) {
  return static_cast<int>((t + static_cast<int64_t>(kPieceCost) * (b + 1)) * C / total);
}
__device__ __forceinline__ int seq_len_eff(const MlaParams& p, int b, bool* clipped) {
  int L = __ldg(p.context_lens + b);
  L = L < 0 ? 0 : L;
  const int64_t cap = static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size;
  *clipped = static_cast<int64_t>(L) > cap;
  return *clipped ? static_cast<int>(cap) : L;
}
__device__ __forceinline__ int seq_tiles(const MlaParams& p, int b) {
  bool c;
  return (seq_len_eff(p, b, &c) + kTile - 1) / kTile;
}
struct Piece {
  int b;       // sequence
  int tb, te;  // tile range [tb, te) of the sequence
  int pre;     // tiles of the sequences before b (position of its first tile)
  int n;       // tiles of the sequence
  bool first;  // the cluster's first piece
};
// Walks this cluster's chunk [g, g1) piece by piece (each role keeps its own).
struct PieceIter {
  int b, pre, g, g1;
  bool started;
  __device__ __forceinline__ bool next(const MlaParams& p, Piece& pc) {
    if (g >= g1) return false;
    int n = seq_tiles(p, b);
    while (pre + n <= g && b + 1 < p.num_seqs) {  // skips finished and empty sequences
      pre += n;
      ++b;
      n = seq_tiles(p, b);
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
__device__ __forceinline__ int piece_slot(const Piece& pc, int c) { return 2 * c + (pc.tb > 0 ? 0 : 1); }

// Merge of output half v of the 128 heads of (sequence b, head tile ht)
// over its pieces, by the whole CTA once its own work is done: the pieces
// are clusters c_first .. c_last; slot of the first one 2 c_first (+1 if it
// is not that cluster's first piece), of the others 2c.  Piece i gets weight
// 2^(lse_i - M) / sum_j 2^(lse_j - M) per head (M the heads' maximum).
// Partials are stored column-quad-major, [slot][half][quad][head] of float4
// (a warp's epilogue stores are then 512 contiguous bytes), so one group of
// kMrgQuads quads of all 128 heads of one piece is one contiguous 16 KB bulk
// copy.  Jobs are (group, batch of up to kMrgPieces pieces); up to kMrgBufs
// jobs are in flight, each buffer on its own barrier.  A thread sums
// (quad, head) pairs with the head fastest (conflict-free shared reads),
// the bf16 results go through a padded tile and leave as 64-byte row
// segments of the output.
constexpr int kMrgQuads = 8;                                // 32 columns per group
constexpr int kMrgGroups = kHalf / 4 / kMrgQuads;           // 8 groups per half row
constexpr int kMrgGroupBytes = kMrgQuads * kHT * 16;        // one piece's rows of a group
constexpr int kMrgPieces = 7;                               // pieces per batch
constexpr int kMrgStageBytes = 9 * kMrgGroupBytes;          // 144 KB of job buffers
constexpr int kMrgOutPitch = kMrgQuads * 8 + 16;            // bf16 tile row: 64 B + pad
constexpr int kMrgOutOff = kMrgStageBytes;
constexpr int kMrgWOff = kMrgOutOff + kHT * kMrgOutPitch;
constexpr int kMrgPairs = (kMrgQuads * kHT + kThreads - 1) / kThreads;  // pairs per thread
static_assert(kMrgWOff + (2 * kHT + kMrgPieces * kHT) * 4 <= kBarOff,
              "merge staging fits below the barriers");
// Merge of NP pieces by plain coalesced loads straight into registers: R
// column groups per round, so that R * NP 16-byte loads per (quad, head)
// pair are in flight per thread (the bulk copies above land at ~30-40 GB/s
// per SM whatever their number; this keeps ~100 KB of loads in flight).
// src(j) is piece j's partial half ([quad][head] float4), w its weights.
template <int NP, int R>
__device__ __forceinline__ void merge_direct(const MlaParams& p, const float4* const (&src)[NP],
                                             const float* wb, int64_t bh0, int v,
                                             uint8_t* otile) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int g0 = 0; g0 < kMrgGroups; g0 += R) {
    float4 x[R][kMrgPairs][NP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int u = 0; u < kMrgPairs; ++u) {
        const int idx = tid + nthr * u;
#pragma unroll
        for (int j = 0; j < NP; ++j)
          if (idx < kMrgQuads * kHT) x[r][u][j] = __ldcg(src[j] + (g0 + r) * kMrgQuads * kHT + idx);
      }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int g = g0 + r;
#pragma unroll
      for (int u = 0; u < kMrgPairs; ++u) {
        const int idx = tid + nthr * u;
        if (idx < kMrgQuads * kHT) {
          const int q = idx / kHT, h = idx % kHT;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            const float w = wb[j * kHT + h];
            a.x += w * x[r][u][j].x;
            a.y += w * x[r][u][j].y;
            a.z += w * x[r][u][j].z;
            a.w += w * x[r][u][j].w;
          }
          *reinterpret_cast<uint2*>(otile + h * kMrgOutPitch + q * 8) =
              make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
        }
      }
      __syncthreads();
      for (int idx = tid; idx < kHT * (kMrgQuads / 2); idx += nthr) {
        const int h = idx / (kMrgQuads / 2), c16 = idx % (kMrgQuads / 2);
        *reinterpret_cast<uint4*>(p.out + (bh0 + h) * kLat + kHalf * v + 4 * kMrgQuads * g +
                                  8 * c16) =
            *reinterpret_cast<const uint4*>(otile + h * kMrgOutPitch + 16 * c16);
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ void merge_pieces(const MlaParams& p, int b, int ht, int v, int pre,
                                             int n, int64_t total, int C, uint8_t* stage,
                                             uint64_t* bar, uint32_t* phase) {
  const int c_first = bal_cluster(pre, b, total, C);
  const int c_last = bal_cluster(pre + n - 1, b, total, C);
  const int np = c_last - c_first + 1;
  const int s0 = 2 * c_first + 1;  // the sequence begins in c_first, continues in the others
  auto slot = [&](int i) { return i == 0 ? s0 : 2 * (c_first + i); };
  const int64_t base = static_cast<int64_t>(ht) * p.num_slots;
  const int64_t bh0 = static_cast<int64_t>(b) * p.num_heads + ht * kHT;
  const int tid = threadIdx.x, nthr = blockDim.x;
  float* wsm = reinterpret_cast<float*>(stage + kMrgWOff);
  float* wmax = wsm;             // [kHT] per-head maximum of the pieces' lse
  float* winv = wsm + kHT;       // [kHT] 1 / sum of the weights
  float* wb = wsm + 2 * kHT;     // [kMrgPieces][kHT] weights of the current batch
  uint8_t* otile = stage + kMrgOutOff;
  for (int h = tid; h < kHT; h += nthr) {
    if (np <= kMrgPieces) {
      // every piece's lse in flight at once; the weights of all pieces here
      float l[kMrgPieces];
#pragma unroll
      for (int j = 0; j < kMrgPieces; ++j)
        l[j] = j < np ? __ldcg(p.ws_lse + (base + slot(j)) * kHT + h) : -INFINITY;
      float M = -INFINITY;
#pragma unroll
      for (int j = 0; j < kMrgPieces; ++j) M = fmaxf(M, l[j]);
      float W = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int j = 0; j < kMrgPieces; ++j) W += exp2f(l[j] - M);  // 2^-inf = 0 for padding
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      wmax[h] = M;
      winv[h] = inv;
#pragma unroll
      for (int j = 0; j < kMrgPieces; ++j)
        if (j < np) wb[j * kHT + h] = M == -INFINITY ? 0.f : exp2f(l[j] - M) * inv;
      continue;
    }
    float M = -INFINITY;
    for (int i0 = 0; i0 < np; i0 += 4) {
      float l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        l[j] = i0 + j < np ? __ldcg(p.ws_lse + (base + slot(i0 + j)) * kHT + h) : -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) M = fmaxf(M, l[j]);
    }
    float W = 0.f;
    if (M != -INFINITY) {
      for (int i0 = 0; i0 < np; i0 += 4) {
        float l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          l[j] = i0 + j < np ? __ldcg(p.ws_lse + (base + slot(i0 + j)) * kHT + h) : -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) W += exp2f(l[j] - M);  // 2^-inf = 0 for the padding
      }
    }
    wmax[h] = M;
    winv[h] = W > 0.f ? 1.f / W : 0.f;
  }
  fence_proxy_async_global();  // the partials were written by ordinary stores
  __syncthreads();
  if (np == 2 || np == 3) {
    const float4* srcs[3];
    for (int j = 0; j < np; ++j)
      srcs[j] = reinterpret_cast<const float4*>(p.ws_o + ((base + slot(j)) * 2 + v) * kHT * kHalf);
    if (np == 2) {
      const float4* const s2[2] = {srcs[0], srcs[1]};
      merge_direct<2, 2>(p, s2, wb, bh0, v, otile);
    } else {
      const float4* const s3[3] = {srcs[0], srcs[1], srcs[2]};
      merge_direct<3, 1>(p, s3, wb, bh0, v, otile);
    }
    return;
  }
  const int nbp = min(np, kMrgPieces);                      // pieces per batch
  const int nbatch = (np + nbp - 1) / nbp;
  const int njobs = kMrgGroups * nbatch;
  const int nbuf = min(kMrgBufs, kMrgStageBytes / (nbp * kMrgGroupBytes));
  auto issue = [&](int job) {  // thread 0: one batch of pieces of one group
    const int g = job / nbatch, i0 = (job % nbatch) * nbp;
    const int npb = min(nbp, np - i0);
    uint64_t* bb = &bar[job % nbuf];
    uint8_t* dst = stage + (job % nbuf) * nbp * kMrgGroupBytes;
    mbar_arrive_expect_tx(bb, static_cast<uint32_t>(npb * kMrgGroupBytes));
    for (int j = 0; j < npb; ++j)
      bulk_load(dst + j * kMrgGroupBytes,
                p.ws_o + ((base + slot(i0 + j)) * 2 + v) * kHT * kHalf +
                    static_cast<int64_t>(g) * kMrgQuads * kHT * 4,
                static_cast<uint32_t>(kMrgGroupBytes), bb);
  };
  if (tid == 0)
    for (int job = 0; job < min(nbuf, njobs); ++job) issue(job);
  float4 acc[kMrgPairs];
  for (int job = 0; job < njobs; ++job) {
    const int g = job / nbatch, bi = job % nbatch, i0 = bi * nbp;
    const int npb = min(nbp, np - i0);
    if (bi == 0) {
#pragma unroll
      for (int u = 0; u < kMrgPairs; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (np > kMrgPieces) {  // this batch's weights
      for (int idx = tid; idx < npb * kHT; idx += nthr) {
        const int j = idx / kHT, h = idx % kHT;
        const float M = wmax[h];
        const float l = __ldcg(p.ws_lse + (base + slot(i0 + j)) * kHT + h);
        wb[j * kHT + h] = M == -INFINITY ? 0.f : exp2f(l - M) * winv[h];
      }
      __syncthreads();
    }
    const int buf = job % nbuf;
    if (!mbar_wait_bounded(&bar[buf], phase[buf], nullptr) && tid == 0)
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    phase[buf] ^= 1u;
    const float4* src = reinterpret_cast<const float4*>(stage + buf * nbp * kMrgGroupBytes);
#pragma unroll
    for (int u = 0; u < kMrgPairs; ++u) {
      const int idx = tid + nthr * u;  // (quad, head), head fastest
      if (idx < kMrgQuads * kHT) {
        const int h = idx % kHT;
        for (int j = 0; j < npb; ++j) {
          const float4 x = src[j * (kMrgQuads * kHT) + idx];
          const float w = wb[(np > kMrgPieces ? j : i0 + j) * kHT + h];
          acc[u].x += w * x.x;
          acc[u].y += w * x.y;
          acc[u].z += w * x.z;
          acc[u].w += w * x.w;
        }
      }
    }
    __syncthreads();  // buffer `buf` (and this batch's weights) are free again
    if (tid == 0 && job + nbuf < njobs) issue(job + nbuf);
    if (bi + 1 == nbatch) {
      // group g done: bf16 through the padded tile, out as 64-byte row segments
#pragma unroll
      for (int u = 0; u < kMrgPairs; ++u) {
        const int idx = tid + nthr * u;
        if (idx < kMrgQuads * kHT) {
          const int q = idx / kHT, h = idx % kHT;
          *reinterpret_cast<uint2*>(otile + h * kMrgOutPitch + q * 8) =
              make_uint2(pack_bf16x2(acc[u].x, acc[u].y), pack_bf16x2(acc[u].z, acc[u].w));
        }
      }
      __syncthreads();
      for (int idx = tid; idx < kHT * (kMrgQuads / 2); idx += nthr) {
        const int h = idx / (kMrgQuads / 2), c16 = idx % (kMrgQuads / 2);
        *reinterpret_cast<uint4*>(p.out + (bh0 + h) * kLat + kHalf * v + 4 * kMrgQuads * g +
                                  8 * c16) =
            *reinterpret_cast<const uint4*>(otile + h * kMrgOutPitch + 16 * c16);
      }
      // the tile is rewritten only after the next job's barrier, which every
      // thread reaches after its share of this write-out
    }
  }
}

// ------------------------------------------------------------------ kernel --
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_kv,
                         const __grid_constant__ CUtensorMap tm_rope, const MlaParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars + 0;                   // q_lat of the current piece loaded (128 threads)
  uint64_t* kv_full = bars + 1;                  // [kStages] tile landed
  uint64_t* kv_empty = kv_full + kStages;        // [kStages] P.V of the stage's tile done
  uint64_t* s_full = kv_empty + kStages;         // [2] partial scores in TMEM (commit)
  uint64_t* p_full = s_full + 2;                 // [2] weights written over them (128 threads)
  uint64_t* pv_done = p_full + 2;                // [2] P.V done, score buffer free (commit)
  uint64_t* recv_full = pv_done + 2;             // [2] the other CTA's partials landed here
  uint64_t* sent_free = recv_full + 2;           // [2] the other CTA consumed what we sent
  uint64_t* o_done = sent_free + 2;              // every product of the current piece done
  uint64_t* drain = o_done + 1;                  // [2] each issuer's products done
  uint64_t* part_done = drain + 2;               // a partial's 128 rows are written
  uint64_t* sum_full = part_done + 1;            // [2] full scores back in TMEM (128 threads)
  uint64_t* mrg_full = sum_full + 2;             // [kMrgBufs] a merge batch's partial rows landed
  uint64_t* tile_mask = reinterpret_cast<uint64_t*>(smem + kMaskOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  int* flags = reinterpret_cast<int*>(smem + kMiscOff + 8);  // [0] abort
  int* sched = reinterpret_cast<int*>(smem + kSchedOff);      // T, -, g0, g1, b0, pre0, merges
  int* merges = sched + 8;                                    // (b, pre, n) per sequence to merge

  const int v = static_cast<int>(cluster_rank());  // output half = element slice
  const int c = blockIdx.x >> 1;                   // cluster = chunk of the tile list
  const int C = gridDim.x >> 1;
  const int ht = blockIdx.y;                       // 128-head tile
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h0 = ht * kHT;
  const int B = p.num_seqs;

  // ---- schedule (warp 0): total tiles, this cluster's chunk, its first sequence
  if (warp == 0) {
    // tiles per sequence: up to 32 * kR sequences in registers (their loads
    // in flight together), which the two cuts below then read
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
          nreg[r] = (seq_len_eff(p, 32 * r + lane, &cl) + kTile - 1) / kTile;
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
          n = (seq_len_eff(p, b0 + lane, &cl) + kTile - 1) / kTile;
          any_clip |= cl;
        }
        T += static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(n)));
      }
    }
    if (__any_sync(0xffffffffu, any_clip) && c == 0 && ht == 0 && v == 0 && lane == 0)
      atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
    // first tile of cluster k: the smallest t with cost(t) * C >= k * total,
    // found in the first non-empty sequence whose last tile reaches that
    // cost (T when none does); also that sequence and its first tile
    const int64_t total = static_cast<int64_t>(T) + static_cast<int64_t>(kPieceCost) * B;
    const int Ce = total < C ? static_cast<int>(total) : C;  // parts of the cost line
    auto cut = [&](int k, int& bk, int& prek) -> int {
      if (k >= Ce) return T;
      const int64_t x = (static_cast<int64_t>(k) * total + Ce - 1) / Ce;  // cost(t) >= x
      int pre = 0;
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int bb = b0 + lane;
        int n = 0;
        if (in_regs) {
#pragma unroll
          for (int r = 0; r < kR; ++r) n = 32 * r == b0 ? nreg[r] : n;  // selects, no local array
        } else {
          n = bb < B ? seq_tiles(p, bb) : 0;
        }
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
    }
  }
  if (threadIdx.x == 64) {  // (warp 0 computes the schedule, warp 1 allocates TMEM)
    mbar_init(q_full, kHT);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], kHT);
      mbar_init(&pv_done[s], 1);
      mbar_init(&recv_full[s], 1);   // armed with the byte count by this CTA
      mbar_init(&sent_free[s], 4);   // one arrival per softmax warp of the other CTA
    }
    mbar_init(o_done, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(part_done, kHT);
    for (int i = 0; i < kMrgBufs; ++i) mbar_init(&mrg_full[i], 1);
    mbar_init(&sum_full[0], kHT);
    mbar_init(&sum_full[1], kHT);
    flags[0] = 0;
    mbar_init_fence();
    // the first two exchanges: expect one tile of partials in each buffer
    mbar_arrive_expect_tx(&recv_full[0], kRecvBytes);
    mbar_arrive_expect_tx(&recv_full[1], kRecvBytes);
  }
  if (warp == 1) {  // this warp owns the CTA's tensor memory
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either arrives on the other's
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort_flag = flags;
  const int g0 = sched[2], g1 = sched[3];
  const int64_t total = static_cast<int64_t>(sched[0]) + static_cast<int64_t>(kPieceCost) * B;
  const int Ce = total < C ? static_cast<int>(total) : C;  // clusters with work
  const int ntotal = g1 - g0;  // tiles of this cluster
  const PieceIter it0{sched[4], sched[5], g0, g1, false};
  const uint32_t peer = static_cast<uint32_t>(v ^ 1);

  // sequences without tokens: zero output rows (cluster c takes b = c mod C)
  for (int b = c; b < B; b += C) {
    if (seq_tiles(p, b) != 0) continue;
    for (int i = threadIdx.x; i < kHT * (kHalf / 8); i += kThreads) {
      const int h = i / (kHalf / 8), e = i % (kHalf / 8);
      reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * p.num_heads + h0 + h) * kLat +
                               kHalf * v)[e] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  int issued = 0;

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    const uint64_t pol = l2_policy_evict_first();  // each row is read once (the rope chunk twice)
    if (lane == 0) {
      prefetch_tensormap(&tm_kv);
      prefetch_tensormap(&tm_rope);
    }
    bool ok = true;
    PieceIter it = it0;
    Piece pc;
    int gt = 0;
    while (ok && it.next(p, pc)) {
      const int32_t* bt = p.block_tables + static_cast<int64_t>(pc.b) * p.max_blocks_per_seq;
      bool cl;
      const int L = seq_len_eff(p, pc.b, &cl);
      for (int tl = pc.tb; tl < pc.te; ++tl, ++gt) {
        const int stage = gt % kStages;
        if (gt >= kStages) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&kv_empty[stage],
                                                         ((gt / kStages) - 1) & 1, abort_flag));
          if (!ok) break;
        }
        issue_half_tile(p, &tm_kv, &tm_rope, smem + kStageOff + stage * kStageBytes, &kv_full[stage],
                        &tile_mask[stage], bt, tl * kTile, L, v, pol, lane);
        issued = gt + 1;
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1 || warp == kPVWarp) {
    // -------------------------------------------------------- MMA issuers
    // One thread of warp 1 issues the score products, one thread of the P.V
    // warp the output products; each blocks in its own bounded waits and
    // commits its own products (a commit tracks the issuing thread's).
    if (lane == 0) {
      const bool is_s = warp == 1;
      const uint32_t st_base = smem_u32(smem + kStageOff);
      const uint32_t qr_base = smem_u32(smem + kQRopeOff);
      PieceIter itr = it0;
      Piece pcr;
      bool ok = true;
      int t = 0;    // this cluster's tile counter
      int kp = 0;   // piece ordinal
      while (ok && itr.next(p, pcr)) {
        for (int tl = pcr.tb; tl < pcr.te && ok; ++tl, ++t) {
          if (is_s) {
            // partial S(t) = Q_v . K_v(t)^T over this CTA's 288 elements:
            // 16 latent k-steps with A = q_lat latent part in TMEM and B =
            // chunk slots 0..3 (K-major, 128-byte swizzle: a k-step advances
            // the start by 32 bytes inside a 64-element chunk), then 2 rope
            // k-steps with A = the rope part of q_lat and B = the stage's
            // rope rows (both K-major 64-byte rows, 64-byte swizzle).  Score
            // buffer t & 1 is free once P.V(t - 2), which read the weights
            // written over it, is done.  A piece's first tile waits for that
            // piece's q_lat.
            ok = (tl != pcr.tb || mbar_wait_bounded_long(q_full, kp & 1, abort_flag)) &&
                 mbar_wait_bounded_long(&kv_full[t % kStages], (t / kStages) & 1, abort_flag) &&
                 (t < 2 || mbar_wait_bounded_long(&pv_done[t & 1], ((t - 2) >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const uint32_t kb = st_base + (t % kStages) * kStageBytes;
            const uint32_t d = tmem + kSCol + kTile * (t & 1);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              tc_mma_ts(d, tmem + kQCol + 8 * i,
                        smem_desc(kb + (i >> 2) * kChunkBytes + 32 * (i & 3), 16, 1024), kIdescS,
                        i > 0 ? 1u : 0u);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              tc_mma_ss(d, smem_desc(qr_base + 32 * i, 16, 512, kSwizzle64),
                        smem_desc(kb + kLatChunks * kChunkBytes + 32 * i, 16, 512, kSwizzle64),
                        kIdescS, 1u);
            tc_commit(&s_full[t & 1]);
          } else {
            // O[:, this half] += P(t) . V(t): P = the bf16 weights in TMEM
            // (pairs, written over the score buffer; 8 columns per 16
            // tokens), V = slots 0..3 of tile t, MN-major (leading offset:
            // next 64 elements = next slot; stride offset: next 8 tokens =
            // 1 KB).  The first tile of a piece starts the output afresh;
            // after a piece's last tile, o_done tells the softmax its output
            // is complete.
            ok = mbar_wait_bounded_long(&p_full[t & 1], (t >> 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint32_t vb = st_base + (t % kStages) * kStageBytes;
            const uint32_t pcol = tmem + kSCol + kTile * (t & 1);
            const bool fresh = tl == pcr.tb;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              tc_mma_ts(tmem + kOCol, pcol + 8 * kk,
                        smem_desc(vb + kk * 2048, kChunkBytes, 1024), kIdescPV,
                        (!fresh || kk > 0) ? 1u : 0u);
            tc_commit(&pv_done[t & 1]);
            tc_commit(&kv_empty[t % kStages]);
            if (tl + 1 == pcr.te) tc_commit(o_done);
          }
        }
        ++kp;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
      }
      // every product issued completes before tensor memory is freed
      uint64_t* dr = is_s ? &drain[0] : &drain[1];
      tc_commit(dr);
      mbar_wait_bounded(dr, 0, nullptr);
    }
    __syncwarp();
  } else if (warp >= kXWarp0) {
    // -------------------------------------------------------- score exchange
    // Warps 7-10 (one per TMEM lane quadrant) trade partial scores with the
    // other CTA, tile by tile and ahead of the softmax: read this CTA's
    // partial S(u) (u counts this cluster's tiles), send it into the other
    // CTA's exchange buffer u & 1 once that CTA has consumed what we sent two
    // tiles ago (asynchronous stores counted in bytes on its recv_full[u &
    // 1]), add the other CTA's partial from our buffer u & 1 (own + other is
    // the same sum on both CTAs: addition commutes, so both run an identical
    // softmax), and write the full scores back over the partials.  Layout of
    // an exchange buffer: [4-token group][row] of float4, so a warp's 16-byte
    // stores are contiguous.
    const int row = 32 * (warp & 3) + lane;  // head within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t recv_peer = peer_addr(smem_u32(smem + kRecvOff), peer);
    const uint32_t recv_full_peer = peer_addr(smem_u32(recv_full), peer);
    const uint32_t sent_free_peer = peer_addr(smem_u32(sent_free), peer);
    bool ok = true;
    for (int u = 0; u < ntotal; ++u) {
      const int k = u & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded_long(&s_full[k], (u >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float sp[kTile];
      tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k, &sp[0]);
      tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k + 32, &sp[32]);
      tc_wait_ld();
      if (u >= 2) {
        ok = __all_sync(0xffffffffu, wait_cluster_bounded(&sent_free[k], ((u - 2) >> 1) & 1,
                                                          abort_flag));
        if (!ok) break;
      }
      const uint32_t slot = static_cast<uint32_t>((k * (kTile / 4) * kHT + row) * 16);
#pragma unroll
      for (int g = 0; g < kTile / 4; ++g)
        st_async_peer(recv_peer + slot + g * kHT * 16,
                      make_float4(sp[4 * g], sp[4 * g + 1], sp[4 * g + 2], sp[4 * g + 3]),
                      recv_full_peer + 8 * k);
      ok = __all_sync(0xffffffffu, wait_cluster_bounded(&recv_full[k], (u >> 1) & 1, abort_flag));
      if (!ok) break;
      const float4* other =
          reinterpret_cast<const float4*>(smem + kRecvOff) + k * (kTile / 4) * kHT + row;
#pragma unroll
      for (int g = 0; g < kTile / 4; ++g) {
        const float4 o = other[g * kHT];
        sp[4 * g] += o.x;
        sp[4 * g + 1] += o.y;
        sp[4 * g + 2] += o.z;
        sp[4 * g + 3] += o.w;
      }
      // buffer k is consumed (the values are in registers): re-arm it for
      // tile u + 2 and tell the other CTA
      __syncwarp();
      if (row == 0 && u + 2 < ntotal) mbar_arrive_expect_tx(&recv_full[k], kRecvBytes);
      if (lane == 0) arrive_peer_relaxed(sent_free_peer + 8 * k);
      tc_st32u_nowait(tmem + lane_addr + kSCol + kTile * k, reinterpret_cast<const uint32_t*>(&sp[0]));
      tc_st32u_nowait(tmem + lane_addr + kSCol + kTile * k + 32,
                      reinterpret_cast<const uint32_t*>(&sp[32]));
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&sum_full[k]);
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = 32 * (warp & 3) + lane;  // head within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    bool ok = true;
    PieceIter it = it0;
    Piece pc;
    int gbase = 0;    // this cluster's tiles before the current piece
    int npiece = 0;   // pieces done
    int npart = 0;    // partial pieces done
    // this CTA's slice of a piece's q_lat: latent elements 256v .. 256v + 255
    // as bf16 pairs in TMEM, rope elements 32v .. 32v + 31 in shared memory
    // (64-byte swizzle).  Called once every score product of the previous
    // piece is done (its last scores were read), so both may be overwritten:
    // the next piece's score products start while this piece's last output
    // products and its epilogue run.
    auto load_q = [&](const Piece& q) {
      const int64_t qbh = static_cast<int64_t>(q.b) * p.num_heads + h0 + row;
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_latent + qbh * kRow);
        // the whole slice in one global round trip (4 x 64 latent elements
        // = 128 columns, and the rope part)
        uint4 rope[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) rope[u] = __ldg(src + (kLat + kRopeHalf * v) / 8 + u);
        uint32_t w[128];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const uint4 x = __ldg(src + (kHalf * v) / 8 + u);
          w[4 * u] = x.x;
          w[4 * u + 1] = x.y;
          w[4 * u + 2] = x.z;
          w[4 * u + 3] = x.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) tc_st32u_nowait(tmem + lane_addr + kQCol + 32 * j, &w[32 * j]);
        tc_wait_st();
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(smem + kQRopeOff + row * 64 + ((u ^ ((row >> 1) & 3)) << 4)) =
              rope[u];
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(q_full);
      }
    };
    // the next piece's slice of q_lat into L2 while this piece runs
    auto prefetch_q = [&](const Piece& q) {
      const char* src = reinterpret_cast<const char*>(
          p.q_latent + (static_cast<int64_t>(q.b) * p.num_heads + h0 + row) * kRow);
#pragma unroll
      for (int u = 0; u < 4; ++u) prefetch_l2(src + kHalf * 2 * v + 128 * u);
      prefetch_l2(src + (kLat + kRopeHalf * v) * 2);
    };
    bool have = it.next(p, pc);
    if (have) load_q(pc);
    while (ok && have) {
      const int64_t bh = static_cast<int64_t>(pc.b) * p.num_heads + h0 + row;
      PieceIter it_next = it;
      Piece nx;
      const bool has_next = it_next.next(p, nx);
      if (has_next) prefetch_q(nx);
      const int n = pc.te - pc.tb;
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < n && ok; ++t) {
        const int gt = gbase + t;
        const int stage = gt % kStages;
        const int k = gt & 1;
        // ---- the full scores of tile gt (summed by the exchange warps), and
        // the tile itself, whose row mask is read here
        const bool w = mbar_wait_bounded(&sum_full[k], (gt >> 1) & 1, abort_flag) &&
                       mbar_wait_bounded(&kv_full[stage], (gt / kStages) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[kTile];
        tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k, &s[0]);
        tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k + 32, &s[32]);
        tc_wait_ld();
        const uint64_t mask = tile_mask[stage];
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
        for (int i = 0; i < kTile; ++i) {
          s[i] = ((mask >> i) & 1ull) ? s[i] * p.scale_log2 : -INFINITY;
          mq[i & 3] = fmaxf(mq[i & 3], s[i]);
        }
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        // lazy rescale; tcgen05.ld/st are warp-wide, so the warp rescales
        // together when any of its rows needs it (the others scale by 1)
        const bool need = mx > m_run + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float corr = need ? fast_exp2(m_run - mx) : 1.f;
          if (t > 0) {
            // the output row holds this piece's P.V up to tile gt - 1: wait for it
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[(gt - 1) & 1],
                                                           ((gt - 1) >> 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int cq = 0; cq < kHalf / 32; ++cq) {
              float o[32];
              tc_ld32(tmem + lane_addr + kOCol + 32 * cq, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= corr;
              tc_st32(tmem + lane_addr + kOCol + 32 * cq, o);
            }
          }
          if (need) {
            l_run *= corr;
            m_run = mx;
          }
        }
        uint32_t pr[kTile / 2];
        float lq[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains
#pragma unroll
        for (int i = 0; i < kTile / 2; ++i) {
          // a masked score is -inf and m_run is finite once a token was seen
          const float p0 = s[2 * i] == -INFINITY ? 0.f : fast_exp2(s[2 * i] - m_run);
          const float p1 = s[2 * i + 1] == -INFINITY ? 0.f : fast_exp2(s[2 * i + 1] - m_run);
          lq[i & 3] += p0 + p1;
          pr[i] = pack_bf16x2(p0, p1);
        }
        l_run += (lq[0] + lq[1]) + (lq[2] + lq[3]);
        // tokens that do not exist: zero their value rows (slots 0..3; 0 x NaN
        // would poison P.V); piece j = (token j / 4, slot j % 4), two per thread
        if (mask != ~0ull) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int j = row + kHT * hh;
            const int r = j >> 2;
            if (!((mask >> r) & 1ull)) {
              uint4* dst = reinterpret_cast<uint4*>(smem + kStageOff + stage * kStageBytes +
                                                    (j & 3) * kChunkBytes + r * 128);
#pragma unroll
              for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();  // generic writes before the tensor core reads them
        }
        // weights, as bf16 pairs, over this tile's score buffer in TMEM (the
        // scores are in registers): the A operand of P.V(gt)
        tc_st32u_nowait(tmem + lane_addr + kSCol + kTile * k, pr);
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[k]);
      }
      if (!ok) break;
      gbase += n;
      // every score product of this piece is done: the next piece's q_lat
      // goes in now, ahead of this piece's epilogue
      if (has_next) load_q(nx);
      // ---- epilogue of the piece: this thread's output row, elements
      // 256v .. 256v + 255; bf16 when the piece is its whole sequence, else an
      // fp32 partial in the piece's slot (and its log2-sum-exp)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_done, npiece & 1, abort_flag));
      if (!ok) break;
      ++npiece;
      tc_fence_after();
      const bool whole = pc.tb == 0 && pc.te == pc.n;
      const int64_t slot = static_cast<int64_t>(ht) * p.num_slots + piece_slot(pc, c);
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int cq = 0; cq < kHalf / 32; ++cq) {
        float o[32];
        tc_ld32(tmem + lane_addr + kOCol + 32 * cq, o);
        if (whole) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + bh * kLat + kHalf * v + 32 * cq);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pack_bf16x2(o[8 * u] * inv, o[8 * u + 1] * inv),
                                pack_bf16x2(o[8 * u + 2] * inv, o[8 * u + 3] * inv),
                                pack_bf16x2(o[8 * u + 4] * inv, o[8 * u + 5] * inv),
                                pack_bf16x2(o[8 * u + 6] * inv, o[8 * u + 7] * inv));
        } else {
          // partials are column-quad-major, [slot][half][quad][head] of
          // float4: the warp's 32 rows of one quad are 512 contiguous bytes
          float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * 2 + v) * kHT * kHalf) + row;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[(8 * cq + u) * kHT] = make_float4(o[4 * u] * inv, o[4 * u + 1] * inv,
                                                  o[4 * u + 2] * inv, o[4 * u + 3] * inv);
        }
      }
      if (!whole) {
        // both halves write the (identical) log2-sum-exp, each for its own merge
        p.ws_lse[slot * kHT + row] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
        // count this CTA's part once its 128 rows are written; the CTA
        // completing the pieces of b for its half merges that half after its
        // own work
        mbar_arrive(part_done);
        if (row == 0) {
          if (!mbar_wait_bounded(part_done, npart & 1, abort_flag)) {
            *abort_flag = 1;
            atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
          }
          __threadfence();
          const int np = bal_cluster(pc.pre + pc.n - 1, pc.b, total, Ce) -
                         bal_cluster(pc.pre, pc.b, total, Ce) + 1;
          // one count per output half: the CTA completing half v merges half v
          unsigned* ctr = p.counters + (static_cast<int64_t>(pc.b) * gridDim.y + ht) * 2 + v;
          const unsigned prev = atomicAdd(ctr, 1u);
          if (prev + 1u == static_cast<unsigned>(np)) {
            atomicExch(ctr, 0u);
            __threadfence();
            const int m = sched[6];
            if (m < kMaxMerges) {
              merges[3 * m] = pc.b;
              merges[3 * m + 1] = pc.pre;
              merges[3 * m + 2] = pc.n;
              sched[6] = m + 1;
            }
          }
        }
        ++npart;
      }
      it = it_next;
      pc = nx;
      have = has_next;
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  }

  // ---- end: drain on error, free TMEM, leave the cluster together, merge
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait_bounded(&kv_full[t % kStages], (t / kStages) & 1, nullptr);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  // neither CTA leaves while the other may still write into its shared memory
  cluster_sync_all();
  const int nm = sched[6];
  uint32_t mrg_phase[kMrgBufs] = {};
  for (int i = 0; i < nm; ++i)
    merge_pieces(p, merges[3 * i], ht, v, merges[3 * i + 1], merges[3 * i + 2], total, Ce,
                 smem + kStageOff, mrg_full, mrg_phase);
}

}  // namespace

int mla_tc_tile() { return kTile; }

pa_status launch_mla_tc(const CUtensorMap& mrope, const CUtensorMap& mkv, const MlaParams& p,
                        dim3 grid, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_raised{0};
  if (!ensure_smem_limit(mla_decode_tc_kernel, kAlloc, smem_raised)) return PA_ERR_CUDA;
  mla_decode_tc_kernel<<<grid, kThreads, kAlloc, stream>>>(mkv, mrope, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
