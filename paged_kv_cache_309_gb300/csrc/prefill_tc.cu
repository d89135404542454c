// prefill_tc.cu -- causal varlen prefill attention over the paged cache on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What is computed (as prefill.cu): sequence b has n_b = cu_seqlens_q[b+1]
// - cu_seqlens_q[b] new tokens, the last n_b of its context_lens[b] = L_b
// cached tokens; new token j sits at position p = L_b - n_b + j and attends
// causally to tokens 0..p, read along the block table (nano-vLLM
// walkthrough, section 2.6; it names varlen flash prefill with
// cu_seqlens_q).  Query head h uses KV head h / G.
//
// How (sm_103a), FlashAttention style with the products on tcgen05:
//  * grid = (query tile, kv head, sequence), heaviest tiles first; a CTA owns
//    128 rows = 128/G new tokens x the G query heads of one kv head: the M
//    dimension of both products, one TMEM lane per row.
//  * warp 0 streams the key tiles (128 keys: K and V, each two 64-element
//    chunks of [128 rows x 128 B], 128-byte swizzled) through a 3-stage TMA
//    ring, one box per block piece, with a 128-bit row mask per tile.
//  * warp 1 owns TMEM and issues the products from one thread, whichever is
//    ready: S = Q.K^T (8 tcgen05.mma, M=128, N=128 keys, K=16; Q and K from
//    shared memory, K-major) into one of two 128-column score tiles, and
//    O += P.V (8 tcgen05.mma, N=128 head elements) with P (bf16) from TMEM
//    and V read in place as an MN-major operand.
//  * warps 2-9 load the CTA's Q rows into shared memory, then per tile read
//    scores (tcgen05.ld), apply the causal and validity masks, run an fp32
//    online softmax in base 2 with a lazy rescale (the running max moves
//    only when a score beats it by more than 2^8; the rescale reads, scales
//    and writes back the TMEM output row), and write the weights, rounded to
//    bf16, to TMEM (tcgen05.st).  Two warps share each TMEM lane quadrant,
//    one per half of the key columns (and of the output columns), and agree
//    on the row maximum through shared memory: each thread does 64 of its
//    row's 128 exponentials, and two warps per SM sub-partition hide each
//    other's TMEM and exponential latencies.  S of the next tile runs on the
//    tensor core while they work.
//  * TMEM: output 128 columns, two score tiles of 128, two weight tiles of 64.
// Every wait is bounded (2 s); a timeout sets an error bit, drains what was
// issued and frees TMEM before the CTA exits.
#include <atomic>

#include "pa_internal.cuh"
#include "tc_ops.cuh"

namespace pa_detail {
namespace {

using namespace pa;
using namespace tc;

constexpr int kD = 128;
constexpr int kM = 128;                        // rows per CTA (tokens x heads)
constexpr int kTile = 128;                     // keys per tile
constexpr int kStages = 3;
constexpr int kSoftmaxThreads = 8 * 32;         // two warps per TMEM lane quadrant
constexpr int kThreads = 4 * 32 + kSoftmaxThreads;
constexpr int kVWarp = 10;   // value loads (warp 0: key loads)
constexpr int kPVWarp = 11;  // P.V products (warp 1: score products, TMEM owner)
constexpr int kChunk = 128 * 128;              // 64 elements of 128 rows: 16 KB
constexpr int kQOff = 0;                       // Q: two chunks
constexpr int kStageOff = 2 * kChunk;          // per stage: K lo, K hi, V lo, V hi
constexpr int kStageBytes = 4 * kChunk;        // 64 KB
constexpr int kBarOff = kStageOff + kStages * kStageBytes;
// Row masks live in their own ring with their own barriers: the K slot of
// tile t is reloaded once S(t) is done, possibly before the softmax of tile
// t has read the mask (and its k_full phase may then have moved on); mask
// slot t % 8 is next written for tile t + 8, whose K load needs S(t + 5),
// which needs the softmax of tile t + 3 to have read its scores.
constexpr int kMaskSlots = 8;
// q_full, k_full[3], k_empty[3], v_full[3], v_empty[3], mask_full[8],
// s_full[2], s_empty[2], p_full[2], pv_done[2], o_final, drain[2]
constexpr int kNumBars = 12 + 4 * kStages + kMaskSlots;
constexpr int kMaskOff = kBarOff + kNumBars * 8;  // two 64-bit words per slot
constexpr int kMiscOff = kMaskOff + kMaskSlots * 16;
constexpr int kXchgOff = kMiscOff + 32;           // [2][kM] floats: pair exchange
constexpr int kBytes = kXchgOff + 2 * kM * 4;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;      // [0, 128): output
constexpr uint32_t kSCol = 128;    // [128, 384): two score tiles
constexpr uint32_t kPCol = 384;    // [384, 512): two weight tiles (bf16 pairs)
constexpr uint32_t kIdescS = instr_desc(kM, kTile, false);
constexpr uint32_t kIdescPV = instr_desc(kM, kD, true);
constexpr float kRescaleLog2 = 8.0f;

struct PrefillTcParams {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  unsigned* err;
  int64_t num_blocks;
  int32_t num_q_heads;
  int32_t group;
  int32_t tokens_per_cta;  // kM / group
  int32_t block_size;
  int32_t log2_bs;
  int32_t max_blocks_per_seq;
  float scale_log2;
};

// bit c of a tile's 128-bit row mask
__device__ __forceinline__ bool mask_bit(uint64_t lo, uint64_t hi, int c) {
  return ((c < 64 ? lo >> c : hi >> (c - 64)) & 1ull) != 0ull;
}

// Loads of the keys or the values of key tile t (warp 0, all lanes): lane
// i < nbox looks up block piece i; for the keys (mask_slot given) the lanes
// agree on the 128-bit row mask and lane 0 posts it; lane 0 posts the byte
// count and each lane with a valid piece issues its two boxes (64 head
// elements each).
__device__ __forceinline__ void issue_tile_half(const PrefillTcParams& p, const CUtensorMap* tm,
                                                uint8_t* dst, uint64_t* full, uint64_t* mask_slot,
                                                uint64_t* mask_bar, const int32_t* bt, int g,
                                                int tok0, int kend, uint64_t pol, int lane) {
  const int bs = p.block_size;
  const int rpb = bs < kTile ? bs : kTile;
  const int nbox = kTile / rpb;
  const int nval = min(kTile, kend - tok0);
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
  // rows of this piece as bits of the 128-bit mask (a piece never straddles
  // the two words unless it is the whole tile)
  uint64_t lo = 0, hi = 0;
  if (valid) {
    const int start = lane * rpb;
    const int r_lo = max(0, min(rows, 64 - start));
    const int r_hi = rows - r_lo;
    if (r_lo > 0) lo = (r_lo >= 64 ? ~0ull : ((1ull << r_lo) - 1ull)) << start;
    if (r_hi > 0) hi = (r_hi >= 64 ? ~0ull : ((1ull << r_hi) - 1ull)) << max(0, start - 64);
  }
  const uint32_t w0 = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(lo));
  const uint32_t w1 = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(lo >> 32));
  const uint32_t w2 = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(hi));
  const uint32_t w3 = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(hi >> 32));
  const uint32_t vb = __ballot_sync(0xffffffffu, valid);
  if (lane == 0) {
    if (mask_slot != nullptr) {
      mask_slot[0] = (static_cast<uint64_t>(w1) << 32) | w0;
      mask_slot[1] = (static_cast<uint64_t>(w3) << 32) | w2;
      mbar_arrive(mask_bar);
    }
    mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(vb) * rpb * 128 * 2));
  }
  __syncwarp();
  if (valid) {
    const int32_t row = bid * bs + row0;
    uint8_t* st = dst + lane * rpb * 128;
    tma_load_3d(st, tm, 0, g, row, full, pol);
    tma_load_3d(st + kChunk, tm, 64, g, row, full, pol);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v,
                                 const PrefillTcParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars + 0;                 // Q rows in shared memory (256 threads)
  uint64_t* k_full = bars + 1;                 // [kStages] keys of the tile landed
  uint64_t* k_empty = k_full + kStages;        // [kStages] S of the slot's tile done
  uint64_t* v_full = k_empty + kStages;        // [kStages] values of the tile landed
  uint64_t* v_empty = v_full + kStages;        // [kStages] P.V of the slot's tile done
  uint64_t* mask_full = v_empty + kStages;     // [kMaskSlots] row mask posted (1 thread)
  uint64_t* s_full = mask_full + kMaskSlots;   // [2] scores in TMEM (commit)
  uint64_t* s_empty = s_full + 2;              // [2] scores read (256 threads)
  uint64_t* p_full = s_empty + 2;              // [2] weights in TMEM (256 threads)
  uint64_t* pv_done = p_full + 2;              // [2] P.V done (commit)
  uint64_t* o_final = pv_done + 2;             // every product done (commit)
  uint64_t* drain = o_final + 1;               // [2] each issuer's products done
  uint64_t* tile_mask = reinterpret_cast<uint64_t*>(smem + kMaskOff);  // [kMaskSlots][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  int* flags = reinterpret_cast<int*>(smem + kMiscOff + 8);

  const int qtile = gridDim.x - 1 - blockIdx.x;  // latest positions first
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int n = __ldg(p.cu_seqlens_q + b + 1) - q0;
  int L = __ldg(p.context_lens + b);
  const int Lcap = p.max_blocks_per_seq * p.block_size;
  if (L > Lcap) {
    if (qtile == 0 && g == 0 && threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
    L = Lcap;
  }
  const int qt0 = qtile * p.tokens_per_cta;
  if (qt0 >= n) return;
  const int ntok = min(p.tokens_per_cta, n - qt0);
  const int pos0 = L - n + qt0;           // position of the CTA's first token
  const int kend = min(L, pos0 + ntok);   // keys 0 .. kend-1 are needed
  const int ntiles = kend > 0 ? (kend + kTile - 1) / kTile : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, kSoftmaxThreads);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < kMaskSlots; ++s) mbar_init(&mask_full[s], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kSoftmaxThreads);
      mbar_init(&p_full[s], kSoftmaxThreads);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_final, 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    flags[0] = 0;
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
  volatile int* abort_flag = flags;
  int issued = 0;  // (load warps) tiles whose keys / values were requested

  if (warp == 0 || warp == kVWarp) {
    // -------------------------------------------------------- TMA producers
    // Warp 0 loads the keys of tile t into K slot t % 3 once S of the slot's
    // previous tile is done and posts the tile's row mask; the V warp loads
    // the values into V slot t % 3 once P.V of the slot's previous tile is
    // done.  Each blocks in its own bounded wait (a suspended warp takes no
    // issue slots from the softmax warps).
    const bool is_k = warp == 0;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    uint64_t* empty = is_k ? k_empty : v_empty;
    uint64_t* full = is_k ? k_full : v_full;
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) prefetch_tensormap(tm);
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kStages;
      if (t >= kStages) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded_long(&empty[st], ((t / kStages) - 1) & 1, abort_flag));
        if (!ok) break;
      }
      issue_tile_half(p, tm, smem + kStageOff + st * kStageBytes + (is_k ? 0 : 2 * kChunk),
                      &full[st], is_k ? &tile_mask[2 * (t % kMaskSlots)] : nullptr,
                      is_k ? &mask_full[t % kMaskSlots] : nullptr, bt, g, t * kTile, kend, pol,
                      lane);
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1 || warp == kPVWarp) {
    // -------------------------------------------------------- MMA issuers
    // One thread of warp 1 issues the score products, one thread of the P.V
    // warp the output products; each commits its own products to their
    // barriers (a commit tracks the issuing thread's products).
    if (lane == 0) {
      const bool is_s = warp == 1;
      const uint32_t q_base = smem_u32(smem + kQOff);
      const uint32_t st_base = smem_u32(smem + kStageOff);
      bool ok = true;
      if (is_s) {
        ok = ntiles == 0 || mbar_wait_bounded(q_full, 0, abort_flag);
        tc_fence_after();
        for (int t = 0; ok && t < ntiles; ++t) {
          ok = mbar_wait_bounded_long(&k_full[t % kStages], (t / kStages) & 1, abort_flag) &&
               (t < 2 || mbar_wait_bounded_long(&s_empty[t & 1], ((t - 2) >> 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          // S(t) = Q . K(t)^T: 8 k-steps of 16 over the 128 head elements,
          // both operands K-major 128-byte swizzled (a k-step inside a chunk
          // advances the start by 32 bytes)
          const uint32_t kb = st_base + (t % kStages) * kStageBytes;
          const uint32_t d = tmem + kSCol + kTile * (t & 1);
#pragma unroll
          for (int j = 0; j < kD / 16; ++j)
            tc_mma_ss(d, smem_desc(q_base + (j >> 2) * kChunk + 32 * (j & 3), 16, 1024),
                      smem_desc(kb + (j >> 2) * kChunk + 32 * (j & 3), 16, 1024), kIdescS,
                      j > 0 ? 1u : 0u);
          tc_commit(&s_full[t & 1]);
          tc_commit(&k_empty[t % kStages]);
        }
      } else {
        for (int u = 0; ok && u < ntiles; ++u) {
          ok = mbar_wait_bounded_long(&p_full[u & 1], (u >> 1) & 1, abort_flag) &&
               mbar_wait_bounded_long(&v_full[u % kStages], (u / kStages) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          // O += P(u) . V(u): 8 k-steps of 16 keys; P from TMEM, V = chunks
          // 2,3 of the slot, MN-major (leading offset: next 64 elements =
          // next chunk; stride offset: next 8 keys = 1 KB)
          const uint32_t vb = st_base + (u % kStages) * kStageBytes + 2 * kChunk;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            tc_mma_ts(tmem + kOCol, tmem + kPCol + (kTile / 2) * (u & 1) + 8 * kk,
                      smem_desc(vb + kk * 2048, kChunk, 1024), kIdescPV,
                      (u > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&pv_done[u & 1]);
          tc_commit(&v_empty[u % kStages]);
        }
        if (ok) tc_commit(o_final);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
      }
      uint64_t* dr = is_s ? &drain[0] : &drain[1];
      tc_commit(dr);
      mbar_wait_bounded(dr, 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Two warps per TMEM lane quadrant: warp w reads lanes 32*(w & 3) ..
    // +31 (one row each) and, by h = (w - 2) / 4, key columns 64h .. 64h+63
    // of every score tile and output columns 64h .. 64h+63.  The pair agrees
    // on each row's tile maximum through shared memory; every wait that can
    // fail feeds the pair barrier's AND, so both warps leave together.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = 32 * quad + lane;  // = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * quad) << 16;
    const int pair_bar = 1 + quad;
    float* xchg = reinterpret_cast<float*>(smem + kXchgOff);  // [2 slots][kM rows]
    const int tok = row / G;
    const bool rvalid = tok < ntok;
    const int pos = pos0 + tok;
    const int64_t qrow =
        (static_cast<int64_t>(q0 + qt0 + (rvalid ? tok : 0)) * p.num_q_heads + g * G + row % G) *
        kD;
    // this half of the Q row -> shared memory chunk h (128-byte swizzle:
    // 16-byte unit u of row r at u ^ (r & 7)); padding rows are zeros
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow) + 8 * half;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 x = rvalid ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + kQOff + half * kChunk + row * 128 +
                                  ((u ^ (row & 7)) << 4)) = x;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    // The pair's exchange slots: at step t half h writes slot (t + h) & 1 and
    // reads the other one.  The next write to a slot comes either from the
    // warp that read it or after the following pair barrier, so one barrier
    // per step suffices.
    float m_run = -INFINITY, l_part = 0.f;  // l_part: this half's columns only
    const bool pos_scale = p.scale_log2 > 0.f;
    const float sc = pos_scale ? p.scale_log2 : 1.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      const int k = t & 1;
      bool w = ok && mbar_wait_bounded(&s_full[k], (t >> 1) & 1, abort_flag) &&
               mbar_wait_bounded(&mask_full[t % kMaskSlots], (t / kMaskSlots) & 1, abort_flag);
      w = __all_sync(0xffffffffu, w);
      float s[kTile / 2];
      float mx_part = -INFINITY;
      if (w) {
        tc_fence_after();
        tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k + 64 * half, &s[0]);
        tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k + 64 * half + 32, &s[32]);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_empty[k]);
        const uint64_t mw = tile_mask[2 * (t % kMaskSlots) + half];
        const int kc0 = t * kTile + 64 * half;  // position of this half's first key
        // with a positive scale the maximum is taken on the raw scores and
        // the scale folds into the exponent's argument; otherwise the scores
        // are scaled first
        if (!pos_scale) {
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] *= p.scale_log2;
        }
        // no mask needed when every key of the half exists and precedes the row
        if (!(rvalid && mw == ~0ull && kc0 + 63 <= pos)) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (!(rvalid && ((mw >> c) & 1ull) && kc0 + c <= pos)) s[c] = -INFINITY;
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          mq[0] = fmax3(mq[0], s[c], s[c + 1]);
          mq[1] = fmax3(mq[1], s[c + 2], s[c + 3]);
          mq[2] = fmax3(mq[2], s[c + 4], s[c + 5]);
          mq[3] = fmax3(mq[3], s[c + 6], s[c + 7]);
        }
        mx_part = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      }
      xchg[((t + half) & 1) * kM + row] = mx_part;
      if (!named_barrier_and(pair_bar, 64, w)) {
        ok = false;
        break;
      }
      // both halves take the same maximum (fmax is exact and commutative);
      // scaled to base-2 units (a scale of a masked -inf stays -inf)
      const float mx_raw = fmaxf(mx_part, xchg[((t + half + 1) & 1) * kM + row]);
      const float mx = pos_scale ? mx_raw * p.scale_log2 : mx_raw;
      // lazy rescale; tcgen05.ld/st are warp-wide, so the warp rescales
      // together when any of its rows needs it (the others scale by 1); the
      // two warps of a pair hold the same rows and decide alike
      const bool need = mx > m_run + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float corr = need ? fast_exp2(m_run - mx) : 1.f;
        if (t > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[(t - 1) & 1],
                                                         ((t - 1) >> 1) & 1, abort_flag));
          if (ok) {
            tc_fence_after();
            float o[64];
            tc_ld32_nowait(tmem + lane_addr + kOCol + 64 * half, &o[0]);
            tc_ld32_nowait(tmem + lane_addr + kOCol + 64 * half + 32, &o[32]);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 64; ++i) o[i] *= corr;
            tc_st32u_nowait(tmem + lane_addr + kOCol + 64 * half,
                            reinterpret_cast<const uint32_t*>(&o[0]));
            tc_st32u_nowait(tmem + lane_addr + kOCol + 64 * half + 32,
                            reinterpret_cast<const uint32_t*>(&o[32]));
            tc_wait_st();
          }
        }
        if (need) {
          l_part *= corr;
          m_run = mx;
        }
      }
      if (!ok) continue;  // the next pair barrier ends the loop for both warps
      // keys without a cache row: zero their V rows (0 x NaN would poison
      // P.V); piece j = (key j / 2, V chunk j % 2), one per thread
      const uint64_t mlo = tile_mask[2 * (t % kMaskSlots)];
      const uint64_t mhi = tile_mask[2 * (t % kMaskSlots) + 1];
      if (mlo != ~0ull || mhi != ~0ull) {
        // the values of tile t must have landed before rows are zeroed
        // (their slot's previous tile is then done with them as well)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&v_full[stage], (t / kStages) & 1,
                                                       abort_flag));
        if (!ok) continue;
        const int j = row + kM * half;
        const int r = j >> 1;
        if (!mask_bit(mlo, mhi, r)) {
          uint4* dst = reinterpret_cast<uint4*>(smem + kStageOff + stage * kStageBytes +
                                                (2 + (j & 1)) * kChunk + r * 128);
#pragma unroll
          for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // generic writes before the tensor core reads them
      }
      // the weight tile of tile t - 2 must have been consumed
      if (t >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[k], ((t - 2) >> 1) & 1,
                                                       abort_flag));
        if (!ok) continue;
      }
      // weights, rounded to bf16, as bf16 pairs in TMEM; the row sum of this
      // half in four independent chains
      // weight = 2^(s * scale - m): one paired multiply-add per two keys; a
      // masked score is -inf and 2^-inf = +0 (m is taken as 0 while the row
      // has seen no key, so the argument is never -inf + inf)
      const float2 sc2 = make_float2(sc, sc);
      const float mneg = m_run == -INFINITY ? 0.f : -m_run;
      const float2 mn2 = make_float2(mneg, mneg);
      float2 lq[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pr[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), sc2, mn2);
        const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        lq[i & 1] = fadd2(lq[i & 1], e);
        pr[i] = pack_bf16x2(e.x, e.y);
      }
      l_part += (lq[0].x + lq[0].y) + (lq[1].x + lq[1].y);
      tc_st32u_nowait(tmem + lane_addr + kPCol + (kTile / 2) * k + 32 * half, &pr[0]);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[k]);
    }
    // row sum: this half's part plus the partner's (one more exchange step)
    if (ok && ntiles > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_final, 0, abort_flag));
    xchg[((ntiles + half) & 1) * kM + row] = l_part;
    ok = named_barrier_and(pair_bar, 64, ok);
    const float l_run = l_part + xchg[((ntiles + half + 1) & 1) * kM + row];
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    } else if (ntiles == 0) {
      // no key at all: a zero row (this half's 64 columns)
      if (rvalid) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + qrow + 64 * half);
#pragma unroll
        for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
      // ---- epilogue: this half of the thread's output row
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int cq = 0; cq < 2; ++cq) {
        float o[32];
        tc_ld32(tmem + lane_addr + kOCol + 64 * half + 32 * cq, o);  // warp-wide
        if (rvalid) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + qrow + 64 * half + 32 * cq);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pack_bf16x2(o[8 * u] * inv, o[8 * u + 1] * inv),
                                pack_bf16x2(o[8 * u + 2] * inv, o[8 * u + 3] * inv),
                                pack_bf16x2(o[8 * u + 4] * inv, o[8 * u + 5] * inv),
                                pack_bf16x2(o[8 * u + 6] * inv, o[8 * u + 7] * inv));
        }
      }
    }
  }

  // ---- end: drain on error, free TMEM
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if ((warp == 0 || warp == kVWarp) && lane == 0) {
      uint64_t* full = warp == 0 ? k_full : v_full;
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait_bounded(&full[t % kStages], (t / kStages) & 1, nullptr);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

pa_status launch_paged_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.max_q_len == 0) return PA_OK;
  const int32_t G = a.num_q_heads / a.num_kv_heads;
  const int64_t rows = a.num_blocks * a.block_size;
  const int32_t box_rows = a.block_size < kTile ? a.block_size : kTile;
  CUtensorMap mk, mv;
  if (!make_kv_map_swizzled(&mk, a.k_cache, rows, a.num_kv_heads, box_rows) ||
      !make_kv_map_swizzled(&mv, a.v_cache, rows, a.num_kv_heads, box_rows))
    return PA_ERR_CUDA;
  PrefillTcParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.context_lens = a.context_lens;
  p.err = a.error_word;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.group = G;
  p.tokens_per_cta = kM / G;
  p.block_size = a.block_size;
  int lg = 0;
  while ((1 << lg) < a.block_size) ++lg;
  p.log2_bs = lg;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const int64_t qtiles = (static_cast<int64_t>(a.max_q_len) + p.tokens_per_cta - 1) / p.tokens_per_cta;
  if (qtiles > 0x7FFFFFFF) return PA_ERR_UNSUPPORTED;
  static std::atomic<bool> attr_set{false};
  if (!attr_set.load()) {
    if (cudaFuncSetAttribute(paged_prefill_tcgen05_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_set.store(true);
  }
  const dim3 grid(static_cast<unsigned>(qtiles), static_cast<unsigned>(a.num_kv_heads),
                  static_cast<unsigned>(a.num_seqs));
  paged_prefill_tcgen05_kernel<<<grid, kThreads, kAlloc, stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
