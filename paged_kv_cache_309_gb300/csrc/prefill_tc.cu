// prefill_tc.cu -- causal varlen prefill attention over the paged cache on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What is computed: sequence b has n_b = cu_seqlens_q[b+1]
// - cu_seqlens_q[b] new tokens, the last n_b of its context_lens[b] = L_b
// cached tokens; new token j sits at position p = L_b - n_b + j and attends
// causally to tokens 0..p, read along the block table (nano-vLLM
// walkthrough, section 2.6; it names varlen flash prefill with
// cu_seqlens_q).  Query head h uses KV head h / G.
//
// How (sm_103a), FlashAttention style with the products on tcgen05:
//  * grid = (query tile pair, kv head, sequence), heaviest first; a CTA owns
//    TWO query tiles of 128 rows (128/G consecutive new tokens x the G
//    query heads of one kv head each), which share every key/value tile:
//    half the L2 reads and TMA boxes per flop of one tile per CTA, and the
//    two tiles' softmax and products interleave.
//  * TMEM (512 columns): outputs O0, O1 (128 each) and score tiles S0, S1
//    (128 each); tile i's weights (bf16 pairs) are written over the upper
//    half of S_i, so S_i(t+1) waits for P.V_i(t).
//  * warp 0 loads the keys of tile t (two 64-element chunks of [128 rows x
//    128 B], 128-byte swizzled, one box per block piece) into a 3-slot ring
//    and posts its 128-bit row mask in an 8-slot ring; warp 2 loads the
//    values into a 2-slot ring; one thread of warp 1 (the TMEM owner)
//    issues S_i(t) = Q_i . K(t)^T (8 tcgen05.mma, N = 128 keys, K-major Q and
//    K), one thread of warp 3 issues O_i += P_i(t) . V(t) (8 tcgen05.mma,
//    P from TMEM, V read in place as an MN-major operand); each role blocks
//    in its own bounded waits.
//  * warps 4-7 run the softmax of query tile 0, warps 8-11 that of tile 1:
//    one thread per row (its TMEM lane), all 128 keys.  Pass 1 reads the
//    row's scores in two 64-column halves for the maximum (the upper half
//    stays in registers); pass 2 turns the upper half and then the re-read
//    lower half into weights, 2^(s * scale - m) by one paired FMA per two
//    keys and ex2.approx, written as bf16 pairs over score columns already
//    read.  fp32 online softmax in base 2 with a lazy rescale (the running
//    max moves only when a score beats it by more than 2^8).
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
constexpr int kM = 128;                        // rows per query tile (tokens x heads)
constexpr int kQTiles = 2;                     // query tiles per CTA
constexpr int kTile = 128;                     // keys per tile
constexpr int kKSlots = 3;                     // key ring
constexpr int kVSlots = 2;                     // value ring
constexpr int kThreads = 12 * 32;              // 4 role warps + 2 x 4 softmax warps
constexpr int kChunk = 128 * 128;              // 64 elements of 128 rows: 16 KB
constexpr int kQOff = 0;                       // Q tile i: two chunks at 2i, 2i+1
constexpr int kKOff = kQTiles * 2 * kChunk;    // key slots: lo, hi chunks
constexpr int kVOff = kKOff + kKSlots * 2 * kChunk;  // value slots: lo, hi chunks
constexpr int kBarOff = kVOff + kVSlots * 2 * kChunk;
// Row masks live in their own ring with their own barriers: the key slot of
// tile t is refilled once S_0(t) and S_1(t) are done, possibly before the
// softmax of tile t has read the mask; mask slot t % 8 is next written for
// tile t + 8, whose keys need S(t + 5), which needs P.V(t + 4), which needs
// both softmax groups past tile t + 4.
constexpr int kMaskSlots = 8;
// q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], mask_full[8],
// s_full[2], p_full[2], pv_done[2], o_final[2], drain[2], hand[2][4]
constexpr int kNumBars = 1 + 2 * kKSlots + 2 * kVSlots + kMaskSlots + 5 * kQTiles + 2 * 4;
constexpr int kMaskOff = kBarOff + kNumBars * 8;  // two 64-bit words per slot
constexpr int kMiscOff = kMaskOff + kMaskSlots * 16;
constexpr int kBytes = kMiscOff + 32;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;      // [0, 256): outputs O0, O1
constexpr uint32_t kSCol = 256;    // [256, 512): score tiles S0, S1 (weights over their upper halves)
constexpr uint32_t kPHalf = 64;    // weights of tile i at kSCol + 128 i + 64
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
  int32_t tokens_per_tile;  // kM / group
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
  uint64_t* q_full = bars + 0;                   // both Q tiles in shared memory (256 threads)
  uint64_t* k_full = bars + 1;                   // [kKSlots] keys of the tile landed
  uint64_t* k_empty = k_full + kKSlots;          // [kKSlots] S_0 and S_1 of the slot's tile done
  uint64_t* v_full = k_empty + kKSlots;          // [kVSlots] values of the tile landed
  uint64_t* v_empty = v_full + kVSlots;          // [kVSlots] P.V_0 and P.V_1 of the slot's tile done
  uint64_t* mask_full = v_empty + kVSlots;       // [kMaskSlots] row mask posted (1 thread)
  uint64_t* s_full = mask_full + kMaskSlots;     // [2] S_i in TMEM (commit)
  uint64_t* p_full = s_full + kQTiles;           // [2] weights of tile i in TMEM (128 threads)
  uint64_t* pv_done = p_full + kQTiles;          // [2] P.V_i done: S_i free (commit)
  uint64_t* o_final = pv_done + kQTiles;         // [2] every product into O_i done (commit)
  uint64_t* drain = o_final + kQTiles;           // [2] each issuer's products done
  uint64_t* hand = drain + kQTiles;              // [2][4] weights pass of tile i done (per quadrant)
  uint64_t* tile_mask = reinterpret_cast<uint64_t*>(smem + kMaskOff);  // [kMaskSlots][2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  int* flags = reinterpret_cast<int*>(smem + kMiscOff + 8);

  const int qpair = gridDim.x - 1 - blockIdx.x;  // latest positions first
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int tpt = p.tokens_per_tile;

  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int n = __ldg(p.cu_seqlens_q + b + 1) - q0;
  int L = __ldg(p.context_lens + b);
  const int Lcap = p.max_blocks_per_seq * p.block_size;
  if (L > Lcap) {
    if (qpair == 0 && g == 0 && threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
    L = Lcap;
  }
  const int qt0 = qpair * kQTiles * tpt;  // the CTA's first new token
  if (qt0 >= n) return;
  const int ntok = min(kQTiles * tpt, n - qt0);
  const int pos0 = L - n + qt0;           // position of the CTA's first token
  const int kend = min(L, pos0 + ntok);   // keys 0 .. kend-1 are needed
  const int ntiles = kend > 0 ? (kend + kTile - 1) / kTile : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, kQTiles * kM);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < kMaskSlots; ++s) mbar_init(&mask_full[s], 1);
    for (int i = 0; i < kQTiles; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kM);
      mbar_init(&pv_done[i], 1);
      mbar_init(&o_final[i], 1);
      mbar_init(&drain[i], 1);
    }
    for (int i = 0; i < 2 * 4; ++i) mbar_init(&hand[i], 1);
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

  if (warp == 0 || warp == 2) {
    // -------------------------------------------------------- TMA producers
    // Warp 0 loads the keys of tile t into key slot t % 3 once S_0 and S_1
    // of the slot's previous tile are done, and posts the tile's row mask;
    // warp 2 loads the values into value slot t % 2 once P.V_0 and P.V_1 of
    // the slot's previous tile are done.
    const bool is_k = warp == 0;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    const int nslots = is_k ? kKSlots : kVSlots;
    uint64_t* empty = is_k ? k_empty : v_empty;
    uint64_t* full = is_k ? k_full : v_full;
    uint8_t* ring = smem + (is_k ? kKOff : kVOff);
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) prefetch_tensormap(tm);
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % nslots;
      if (t >= nslots) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded_long(&empty[st], ((t / nslots) - 1) & 1, abort_flag));
        if (!ok) break;
      }
      issue_tile_half(p, tm, ring + st * 2 * kChunk, &full[st],
                      is_k ? &tile_mask[2 * (t % kMaskSlots)] : nullptr,
                      is_k ? &mask_full[t % kMaskSlots] : nullptr, bt, g, t * kTile, kend, pol,
                      lane);
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1 || warp == 3) {
    // -------------------------------------------------------- MMA issuers
    // One thread of warp 1 issues the score products, one thread of warp 3
    // the output products, tile by tile and query tile 0 before 1; each
    // blocks in its own bounded waits and commits its own products.
    if (lane == 0) {
      const bool is_s = warp == 1;
      const uint32_t q_base = smem_u32(smem + kQOff);
      const uint32_t k_base = smem_u32(smem + kKOff);
      const uint32_t v_base = smem_u32(smem + kVOff);
      bool ok = true;
      if (is_s) {
        ok = ntiles == 0 || mbar_wait_bounded_long(q_full, 0, abort_flag);
        tc_fence_after();
        for (int t = 0; ok && t < ntiles; ++t) {
          ok = mbar_wait_bounded_long(&k_full[t % kKSlots], (t / kKSlots) & 1, abort_flag);
          const uint32_t kb = k_base + (t % kKSlots) * 2 * kChunk;
          for (int i = 0; ok && i < kQTiles; ++i) {
            // S_i is free once P.V_i(t - 1), which read the weights over it, is done
            ok = t == 0 || mbar_wait_bounded_long(&pv_done[i], (t - 1) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            // S_i(t) = Q_i . K(t)^T: 8 k-steps of 16 over the 128 head
            // elements, both operands K-major 128-byte swizzled (a k-step
            // inside a chunk advances the start by 32 bytes)
            const uint32_t qb = q_base + i * 2 * kChunk;
            const uint32_t d = tmem + kSCol + kTile * i;
#pragma unroll
            for (int j = 0; j < kD / 16; ++j)
              tc_mma_ss(d, smem_desc(qb + (j >> 2) * kChunk + 32 * (j & 3), 16, 1024),
                        smem_desc(kb + (j >> 2) * kChunk + 32 * (j & 3), 16, 1024), kIdescS,
                        j > 0 ? 1u : 0u);
            tc_commit(&s_full[i]);
          }
          if (ok) tc_commit(&k_empty[t % kKSlots]);
        }
      } else {
        for (int t = 0; ok && t < ntiles; ++t) {
          ok = mbar_wait_bounded_long(&v_full[t % kVSlots], (t / kVSlots) & 1, abort_flag);
          const uint32_t vb = v_base + (t % kVSlots) * 2 * kChunk;
          for (int i = 0; ok && i < kQTiles; ++i) {
            ok = mbar_wait_bounded_long(&p_full[i], t & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            // O_i += P_i(t) . V(t): 8 k-steps of 16 keys; P_i from TMEM (bf16
            // pairs, 8 columns per k-step), V MN-major (leading offset: next
            // 64 elements = next chunk; stride offset: next 8 keys = 1 KB)
            const uint32_t pa = tmem + kSCol + kTile * i + kPHalf;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              tc_mma_ts(tmem + kOCol + kD * i, pa + 8 * kk, smem_desc(vb + kk * 2048, kChunk, 1024),
                        kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&pv_done[i]);
            if (t + 1 == ntiles) tc_commit(&o_final[i]);
          }
          if (ok) tc_commit(&v_empty[t % kVSlots]);
        }
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
    // warps 4-7: query tile 0, warps 8-11: query tile 1; one thread per row
    // (its TMEM lane), all 128 keys of every tile.
    const int qi = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = 32 * quad + lane;  // = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * quad) << 16;
    const uint32_t s_addr = tmem + lane_addr + kSCol + kTile * qi;
    const uint32_t o_addr = tmem + lane_addr + kOCol + kD * qi;
    const int tok = qi * tpt + row / G;  // the row's token among the CTA's
    const bool rvalid = tok < ntok;
    const int pos = pos0 + tok;
    const int64_t qrow =
        (static_cast<int64_t>(q0 + qt0 + (rvalid ? tok : 0)) * p.num_q_heads + g * G + row % G) *
        kD;
    // the Q row -> shared memory (two chunks of 64 elements, 128-byte
    // swizzle: 16-byte unit u of row r at u ^ (r & 7)); padding rows are zeros
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow);
      uint8_t* qdst = smem + kQOff + qi * 2 * kChunk + row * 128;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint4 x = rvalid ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(qdst + (u >> 3) * kChunk + (((u & 7) ^ (row & 7)) << 4)) = x;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    const bool pos_scale = p.scale_log2 > 0.f;
    const float sc = pos_scale ? p.scale_log2 : 1.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    // scores of keys 64h .. 64h + 63 of tile t (already in s): the scale
    // when it is not folded into the exponent, then the causal and validity
    // masks unless every key of the half exists and precedes the row
    auto prep_half = [&](float (&s)[64], int t, int h, uint64_t mw) {
      if (!pos_scale) {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] *= p.scale_log2;
      }
      const int kc0 = t * kTile + 64 * h;
      if (!(rvalid && mw == ~0ull && kc0 + 63 <= pos)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (!(rvalid && ((mw >> c) & 1ull) && kc0 + c <= pos)) s[c] = -INFINITY;
      }
    };
    auto max_half = [&](const float (&s)[64]) -> float {
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 64; c += 8) {
        mq[0] = fmax3(mq[0], s[c], s[c + 1]);
        mq[1] = fmax3(mq[1], s[c + 2], s[c + 3]);
        mq[2] = fmax3(mq[2], s[c + 4], s[c + 5]);
        mq[3] = fmax3(mq[3], s[c + 6], s[c + 7]);
      }
      return fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
    };
    // weights of 64 keys as bf16 pairs into 32 TMEM columns; returns their
    // sum.  2^(s * scale - m): a masked score is -inf and 2^-inf = +0 (m is
    // taken as 0 while the row has seen no key, so no -inf + inf)
    auto weights_half = [&](const float (&s)[64], uint32_t dst) -> float {
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
      tc_st32u_nowait(dst, pr);
      return (lq[0].x + lq[0].y) + (lq[1].x + lq[1].y);
    };
    for (int t = 0; t < ntiles; ++t) {
      ok = mbar_wait_bounded(&s_full[qi], t & 1, abort_flag) &&
           mbar_wait_bounded(&mask_full[t % kMaskSlots], (t / kMaskSlots) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint64_t mlo = tile_mask[2 * (t % kMaskSlots)];
      const uint64_t mhi = tile_mask[2 * (t % kMaskSlots) + 1];
      tc_fence_after();
      // pass 1: the row maximum over both halves; the upper half stays in s
      float s[64];
      tc_ld32_nowait(s_addr, &s[0]);
      tc_ld32_nowait(s_addr + 32, &s[32]);
      tc_wait_ld();
      prep_half(s, t, 0, mlo);
      const float mx_lo = max_half(s);
      tc_ld32_nowait(s_addr + 64, &s[0]);
      tc_ld32_nowait(s_addr + 96, &s[32]);
      tc_wait_ld();
      prep_half(s, t, 1, mhi);
      const float mx_raw = fmaxf(mx_lo, max_half(s));
      const float mx = pos_scale ? mx_raw * p.scale_log2 : mx_raw;
      // lazy rescale; tcgen05.ld/st are warp-wide, so the warp rescales
      // together when any of its rows needs it (the others scale by 1).
      // P.V_i(t - 1) is complete: S_i(t) waited for it.
      const bool need = mx > m_run + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float corr = need ? fast_exp2(m_run - mx) : 1.f;
        if (t > 0) {
#pragma unroll 1
          for (int cq = 0; cq < kD / 64; ++cq) {
            float o[64];
            tc_ld32_nowait(o_addr + 64 * cq, &o[0]);
            tc_ld32_nowait(o_addr + 64 * cq + 32, &o[32]);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 64; ++i) o[i] *= corr;
            tc_st32u_nowait(o_addr + 64 * cq, reinterpret_cast<const uint32_t*>(&o[0]));
            tc_st32u_nowait(o_addr + 64 * cq + 32, reinterpret_cast<const uint32_t*>(&o[32]));
            tc_wait_st();
          }
        }
        if (need) {
          l_run *= corr;
          m_run = mx;
        }
      }
      // ping-pong: the two query tiles' weights passes alternate on each SM
      // sub-partition (tile 1's pass of tile t follows tile 0's, tile 0's
      // pass of tile t + 1 follows tile 1's of tile t), so each runs with the
      // sub-partition mostly to itself while the tensor core works for the
      // other query tile
      if (qi == 1 || t > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&hand[(qi ^ 1) * 4 + quad],
                                                       (qi == 1 ? t : t - 1) & 1, abort_flag));
        if (!ok) break;
      }
      // pass 2: weights of keys 64..127 (in registers) over score columns
      // 96..127, then of the re-read keys 0..63 over columns 64..95 (both
      // already read): the A operand of P.V_i, keys 2j, 2j+1 in column 64 + j
      float lsum = weights_half(s, s_addr + kPHalf + 32);
      tc_ld32_nowait(s_addr, &s[0]);
      tc_ld32_nowait(s_addr + 32, &s[32]);
      tc_wait_ld();
      prep_half(s, t, 0, mlo);
      lsum += weights_half(s, s_addr + kPHalf);
      l_run += lsum;
      __syncwarp();
      if (lane == 0) mbar_arrive(&hand[qi * 4 + quad]);
      tc_wait_st();
      // keys without a cache row: zero their value rows (0 x NaN would
      // poison P.V), by query tile 0's threads (P.V_1(t) follows P.V_0(t));
      // piece j = (key j / 2, value chunk j % 2), two per thread
      if (qi == 0 && (mlo != ~0ull || mhi != ~0ull)) {
        // the values of tile t must have landed (their slot's previous tile
        // is then done with them as well)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&v_full[t % kVSlots], (t / kVSlots) & 1,
                                                       abort_flag));
        if (!ok) break;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int j = row + kM * hh;
          const int r = j >> 1;
          if (!mask_bit(mlo, mhi, r)) {
            uint4* dst = reinterpret_cast<uint4*>(smem + kVOff + (t % kVSlots) * 2 * kChunk +
                                                  (j & 1) * kChunk + r * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();  // generic writes before the tensor core reads them
      }
      tc_fence_before();
      mbar_arrive(&p_full[qi]);
    }
    if (ok && ntiles > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&o_final[qi], 0, abort_flag));
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    } else if (ntiles == 0) {
      if (rvalid) {  // no key at all: a zero row
        uint4* dst = reinterpret_cast<uint4*>(p.out + qrow);
#pragma unroll
        for (int u = 0; u < kD / 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
      // ---- epilogue: this thread's output row
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int cq = 0; cq < kD / 32; ++cq) {
        float o[32];
        tc_ld32(o_addr + 32 * cq, o);  // warp-wide: every lane loads
        if (rvalid) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + qrow + 32 * cq);
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
    if ((warp == 0 || warp == 2) && lane == 0) {
      uint64_t* full = warp == 0 ? k_full : v_full;
      const int nslots = warp == 0 ? kKSlots : kVSlots;
      for (int t = max(0, issued - nslots); t < issued; ++t)
        mbar_wait_bounded(&full[t % nslots], (t / nslots) & 1, nullptr);
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

pa_status launch_paged_prefill(const PrefillArgs& a, cudaStream_t stream) {
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
  p.tokens_per_tile = kM / G;
  p.block_size = a.block_size;
  int lg = 0;
  while ((1 << lg) < a.block_size) ++lg;
  p.log2_bs = lg;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const int64_t per_cta = static_cast<int64_t>(kQTiles) * p.tokens_per_tile;
  const int64_t qpairs = (static_cast<int64_t>(a.max_q_len) + per_cta - 1) / per_cta;
  if (qpairs > 0x7FFFFFFF) return PA_ERR_UNSUPPORTED;
  static std::atomic<uint64_t> smem_raised{0};
  if (!ensure_smem_limit(paged_prefill_tcgen05_kernel, kAlloc, smem_raised)) return PA_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(qpairs), static_cast<unsigned>(a.num_kv_heads),
                  static_cast<unsigned>(a.num_seqs));
  paged_prefill_tcgen05_kernel<<<grid, kThreads, kAlloc, stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
