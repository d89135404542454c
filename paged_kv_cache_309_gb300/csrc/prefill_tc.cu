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
//  * warps 2-5 load the CTA's Q rows into shared memory, then per tile read
//    their row's 128 scores (tcgen05.ld), apply the causal and validity
//    masks, run an fp32 online softmax in base 2 with a lazy rescale (the
//    running max moves only when a score beats it by more than 2^8; the
//    rescale reads, scales and writes back the TMEM output row), and write
//    the weights, rounded to bf16, to TMEM (tcgen05.st).  S of the next tile
//    runs on the tensor core while they work.
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
constexpr int kThreads = 6 * 32;
constexpr int kChunk = 128 * 128;              // 64 elements of 128 rows: 16 KB
constexpr int kQOff = 0;                       // Q: two chunks
constexpr int kStageOff = 2 * kChunk;          // per stage: K lo, K hi, V lo, V hi
constexpr int kStageBytes = 4 * kChunk;        // 64 KB
constexpr int kBarOff = kStageOff + kStages * kStageBytes;
// q_full, kv_full[3], kv_empty[3], s_full[2], s_empty[2], p_full[2],
// pv_done[2], o_final, drain
constexpr int kNumBars = 7 + 2 * kStages + 4;
constexpr int kMaskOff = kBarOff + kNumBars * 8;  // two 64-bit words per stage
constexpr int kMiscOff = kMaskOff + kStages * 16;
constexpr int kBytes = kMiscOff + 32;
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

// Loads of key tile t (warp 0, all lanes): lane i < nbox looks up block
// piece i, the lanes agree on the 128-bit row mask, lane 0 posts it and the
// byte count, and each lane with a valid piece issues its four boxes.
__device__ __forceinline__ void issue_key_tile(const PrefillTcParams& p, const CUtensorMap* tm_k,
                                               const CUtensorMap* tm_v, uint8_t* stage,
                                               uint64_t* full, uint64_t* mask_slot,
                                               const int32_t* bt, int g, int tok0, int kend,
                                               uint64_t pol, int lane) {
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
    mask_slot[0] = (static_cast<uint64_t>(w1) << 32) | w0;
    mask_slot[1] = (static_cast<uint64_t>(w3) << 32) | w2;
    mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(vb) * rpb * 128 * 4));
  }
  __syncwarp();
  if (valid) {
    const int32_t row = bid * bs + row0;
    uint8_t* st = stage + lane * rpb * 128;
    tma_load_3d(st + 0 * kChunk, tm_k, 0, g, row, full, pol);
    tma_load_3d(st + 1 * kChunk, tm_k, 64, g, row, full, pol);
    tma_load_3d(st + 2 * kChunk, tm_v, 0, g, row, full, pol);
    tma_load_3d(st + 3 * kChunk, tm_v, 64, g, row, full, pol);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v,
                                 const PrefillTcParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars + 0;                 // Q rows in shared memory (128 threads)
  uint64_t* kv_full = bars + 1;                // [kStages] key tile landed
  uint64_t* kv_empty = kv_full + kStages;      // [kStages] P.V of the stage's tile done
  uint64_t* s_full = kv_empty + kStages;       // [2] scores in TMEM (commit)
  uint64_t* s_empty = s_full + 2;              // [2] scores read (128 threads)
  uint64_t* p_full = s_empty + 2;              // [2] weights in TMEM (128 threads)
  uint64_t* pv_done = p_full + 2;              // [2] P.V done (commit)
  uint64_t* o_final = pv_done + 2;             // every product done (commit)
  uint64_t* drain = o_final + 1;               // error path: issued products done
  uint64_t* tile_mask = reinterpret_cast<uint64_t*>(smem + kMaskOff);  // [kStages][2]
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
    mbar_init(q_full, kM);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kM);
      mbar_init(&p_full[s], kM);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
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
  int issued = 0;

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      if (t >= kStages) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&kv_empty[stage],
                                                       ((t / kStages) - 1) & 1, abort_flag));
        if (!ok) break;
      }
      issue_key_tile(p, &tm_k, &tm_v, smem + kStageOff + stage * kStageBytes, &kv_full[stage],
                     &tile_mask[2 * stage], bt, g, t * kTile, kend, pol, lane);
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(smem + kQOff);
      const uint32_t st_base = smem_u32(smem + kStageOff);
      auto issue_s = [&](int t) {
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
      };
      auto issue_pv = [&](int u) {
        // O += P(u) . V(u): 8 k-steps of 16 keys; P from TMEM, V = chunks 2,3
        // of the stage, MN-major (leading offset: next 64 elements = next
        // chunk; stride offset: next 8 keys = 1 KB)
        const uint32_t vb = st_base + (u % kStages) * kStageBytes + 2 * kChunk;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma_ts(tmem + kOCol, tmem + kPCol + (kTile / 2) * (u & 1) + 8 * kk,
                    smem_desc(vb + kk * 2048, kChunk, 1024), kIdescPV,
                    (u > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pv_done[u & 1]);
        tc_commit(&kv_empty[u % kStages]);
      };
      bool ok = ntiles == 0 || mbar_wait_bounded(q_full, 0, abort_flag);
      tc_fence_after();
      int ns = 0, npv = 0;
      uint64_t idle_since = 0;
      uint32_t idle = 0;
      while (ok && npv < ntiles) {
        bool progressed = false;
        if (ns < ntiles && mbar_test_wait(&kv_full[ns % kStages], (ns / kStages) & 1) &&
            (ns < 2 || mbar_test_wait(&s_empty[ns & 1], ((ns - 2) >> 1) & 1))) {
          tc_fence_after();
          issue_s(ns);
          ++ns;
          progressed = true;
        }
        if (npv < ns && mbar_test_wait(&p_full[npv & 1], (npv >> 1) & 1)) {
          tc_fence_after();
          issue_pv(npv);
          ++npv;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if ((++idle & 4095u) == 0u) {  // bounded: 2 s without progress
          const uint64_t now = globaltimer_ns();
          if (idle == 4096u) idle_since = now;
          else if (*abort_flag || now - idle_since > kWaitTimeoutNs) ok = false;
        }
      }
      if (ok) {
        tc_commit(o_final);
      } else {
        *abort_flag = 1;
        atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
      }
      tc_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = 32 * (warp & 3) + lane;  // = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int tok = row / G;
    const bool rvalid = tok < ntok;
    const int pos = pos0 + tok;
    const int64_t qrow =
        (static_cast<int64_t>(q0 + qt0 + (rvalid ? tok : 0)) * p.num_q_heads + g * G + row % G) *
        kD;
    // Q rows -> shared memory (two chunks of 64 elements, 128-byte swizzle:
    // 16-byte unit u of row r at u ^ (r & 7)); padding rows are zeros
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint4 x = rvalid ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + kQOff + (u >> 3) * kChunk + row * 128 +
                                  (((u & 7) ^ (row & 7)) << 4)) = x;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      const int k = t & 1;
      ok = mbar_wait_bounded(&s_full[k], (t >> 1) & 1, abort_flag) &&
           mbar_wait_bounded(&kv_full[stage], (t / kStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kTile];
#pragma unroll
      for (int i = 0; i < kTile / 32; ++i)
        tc_ld32_nowait(tmem + lane_addr + kSCol + kTile * k + 32 * i, &s[32 * i]);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(&s_empty[k]);
      const uint64_t mlo = tile_mask[2 * stage], mhi = tile_mask[2 * stage + 1];
      const int kt0 = t * kTile;
      // no mask needed when every key of the tile exists and precedes the row
      const bool plain = rvalid && mlo == ~0ull && mhi == ~0ull && kt0 + kTile - 1 <= pos;
      if (!plain) {
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (!(rvalid && mask_bit(mlo, mhi, c) && kt0 + c <= pos)) s[c] = -INFINITY;
      }
      // scale and max with four independent chains
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < kTile; ++c) {
        s[c] *= p.scale_log2;
        mq[c & 3] = fmaxf(mq[c & 3], s[c]);
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      // lazy rescale; tcgen05.ld/st are warp-wide, so the warp rescales
      // together when any of its rows needs it (the others scale by 1)
      const bool need = mx > m_run + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float corr = need ? fast_exp2(m_run - mx) : 1.f;
        if (t > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[(t - 1) & 1],
                                                         ((t - 1) >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int cq = 0; cq < kD / 32; ++cq) {
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
      // keys without a cache row: zero their V rows (0 x NaN would poison
      // P.V); piece j = (key j / 2, V chunk j % 2), two per thread
      if (mlo != ~0ull || mhi != ~0ull) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int j = row + kM * hh;
          const int r = j >> 1;
          if (!mask_bit(mlo, mhi, r)) {
            uint4* dst = reinterpret_cast<uint4*>(smem + kStageOff + stage * kStageBytes +
                                                  (2 + (j & 1)) * kChunk + r * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();  // generic writes before the tensor core reads them
      }
      // the weight tile of tile t - 2 must have been consumed
      if (t >= 2) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[k], ((t - 2) >> 1) & 1,
                                                       abort_flag))) {
          ok = false;
          break;
        }
      }
      // weights, rounded to bf16, as bf16 pairs in TMEM (64 keys per store,
      // one wait for both); the row sum in four independent chains
      float lq[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pr[kTile / 2];
#pragma unroll
      for (int i = 0; i < kTile / 2; ++i) {
        const float x0 = s[2 * i], x1 = s[2 * i + 1];
        const float p0 = x0 == -INFINITY ? 0.f : fast_exp2(x0 - m_run);
        const float p1 = x1 == -INFINITY ? 0.f : fast_exp2(x1 - m_run);
        lq[i & 3] += p0 + p1;
        pr[i] = pack_bf16x2(p0, p1);
      }
      l_run += (lq[0] + lq[1]) + (lq[2] + lq[3]);
      tc_st32u_nowait(tmem + lane_addr + kPCol + (kTile / 2) * k, &pr[0]);
      tc_st32u_nowait(tmem + lane_addr + kPCol + (kTile / 2) * k + 32, &pr[32]);
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[k]);
    }
    if (ok && ntiles > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_final, 0, abort_flag));
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    } else if (rvalid) {
      // ---- epilogue: this thread's output row (no key at all: a zero row)
      __nv_bfloat16* dst = p.out + qrow;
      if (ntiles == 0) {
#pragma unroll
        for (int u = 0; u < kD / 8; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (ok && ntiles > 0) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int cq = 0; cq < kD / 32; ++cq) {
        float o[32];
        tc_ld32(tmem + lane_addr + kOCol + 32 * cq, o);  // warp-wide: every lane loads
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
