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
//    TMEM columns, leaving none for the scores, so a PAIR of CTAs serves
//    each (head tile, split, sequence): CTA v accumulates output elements
//    256v .. 256v + 255 (256 columns) and both compute the whole score tile
//    (the second one reads the latent rows from L2).  grid = (2 * H / 128,
//    splits, B), the pair adjacent in launch order.
//  * per CTA: q_lat of its 128 heads (9 chunks of 128 rows x 128 bytes,
//    144 KB, the A operand of S) stays in shared memory; the split's tokens
//    stream through a TMA ring in tiles of kTile (9 chunks of kTile rows x
//    128 bytes), 128-byte swizzled, with as many stages as fit beside q_lat.
//  * S[128 x 32] = Q . K^T: 36 tcgen05.mma (M=128, N=32, K=16, bf16 in,
//    fp32 out) from K-major shared-memory descriptors into a double-buffered
//    32-column TMEM tile.  O[128 x 256] += P . V: 2 tcgen05.mma (N=256)
//    with P (bf16, [128 x 32]) from TMEM and V read in place from the same
//    shared-memory tile as an MN-major operand (its 256 elements of each
//    row are contiguous).
//  * warp roles: warp 0 issues the TMA loads, warp 1 owns TMEM and issues
//    the MMAs (one thread), warps 2-5 are the softmax: thread = head row,
//    tcgen05.ld of its 32 scores, fp32 online softmax in base 2 with a lazy
//    rescale (the running max moves only when a score beats it by more than
//    2^8; the rescale reads, scales and writes back the TMEM output row),
//    weights rounded to bf16 and written to TMEM with tcgen05.st.  S(t+1)
//    runs on the tensor core while the softmax works on tile t.
//  * epilogue: the softmax threads read their output row from TMEM; one
//    split writes bf16, several write fp32 partials + log2-sum-exp, and the
//    CTA that completes the per-(sequence, head tile) count (2 * splits
//    arrivals) merges them.
//
// Every wait is bounded (2 s); a timeout sets an error bit, the roles leave
// their loops, the MMAs and copies already issued are drained, and TMEM is
// freed before the CTA exits.
#include <atomic>
#include <cmath>

#include "mla_common.cuh"

namespace pa_detail {
namespace {

using namespace pa;
using namespace mla;

constexpr int kHT = 128;               // heads per CTA (M)
constexpr int kTile = 32;              // tokens per tile (N of S, K of P.V)
// as many stages as fit beside the resident q_lat (144 KB)
constexpr int kStages = kTile == 16 ? 4 : 2;
constexpr int kHalf = kLat / 2;        // output elements per CTA (N of P.V)
constexpr int kThreads = 6 * 32;
constexpr int kQChunkBytes = kHT * 128;              // 16 KB
constexpr int kChunkBytes = kTile * 128;             // 4 KB
constexpr int kStageBytes = kChunks * kChunkBytes;   // 36 KB
constexpr int kQOff = 0;
constexpr int kStageOff = kChunks * kQChunkBytes;    // 144 KB
constexpr int kBarOff = kStageOff + kStages * kStageBytes;
// barriers: q_full, kv_full[kStages], kv_empty[kStages], s_full[2],
// s_empty[2], p_full[2], pv_done[2], o_final, drain; then tile masks, the
// TMEM slot and flags
constexpr int kNumBars = 11 + 2 * kStages;
constexpr int kMaskOff = kBarOff + kNumBars * 8;
constexpr int kMiscOff = kMaskOff + kStages * 8;
constexpr int kBytes = kMiscOff + 32;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "shared memory");

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;      // [0, 256): this CTA's half of the output
constexpr uint32_t kSCol = 256;    // two kTile-column score tiles
constexpr uint32_t kPCol = 320;    // two kTile/2-column weight tiles (bf16 pairs)

// ------------------------------------------------------------ tcgen05 ops --
// Shared-memory matrix descriptor: start, leading and stride byte offsets
// (>> 4), the fixed version bit 46, and the swizzle mode in bits 61-63
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1),
// bf16 A and B (bits 7-9, 10-12 = 1), B major-ness (bit 16: 1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdescS = instr_desc(kHT, kTile, false);
constexpr uint32_t kIdescPV = instr_desc(kHT, kHalf, true);

__device__ __forceinline__ void tc_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive once on `bar` when every tcgen05 operation this thread issued so far completes
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_ld(uint32_t taddr, float (&v)[32]) { tc_ld32(taddr, v); }
__device__ __forceinline__ void tc_ld(uint32_t taddr, float (&v)[16]) { tc_ld16(taddr, v); }
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st(uint32_t taddr, const uint32_t (&r)[16]) { tc_st16(taddr, r); }
__device__ __forceinline__ void tc_st(uint32_t taddr, const uint32_t (&r)[8]) { tc_st8(taddr, r); }

// ------------------------------------------------------------------ kernel --
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_kv, const MlaParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                 // [kStages] tile landed
  uint64_t* kv_empty = kv_full + kStages;       // [kStages] P.V of the stage's tile done (commit)
  uint64_t* s_full = kv_empty + kStages;        // [2] scores in TMEM (commit)
  uint64_t* s_empty = s_full + 2;               // [2] scores read (128 softmax threads)
  uint64_t* p_full = s_empty + 2;               // [2] weights in TMEM (128 softmax threads)
  uint64_t* pv_done = p_full + 2;               // [2] P.V done (commit)
  uint64_t* o_final = pv_done + 2;              // every product done (commit)
  uint64_t* drain = o_final + 1;                // error path: issued products done
  uint64_t* tile_mask = reinterpret_cast<uint64_t*>(smem + kMaskOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  int* flags = reinterpret_cast<int*>(smem + kMiscOff + 8);  // [0] abort, [1] last CTA

  const int ht = blockIdx.x >> 1;  // 128-head tile
  const int v = blockIdx.x & 1;    // output half
  const int split = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h0 = ht * kHT;
  const int64_t bh0 = static_cast<int64_t>(b) * p.num_heads + h0;

  bool clipped;
  const int L = mla_effective_len(p, b, &clipped);
  if (clipped && split == 0 && blockIdx.x == 0 && threadIdx.x == 0)
    atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
  const int tok_begin = split * p.tokens_per_split;
  const int tok_end = min(tok_begin + p.tokens_per_split, L);
  if (tok_begin >= tok_end) {
    if (split == 0) {  // L == 0: zero rows (this CTA's half)
      for (int i = threadIdx.x; i < kHT * (kHalf / 8); i += kThreads) {
        const int h = i / (kHalf / 8), c = i % (kHalf / 8);
        reinterpret_cast<uint4*>(p.out + (bh0 + h) * kLat + kHalf * v)[c] =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  const int ntiles = (tok_end - tok_begin + kTile - 1) / kTile;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kHT);
      mbar_init(&p_full[s], kHT);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
    flags[0] = 0;
    flags[1] = 0;
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
  const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
  int issued = 0;

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    const uint64_t pol = l2_policy_evict_normal();  // the pair's second CTA re-reads the rows
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_kv);
      mbar_arrive_expect_tx(q_full, kHT * kRowBytes);
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c)
        tma_load_2d(smem + kQOff + c * kQChunkBytes, &tm_q, 64 * c, b * p.num_heads + h0, q_full,
                    pol);
    }
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      if (t >= kStages) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(&kv_empty[stage], ((t / kStages) - 1) & 1, abort_flag));
        if (!ok) break;
      }
      mla_issue_tile_at(p, &tm_kv, smem + kStageOff + stage * kStageBytes, kChunkBytes, kTile,
                        &kv_full[stage], &tile_mask[stage], bt, tok_begin + t * kTile, tok_end,
                        pol, lane);
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
      // O[:, this half] += P(u) . V(u): V = elements 256v.. of tile u's rows,
      // MN-major (leading offset: next 64 elements = next chunk; stride
      // offset: next 8 tokens = 1 KB); P from TMEM, 16 tokens per product
      auto issue_s = [&](int t) {
        // S(t) = Q . K(t)^T over 36 k-steps of 16 (K-major, 128-byte swizzle:
        // a k-step inside a 64-element chunk advances the start by 32 bytes)
        const uint32_t kb = st_base + (t % kStages) * kStageBytes;
#pragma unroll 4
        for (int kc = 0; kc < kChunks * 4; ++kc) {
          const int c = kc >> 2, j = kc & 3;
          tc_mma_ss(tmem + kSCol + kTile * (t & 1),
                    smem_desc(q_base + c * kQChunkBytes + 32 * j, 16, 1024),
                    smem_desc(kb + c * kChunkBytes + 32 * j, 16, 1024), kIdescS,
                    kc > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t & 1]);
      };
      auto issue_pv = [&](int u) {
        // O[:, this half] += P(u) . V(u): V = elements 256v.. of tile u's
        // rows, MN-major (leading offset: next 64 elements = next chunk;
        // stride offset: next 8 tokens = 1 KB); P from TMEM, 16 tokens each
        const uint32_t vb = st_base + (u % kStages) * kStageBytes + 4 * v * kChunkBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma_ts(tmem + kOCol, tmem + kPCol + (kTile / 2) * (u & 1) + 8 * kk,
                    smem_desc(vb + kk * 2048, kChunkBytes, 1024), kIdescPV,
                    (u > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pv_done[u & 1]);
        tc_commit(&kv_empty[u % kStages]);
      };
      // Issue whichever product is ready, never blocking on one while the
      // other could go: S(ns) needs its tile and its score buffer (read by
      // the softmax two tiles ago), P.V(npv) needs the softmax's weights.
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag);
      int ns = 0, npv = 0;
      uint64_t idle_since = 0;
      uint32_t idle = 0;
      while (ok && npv < ntiles) {
        bool progressed = false;
        if (ns < ntiles && mbar_try_wait(&kv_full[ns % kStages], (ns / kStages) & 1) &&
            (ns < 2 || mbar_try_wait(&s_empty[ns & 1], ((ns - 2) >> 1) & 1))) {
          tc_fence_after();
          issue_s(ns);
          ++ns;
          progressed = true;
        }
        if (npv < ns && mbar_try_wait(&p_full[npv & 1], (npv >> 1) & 1)) {
          tc_fence_after();
          issue_pv(npv);
          ++npv;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if ((++idle & 255u) == 0u) {  // bounded: 2 s without progress
          const uint64_t now = globaltimer_ns();
          if (idle == 256u) idle_since = now;
          else if (*abort_flag || now - idle_since > kWaitTimeoutNs) ok = false;
        }
      }
      if (ok) {
        tc_commit(o_final);
      } else {
        *abort_flag = 1;
        atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
      }
      // every product issued completes before tensor memory is freed
      tc_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = 32 * (warp & 3) + lane;  // head within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      ok = mbar_wait_bounded(&s_full[t & 1], (t >> 1) & 1, abort_flag) &&
           mbar_wait_bounded(&kv_full[stage], (t / kStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kTile];
      tc_ld(tmem + lane_addr + kSCol + kTile * (t & 1), s);
      tc_fence_before();
      mbar_arrive(&s_empty[t & 1]);
      const uint32_t mask = static_cast<uint32_t>(tile_mask[stage]);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kTile; ++i) {
        s[i] = ((mask >> i) & 1u) ? s[i] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
      // lazy rescale; tcgen05.ld/st are warp-wide, so the warp rescales
      // together when any of its rows needs it (the others scale by 1)
      const bool need = mx > m_run + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float corr = need ? exp2f(m_run - mx) : 1.f;
        if (t > 0) {
          // the output row holds P.V up to tile t - 1: wait for it
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[(t - 1) & 1],
                                                         ((t - 1) >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHalf / 32; ++c) {
            float o[32];
            tc_ld32(tmem + lane_addr + kOCol + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= corr;
            tc_st32(tmem + lane_addr + kOCol + 32 * c, o);
          }
        }
        if (need) {
          l_run *= corr;
          m_run = mx;
        }
      }
      uint32_t pr[kTile / 2];
#pragma unroll
      for (int i = 0; i < kTile / 2; ++i) {
        // a masked score is -inf and m_run is finite once a token was seen
        const float p0 = s[2 * i] == -INFINITY ? 0.f : exp2f(s[2 * i] - m_run);
        const float p1 = s[2 * i + 1] == -INFINITY ? 0.f : exp2f(s[2 * i + 1] - m_run);
        l_run += p0 + p1;
        pr[i] = pack_bf16x2(p0, p1);
      }
      // tokens that do not exist: zero their value rows in this CTA's half
      // (0 x NaN would poison P.V); thread = (token row / 4, chunk row % 4)
      constexpr uint32_t kFull = kTile == 32 ? 0xFFFFFFFFu : ((1u << kTile) - 1u);
      if (mask != kFull) {
        const int r = row >> 2;
        if (r < kTile && !((mask >> r) & 1u)) {
          uint4* dst = reinterpret_cast<uint4*>(smem + kStageOff + stage * kStageBytes +
                                                (4 * v + (row & 3)) * kChunkBytes + r * 128);
#pragma unroll
          for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // generic writes before the tensor core reads them
      }
      // the weight tile of tile t - 2 must have been consumed
      if (t >= 2) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pv_done[t & 1], ((t - 2) >> 1) & 1,
                                                       abort_flag))) {
          ok = false;
          break;
        }
      }
      tc_st(tmem + lane_addr + kPCol + (kTile / 2) * (t & 1), pr);
      tc_fence_before();
      mbar_arrive(&p_full[t & 1]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_final, 0, abort_flag));
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    } else {
      // ---- epilogue: this thread's output row, elements 256v .. 256v + 255
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const int64_t bh = bh0 + row;
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
        float o[32];
        tc_ld32(tmem + lane_addr + kOCol + 32 * c, o);
        if (p.num_splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + bh * kLat + kHalf * v + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pack_bf16x2(o[8 * u] * inv, o[8 * u + 1] * inv),
                                pack_bf16x2(o[8 * u + 2] * inv, o[8 * u + 3] * inv),
                                pack_bf16x2(o[8 * u + 4] * inv, o[8 * u + 5] * inv),
                                pack_bf16x2(o[8 * u + 6] * inv, o[8 * u + 7] * inv));
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.ws_o + (bh * p.num_splits + split) * kLat + kHalf * v + 32 * c);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[u] = make_float4(o[4 * u] * inv, o[4 * u + 1] * inv, o[4 * u + 2] * inv,
                                 o[4 * u + 3] * inv);
        }
      }
      if (p.num_splits > 1 && v == 0)
        p.ws_lse[bh * p.num_splits + split] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
    }
  }

  // ---- error path: wait (bounded) for the copies still in flight
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      mbar_wait_bounded(q_full, 0, nullptr);
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait_bounded(&kv_full[t % kStages], (t / kStages) & 1, nullptr);
    }
    if (p.num_splits > 1 && threadIdx.x < kHT)
      p.ws_lse[(bh0 + threadIdx.x) * p.num_splits + split] = -INFINITY;
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  if (p.num_splits == 1) return;

  // ---- split count and merge: 2 CTAs per split; the CTA that completes
  // the count of its (sequence, head tile) merges all 128 heads
  const int n_valid = (L + p.tokens_per_split - 1) / p.tokens_per_split;
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned* ctr = p.counters + static_cast<int64_t>(b) * (p.num_heads / kHT) + ht;
    const unsigned prev = atomicAdd(ctr, 1u);
    const bool last = prev + 1u == 2u * static_cast<unsigned>(n_valid);
    if (last) {
      atomicExch(ctr, 0u);
      __threadfence();
    }
    flags[1] = last ? 1 : 0;
  }
  __syncthreads();
  if (flags[1]) {
    for (int h = warp; h < kHT; h += kThreads / 32) mla_merge_warp(p, bh0 + h, n_valid, lane);
  }
}

}  // namespace

int mla_tc_tile() { return kTile; }

pa_status launch_mla_tc(const CUtensorMap& mq, const CUtensorMap& mkv, const MlaParams& p,
                        dim3 grid, cudaStream_t stream) {
  static std::atomic<bool> attr_set{false};
  if (!attr_set.load()) {
    if (cudaFuncSetAttribute(mla_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kAlloc) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_set.store(true);
  }
  mla_decode_tc_kernel<<<grid, kThreads, kAlloc, stream>>>(mq, mkv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
