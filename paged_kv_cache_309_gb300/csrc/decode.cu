// decode.cu -- paged GQA decode attention: split kernel + log-sum-exp merge.
//
// What is computed: for sequence b and query head h, softmax attention of
// q[b, h] over the first context_lens[b] logical tokens, read back from the
// paged cache along the block table (nano-vLLM walkthrough, section 2.6:
// decode attention reads the physical blocks via block_tables;
// PagedAttention-principle post, "paged attention原理": blocks may be
// scattered, the table keeps their order).  Query head h uses KV head
// h / (H_Q / H_KV).  The score matrix is never stored (same post, decode
// dataflow: FA/PA-style kernels do not materialise it).
//
// How (sm_103a):
//  * grid = (split, kv head, sequence).  A split is a fixed range of logical
//    tokens; a CTA whose range starts past the sequence's length exits.
//    All G = H_Q / H_KV query heads of the KV head share the CTA, so each
//    K/V byte is read from HBM once and used G times.
//  * one producer warp streams the range in tiles of 64 tokens: per tile it
//    looks up the tile's physical blocks in the block table and issues 3-D
//    TMA copies -- per (block, K|V, 64-element half row) one [rows, 64] box
//    of one KV head -- into a 3-stage shared-memory ring with the 128-byte
//    swizzle, signalling an mbarrier with the byte count; a per-tile 64-bit
//    mask marks the rows that exist (inside the context and in a valid
//    block).  The L2 policy is evict-first: the K/V stream is read once.
//  * four consumer warps each take a 16-token slice of every tile and run
//    the two grouped products on the tensor cores (mma.sync m16n8k16, bf16
//    in, fp32 accumulate): S^T = K.Q^T (tokens x heads), an fp32 online
//    softmax in base 2 with warp-shuffle max reductions and a lazy rescale
//    (the running max moves only when a score beats it by more than 2^8),
//    then O^T += V^T.P^T (head elements x heads).  CUDA-core FMAs were the
//    first design; at G = 4 they needed ~66 instructions per token and KV
//    head and could not keep HBM busy, the tensor cores need a few.
//  * epilogue: the warps' (max, sum, accumulator) are merged in shared
//    memory; one split writes bf16 directly, several splits write an fp32
//    partial and its log2-sum-exp to the workspace and count themselves in
//    a per-(sequence, kv head) counter; the CTA that completes the count
//    merges the splits (weights 2^(lse_s - max)) and zeroes the counter, so
//    no second kernel is launched.
//
// Every mbarrier wait is bounded (2 s); a timeout sets an error bit in the
// workspace's error word, drains the copies already issued, and exits.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>

#include "pa_internal.cuh"

namespace pa_detail {
namespace {

using namespace pa;

constexpr int kD = 128;                 // head size handled by this kernel
constexpr int kTile = 64;               // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowBytes = kD * 2;       // one bf16 row of one KV head (tensor map stride)
constexpr float kRescaleLog2 = 8.0f;    // lazy-rescale threshold (base-2 units)
constexpr size_t kWorkspaceHeader = 256;  // error word + padding

struct DecodeParams {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_lse;
  float* ws_o;
  unsigned* counters;  // [B, H_KV] split arrivals, zero between calls
  unsigned* err;
  int64_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t log2_bs;
  int32_t max_blocks_per_seq;
  int32_t num_splits;
  int32_t tokens_per_split;
  float scale_log2;
  const float* k_scale;  // quantised cache: code * k_scale is the value (else null)
  const float* v_scale;
  // fused decode step (else null): each sequence's newest K/V row
  // [B, H_KV, d] bf16, written at slot_mapping[b] before it is attended to
  const __nv_bfloat16* new_k;
  const __nv_bfloat16* new_v;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
};


// context length used by both kernels: clipped to the plan and the table
__device__ __forceinline__ int effective_len(const DecodeParams& p, int b, bool* clipped) {
  int L = __ldg(p.context_lens + b);
  L = L < 0 ? 0 : L;
  const int64_t cap = min(static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size,
                          static_cast<int64_t>(p.num_splits) * p.tokens_per_split);
  *clipped = static_cast<int64_t>(L) > cap;
  return *clipped ? static_cast<int>(cap) : L;
}

// ===================================================== tensor-core consumer
// The same split kernel with the grouped products on the tensor cores
// (mma.sync m16n8k16, bf16 in, fp32 accumulate).  Per consumer warp and
// tile: a 16-token slice.  S^T = K_slice . Q^T puts tokens on M (16) and
// query heads on N (8 per n-tile, zero-padded past G); O^T += V^T . P^T puts
// head elements on M (8 tiles of 16) and heads on N.  The K/V tiles arrive
// through TMA with the 128-byte swizzle, one box per 64-element half of a
// row, so that ldmatrix reads eight consecutive tokens from eight different
// bank groups.  P enters the second product as a pair of bf16 terms (the
// rounded value and its rounding error), so the weights keep ~16 bits.
constexpr int kHalfBytes = kTile * 128;  // one 64-row x 128-byte region (8 KB)
// Shared memory of one CTA.  bf16 cache: per stage K_lo, K_hi, V_lo, V_hi
// regions (64 rows x 128 B each: one 64-element half of every row).  fp8
// cache: a 128-element row is 128 bytes, so per stage K and V regions and a
// smaller CTA: three per SM, four when G <= 8 (the consumers then fit 96
// registers), for more warps against latency.  All regions 128-byte
// swizzled and 1 KB aligned.
template <bool kFp8>
struct TcLayout {
  static constexpr int kStages = 3;
  static constexpr int kCtasPerSm = kFp8 ? 3 : 2;  // fp8 needs more warps per SM
  static constexpr int kRowBytes = kFp8 ? 128 : 256;  // one row of one kv head
  static constexpr int kStageBytes = (kFp8 ? 2 : 4) * kHalfBytes;
  static constexpr int kVOffset = (kFp8 ? 1 : 2) * kHalfBytes;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kBytes = kBarOffset + 3 * kStages * 8 + 16;  // full, empty, mask, flags
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1 KB
};

// Merge of one (sequence, query head) by one warp: weights 2^(lse_s - max)
// over the n splits that hold tokens, out = sum_s w_s o_s / sum_s w_s,
// rounded to bf16.  Partials are read through L2 (__ldcg): other CTAs wrote
// them during this launch.
__device__ __forceinline__ void merge_splits_warp(const DecodeParams& p, int64_t bh, int n,
                                                  int lane) {
  const float* lse = p.ws_lse + bh * p.num_splits;
  const float* o = p.ws_o + bh * p.num_splits * kD;
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, __ldcg(lse + s));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      const int my = s0 + lane;
      const float wl = my < n ? exp2f(__ldcg(lse + my) - M) : 0.f;
      const int cnt = min(32, n - s0);
      int k = 0;
      for (; k + 8 <= cnt; k += 8) {
        float4 v[8];
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          v[u] = __ldcg(reinterpret_cast<const float4*>(o + static_cast<int64_t>(s0 + k + u) * kD) +
                        lane);
          w[u] = __shfl_sync(0xffffffffu, wl, k + u);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          W += w[u];
          acc.x += w[u] * v[u].x;
          acc.y += w[u] * v[u].y;
          acc.z += w[u] * v[u].z;
          acc.w += w[u] * v[u].w;
        }
      }
      for (; k < cnt; ++k) {
        const float4 v =
            __ldcg(reinterpret_cast<const float4*>(o + static_cast<int64_t>(s0 + k) * kD) + lane);
        const float w = __shfl_sync(0xffffffffu, wl, k);
        W += w;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  *reinterpret_cast<uint2*>(p.out + bh * kD + lane * 4) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

// Decode step, fused write: the warp that owns row L-1 of the last tile
// converts the sequence's new K (lanes 0-15) and V (lanes 16-31) row exactly
// as pa_reshape_and_cache does, stores it at slot_mapping[b], and -- when
// that slot is position L-1's slot -- also puts it into the tile in shared
// memory (the TMA copy may predate the store).  Returns whether shared
// memory was written.
template <bool kFp8>
__device__ __forceinline__ bool fused_token_write(const DecodeParams& p, int b, int g, int L,
                                                  int row, uint8_t* stage_smem, int v_offset,
                                                  int lane) {
  using namespace pa;
  const int64_t slots = p.num_blocks * p.block_size;
  const int64_t s = __ldg(p.slot_mapping + b);
  const int32_t pos_blk = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq +
                                ((L - 1) >> p.log2_bs));
  const int64_t pos_slot = static_cast<int64_t>(pos_blk) * p.block_size + ((L - 1) & (p.block_size - 1));
  if (s < 0 || s >= slots) return false;  // skipped, as in the separate write
  const bool here = s == pos_slot;
  if (!here && lane == 0) atomicOr(p.err, PA_DEVERR_SLOT_MISMATCH);
  const bool is_v = lane >= 16;
  const int e0 = 8 * (lane & 15);
  const int64_t src = (static_cast<int64_t>(b) * p.num_kv_heads + g) * kD + e0;
  const Vec8<bf16> x = load8((is_v ? p.new_v : p.new_k) + src);
  const int64_t dst = (s * p.num_kv_heads + g) * kD + e0;
  uint8_t* region = stage_smem + (is_v ? v_offset : 0);
  if constexpr (kFp8) {
    float f[8];
    const float* sc = is_v ? p.v_scale : p.k_scale;
    if (sc != nullptr) {
      const Divisor d = make_divisor(__ldg(sc));
      div8_for_e4m3(x, f, d, fminf(1.7e38f * d.s, 3.0e38f));
    } else {
      to_f32(x, f);
    }
    const Vec8<e4m3> y = from_f32<e4m3>(f);
    store8(static_cast<e4m3*>(is_v ? p.v_cache : p.k_cache) + dst, y);
    if (here)
      *reinterpret_cast<uint2*>(region + row * 128 + (((e0 >> 4) ^ (row & 7)) << 4) + (e0 & 15)) = y.u;
  } else {
    store8(static_cast<bf16*>(is_v ? p.v_cache : p.k_cache) + dst, x);
    if (here)
      *reinterpret_cast<uint4*>(region + (e0 >> 6) * kHalfBytes + row * 128 +
                                ((((e0 & 63) >> 3) ^ (row & 7)) << 4)) = x.u;
  }
  return here;
}

template <int NT, bool kPairRows>
__device__ __forceinline__ void epilogue_tc(const DecodeParams& p, uint8_t* smem,
                                            float (&o)[8][NT][4], float (&m)[NT][2],
                                            float (&l)[NT][2], int b, int split, int hq0, int G,
                                            int warp, int lane, float out_scale);

// NT: n-tiles of 8 query heads (G <= 8 -> 1, G = 16 -> 2); kFp8: e4m3 cache.
template <int NT, bool kFp8>
__global__ void __launch_bounds__(kThreads, (kFp8 && NT == 1) ? 4 : TcLayout<kFp8>::kCtasPerSm)
    paged_decode_split_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                                 const __grid_constant__ CUtensorMap tm_v, const DecodeParams p,
                                 int G) {
  using namespace pa;
  using Lay = TcLayout<kFp8>;
  constexpr int kStages = Lay::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // 1 KB-aligned base (the 128-byte swizzle pattern repeats every 1 KB)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* tile_mask = empty + kStages;
  int* abort_ptr = reinterpret_cast<int*>(tile_mask + kStages);

  // kv heads fastest in launch order: the H_KV CTAs of one (sequence, split)
  // read the same token rows (each row holds every kv head) at the same time
  const int g = blockIdx.x;
  const int split = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bs = p.block_size;
  const int hq0 = g * G;

  bool clipped;
  const int L = effective_len(p, b, &clipped);
  if (clipped && split == 0 && g == 0 && threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
  const int tok_begin = split * p.tokens_per_split;
  const int tok_end = min(tok_begin + p.tokens_per_split, L);
  if (tok_begin >= tok_end) {
    if (split == 0) {  // only when L == 0: a zero row per head
      for (int i = threadIdx.x; i < G * (kD / 8); i += kThreads) {
        const int h = i / (kD / 8), c = i % (kD / 8);
        reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * p.num_q_heads + hq0 + h) *
                                             kD)[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  const int ntiles = (tok_end - tok_begin + kTile - 1) / kTile;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_ptr = 0;
    mbar_init_fence();
  }
  __syncthreads();
  volatile int* abort_flag = abort_ptr;

  const int gq = lane >> 2;  // mma groupID
  const int tq = lane & 3;   // thread in group
  float o[8][NT][4];
  float m[NT][2], l[NT][2];
  int issued = 0;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int rpb = bs < kTile ? bs : kTile;
    const int nbox = kTile / rpb;
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
    }
    const int32_t* bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq;
    // lane i < nbox: block id of piece i of tile t (-1 past the range); the
    // next tile's ids are read one iteration ahead, before the wait for a
    // free stage, so their global-memory latency is off the issue path
    auto tile_bid = [&](int t) -> int {
      const int first = tok_begin + t * kTile + lane * rpb;
      return (t < ntiles && lane < nbox && first < tok_end) ? __ldg(bt + (first >> p.log2_bs))
                                                            : -1;
    };
    int bid_next = tile_bid(0);
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      const int bid_cur = bid_next;
      bid_next = tile_bid(t + 1);
      if (t >= kStages) {
        const bool w_ok = mbar_wait_bounded(&empty[stage], ((t / kStages) - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
      }
      const int tok0 = tok_begin + t * kTile;
      const int nval = min(kTile, tok_end - tok0);
      bool valid = false;
      int rows = 0, bid = -1, row0 = 0;
      if (lane < nbox) {
        const int first = tok0 + lane * rpb;
        rows = min(rpb, nval - lane * rpb);
        if (rows > 0) {
          row0 = first & (bs - 1);
          bid = bid_cur;
          valid = bid >= 0 && static_cast<int64_t>(bid) < p.num_blocks;
        }
      }
      uint64_t bits = 0;
      if (valid) bits = (rows >= 64 ? ~0ull : ((1ull << rows) - 1ull)) << (lane * rpb);
      const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits));
      const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits >> 32));
      const uint32_t vb = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) {
        tile_mask[stage] = (static_cast<uint64_t>(hi) << 32) | lo;
        mbar_arrive_expect_tx(&full[stage],
                              static_cast<uint32_t>(__popc(vb) * rpb * Lay::kRowBytes * 2));
      }
      __syncwarp();
      if (valid) {
        const int32_t row = bid * bs + row0;
        uint8_t* st = smem + stage * Lay::kStageBytes + lane * rpb * 128;
        if constexpr (kFp8) {  // a whole row is one 128-byte box
          tma_load_3d(st, &tm_k, 0, g, row, &full[stage], pol);
          tma_load_3d(st + kHalfBytes, &tm_v, 0, g, row, &full[stage], pol);
        } else {  // two 64-element halves per row
          tma_load_3d(st + 0 * kHalfBytes, &tm_k, 0, g, row, &full[stage], pol);
          tma_load_3d(st + 1 * kHalfBytes, &tm_k, 64, g, row, &full[stage], pol);
          tma_load_3d(st + 2 * kHalfBytes, &tm_v, 0, g, row, &full[stage], pol);
          tma_load_3d(st + 3 * kHalfBytes, &tm_v, 64, g, row, &full[stage], pol);
        }
      }
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Q^T as the B operand.  bf16 cache: b0 = q[head gq][16kk + 2tq .. +1],
    // b1 = [.. + 8].  fp8 cache: the k index of every 16-wide step is
    // permuted to match how K arrives (see below): b0 = q[16kk + 4tq .. +1],
    // b1 = q[16kk + 4tq + 2 .. +3], in f16 after a power-of-two prescale
    // that puts max|q| in [2^14, 2^15) (undone in the score scale).
    uint32_t qb[NT][8][2];
    float score_scale = p.scale_log2;
    if constexpr (kFp8) {
      float qv[NT][8][4];
      float qmax = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + gq;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            p.q + (static_cast<int64_t>(b) * p.num_q_heads + hq0 + (h < G ? h : 0)) * kD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t w0 = h < G ? __ldg(qrow + 8 * kk + 2 * tq) : 0u;
          const uint32_t w1 = h < G ? __ldg(qrow + 8 * kk + 2 * tq + 1) : 0u;
          qv[nt][kk][0] = __uint_as_float(w0 << 16);
          qv[nt][kk][1] = __uint_as_float(w0 & 0xFFFF0000u);
          qv[nt][kk][2] = __uint_as_float(w1 << 16);
          qv[nt][kk][3] = __uint_as_float(w1 & 0xFFFF0000u);
#pragma unroll
          for (int c = 0; c < 4; ++c) qmax = fmaxf(qmax, fabsf(qv[nt][kk][c]));
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1)
        qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
      // 2^e with e = 14 - floor(log2(qmax)); finite non-zero q only
      int e = 0;
      if (qmax > 0.f && qmax <= 3.0e38f) e = 14 - (static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFF) - 127);
      const float up = ldexpf(1.0f, e);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qb[nt][kk][0] = pack_f16x2(qv[nt][kk][0] * up, qv[nt][kk][1] * up);
          qb[nt][kk][1] = pack_f16x2(qv[nt][kk][2] * up, qv[nt][kk][3] * up);
        }
      const float ks = p.k_scale != nullptr ? __ldg(p.k_scale) : 1.f;
      score_scale = p.scale_log2 * ks * ldexpf(1.0f, -e);
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + gq;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            p.q + (static_cast<int64_t>(b) * p.num_q_heads + hq0 + (h < G ? h : 0)) * kD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qb[nt][kk][0] = h < G ? __ldg(qrow + 8 * kk + tq) : 0u;
          qb[nt][kk][1] = h < G ? __ldg(qrow + 8 * kk + tq + 4) : 0u;
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        m[nt][j] = -INFINITY;
        l[nt][j] = 0.f;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[mt][nt][c] = 0.f;
    }
    const int r0 = warp * 16;  // this warp's 16-token slice of each tile
    // per-lane ldmatrix row offsets (swizzle: 16-byte unit u sits at u ^ (row & 7))
    const int sw = lane & 7;
    const uint32_t k_row = static_cast<uint32_t>((r0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * 128);
    const uint32_t v_row = static_cast<uint32_t>((r0 + (lane & 7) + 8 * (lane >> 4)) * 128);
    const int k_hi = lane >> 4;        // K: second 8 columns of the k-step
    const int v_hi = (lane >> 3) & 1;  // V: second 8 head elements of the m-tile
    const uint32_t smem_base = smem_u32(smem);
    // fp8 V: ldmatrix.trans rows r0 + (lane & 7) (+8 for lanes 8-15, 24-31),
    // 16-byte unit 2j (lanes 0-15) or 2j + 1 (lanes 16-31)
    const int v8_row = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
    const uint32_t v8_off = static_cast<uint32_t>(v8_row * 128);

    // fused decode step: row of position L-1 in the last tile, and its warp
    const bool fused = p.new_k != nullptr && tok_end == L;
    const int new_row = fused ? (L - 1 - tok_begin) % kTile : -1;

    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      const bool w_ok = mbar_wait_bounded(&full[stage], (t / kStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) {
        ok = false;
        break;
      }
      const uint32_t mask16 = static_cast<uint32_t>(tile_mask[stage] >> r0) & 0xFFFFu;
      const uint32_t st_base = smem_base + stage * Lay::kStageBytes;
      bool smem_written = false;
      if (fused && t == ntiles - 1 && (new_row >> 4) == warp) {
        smem_written = fused_token_write<kFp8>(p, b, g, L, new_row,
                                               smem + stage * Lay::kStageBytes, Lay::kVOffset, lane);
        __syncwarp();
      }
      if (mask16 != 0u) {
        if (mask16 != 0xFFFFu) {
          // rows without a token: zero their V rows (0 x NaN would poison P.V)
          uint8_t* vrow0 = smem + stage * Lay::kStageBytes + Lay::kVOffset;
          constexpr int kUnits = kFp8 ? 8 : 16;  // 16-byte units of a V row in the stage
          for (int idx = lane; idx < 16 * kUnits; idx += 32) {
            const int rr = idx / kUnits, unit = idx % kUnits;
            if (!((mask16 >> rr) & 1u))
              *reinterpret_cast<uint4*>(vrow0 + (unit >> 3) * kHalfBytes + (r0 + rr) * 128 +
                                        (unit & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // ---- S^T = K . Q^T (two accumulator chains)
        float s0[NT][4], s1[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) s0[nt][c] = s1[nt][c] = 0.f;
        if constexpr (kFp8) {
          // One ldmatrix.x4 over 32 bytes of 16 fp8 rows (byte pairs as b16)
          // gives each lane 4 consecutive codes per row and 16-byte group:
          // row gq in r[0]/r[2], row gq + 8 in r[1]/r[3].  Within a 16-wide
          // k-step the codes 4tq..4tq+3 serve as k = 2tq, 2tq+1, 2tq+8,
          // 2tq+9 -- the same permutation q's fragments use.
#pragma unroll
          for (int ks2 = 0; ks2 < 4; ++ks2) {
            uint32_t r[4];
            const uint32_t u = static_cast<uint32_t>(2 * ks2 + k_hi);
            ldsm_x4(st_base + k_row + ((u ^ sw) << 4), r);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int kk = 2 * ks2 + half;
              uint32_t a[4];
              e4m3x4_to_f16x2x2(r[2 * half], a[0], a[2]);
              e4m3x4_to_f16x2x2(r[2 * half + 1], a[1], a[3]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (half) mma_f16_16816(s1[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
                else mma_f16_16816(s0[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
              }
            }
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            uint32_t a[4];
            const uint32_t u = static_cast<uint32_t>(((2 * kk) & 7) + k_hi);
            ldsm_x4(st_base + (kk >> 2) * kHalfBytes + k_row + ((u ^ sw) << 4), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (kk & 1) mma_bf16_16816(s1[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
              else mma_bf16_16816(s0[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
            }
          }
        }
        const bool v0 = (mask16 >> gq) & 1u;        // token r0 + gq
        const bool v1 = (mask16 >> (gq + 8)) & 1u;  // token r0 + gq + 8
        uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float s[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) s[c] = (s0[nt][c] + s1[nt][c]) * score_scale;
          if (!v0) s[0] = s[1] = -INFINITY;
          if (!v1) s[2] = s[3] = -INFINITY;
          float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
          for (int off = 4; off <= 16; off <<= 1) {
            mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
            mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (mx[j] > m[nt][j] + kRescaleLog2) {  // new running max (always on the first)
              const float corr = exp2f(m[nt][j] - mx[j]);
              l[nt][j] *= corr;
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) {
                o[mt][nt][j] *= corr;
                o[mt][nt][j + 2] *= corr;
              }
              m[nt][j] = mx[j];
            }
          }
          const float p0 = v0 ? exp2f(s[0] - m[nt][0]) : 0.f;
          const float p1 = v0 ? exp2f(s[1] - m[nt][1]) : 0.f;
          const float p2 = v1 ? exp2f(s[2] - m[nt][0]) : 0.f;
          const float p3 = v1 ? exp2f(s[3] - m[nt][1]) : 0.f;
          l[nt][0] += p0 + p2;
          l[nt][1] += p1 + p3;
          const int srcA = 8 * tq + (gq >> 1);
          const int srcB = srcA + 4;
          const uint32_t sel = (gq & 1) ? 0x7632u : 0x5410u;
          if constexpr (kFp8) {
            // P in f16 (11 significant bits) for the f16 product with V
            const uint32_t f01 = pack_f16x2(p0, p1);
            const uint32_t f23 = pack_f16x2(p2, p3);
            pb[nt][0] = __byte_perm(__shfl_sync(0xffffffffu, f01, srcA),
                                    __shfl_sync(0xffffffffu, f01, srcB), sel);
            pb[nt][1] = __byte_perm(__shfl_sync(0xffffffffu, f23, srcA),
                                    __shfl_sync(0xffffffffu, f23, srcB), sel);
            continue;
          }
          // P as hi + lo bf16 pairs (hi = bf16(p), lo = bf16(p - hi)): the two
          // products together carry ~16 significant bits of each weight
          const uint32_t h01 = pack_bf16x2(p0, p1);  // token gq,     heads 2tq, 2tq+1
          const uint32_t h23 = pack_bf16x2(p2, p3);  // token gq + 8, heads 2tq, 2tq+1
          const uint32_t l01 = pack_bf16x2(p0 - __uint_as_float(h01 << 16),
                                           p1 - __uint_as_float(h01 & 0xFFFF0000u));
          const uint32_t l23 = pack_bf16x2(p2 - __uint_as_float(h23 << 16),
                                           p3 - __uint_as_float(h23 & 0xFFFF0000u));
          // transpose into the B operand: b0 = P[2tq, 2tq+1][gq], b1 = P[2tq+8, 2tq+9][gq]
          pb[nt][0] = __byte_perm(__shfl_sync(0xffffffffu, h01, srcA),
                                  __shfl_sync(0xffffffffu, h01, srcB), sel);
          pb[nt][1] = __byte_perm(__shfl_sync(0xffffffffu, h23, srcA),
                                  __shfl_sync(0xffffffffu, h23, srcB), sel);
          pl[nt][0] = __byte_perm(__shfl_sync(0xffffffffu, l01, srcA),
                                  __shfl_sync(0xffffffffu, l01, srcB), sel);
          pl[nt][1] = __byte_perm(__shfl_sync(0xffffffffu, l23, srcA),
                                  __shfl_sync(0xffffffffu, l23, srcB), sel);
        }
        // ---- O^T += V^T . P^T
        if constexpr (kFp8) {
          // V^T straight from the e4m3 rows: ldmatrix.trans of byte pairs
          // gives lane (gq, tq), for tokens 2tq, 2tq+1 (+8 in r[1], r[3]), the
          // codes of head elements 2gq and 2gq + 1 of a 16-element unit.
          // The rows of an m-tile are therefore paired: A row gq carries
          // element 16mt + 2gq and row gq + 8 element 16mt + 2gq + 1 (the
          // epilogue puts them back in order).  One byte permute per
          // register groups each element's two tokens; two conversions make
          // the f16 pairs.
          const uint32_t vbase = st_base + Lay::kVOffset;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[4];
            const int unit = 2 * j + (lane >> 4);
            ldsm_x4_trans(vbase + v8_off + static_cast<uint32_t>((unit ^ (v8_row & 7)) << 4), r);
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // m-tile 2j + h from r[2h] (tokens 0-7), r[2h+1] (8-15)
              uint32_t a[4];
              e4m3x4_to_f16x2x2(__byte_perm(r[2 * h], 0u, 0x3120u), a[0], a[1]);
              e4m3x4_to_f16x2x2(__byte_perm(r[2 * h + 1], 0u, 0x3120u), a[2], a[3]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_f16_16816(o[2 * j + h][nt], a, pb[nt][0], pb[nt][1]);
            }
          }
          if (mask16 != 0xFFFFu || smem_written)
            fence_proxy_async_smem();  // generic writes before the next TMA
        } else {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a[4];
            const uint32_t u = static_cast<uint32_t>(((2 * mt) & 7) + v_hi);
            ldsm_x4_trans(st_base + (2 + (mt >> 2)) * kHalfBytes + v_row + ((u ^ sw) << 4), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_bf16_16816(o[mt][nt], a, pb[nt][0], pb[nt][1]);
              mma_bf16_16816(o[mt][nt], a, pl[nt][0], pl[nt][1]);
            }
          }
          if (mask16 != 0xFFFFu || smem_written)
            fence_proxy_async_smem();  // generic writes before the next TMA
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // wait (bounded) for copies already in flight, then leave an empty
    // partial so that the split count below still completes
    if (warp == kConsumerWarps && lane == 0) {
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait_bounded(&full[t % kStages], (t / kStages) & 1, nullptr);
    }
    if (p.num_splits > 1 && threadIdx.x < G)
      p.ws_lse[(static_cast<int64_t>(b) * p.num_q_heads + hq0 + threadIdx.x) * p.num_splits +
               split] = -INFINITY;
  } else {
    const float out_scale = (kFp8 && p.v_scale != nullptr) ? __ldg(p.v_scale) : 1.f;
    epilogue_tc<NT, kFp8>(p, smem, o, m, l, b, split, hq0, G, warp, lane, out_scale);
  }
  if (p.num_splits == 1) return;

  // ------------------------------------------------- split count and merge
  // The CTA that completes the count of its (sequence, kv head) merges the
  // splits of its G query heads and returns the counter to zero.
  __syncthreads();  // every partial of this CTA is written
  int* last_flag = abort_ptr + 1;
  const int n_valid = (L + p.tokens_per_split - 1) / p.tokens_per_split;
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned* ctr = p.counters + static_cast<int64_t>(b) * p.num_kv_heads + g;
    const unsigned prev = atomicAdd(ctr, 1u);
    const bool last = prev + 1u == static_cast<unsigned>(n_valid);
    if (last) {
      atomicExch(ctr, 0u);
      __threadfence();
    }
    *last_flag = last ? 1 : 0;
  }
  __syncthreads();
  if (*last_flag) {
    for (int h = warp; h < G; h += kThreads / 32)
      merge_splits_warp(p, static_cast<int64_t>(b) * p.num_q_heads + hq0 + h, n_valid, lane);
  }
}

// Epilogue of the tensor-core split kernel: merge the consumer warps'
// (max, sum, accumulator) in shared memory; one split writes bf16 output,
// several splits write an fp32 partial and its log2-sum-exp.  kPairRows:
// accumulator rows gq / gq + 8 of m-tile mt hold head elements 16mt + 2gq
// and 16mt + 2gq + 1 (fp8 cache) instead of 16mt + gq and 16mt + gq + 8.
template <int NT, bool kPairRows>
__device__ __forceinline__ void epilogue_tc(const DecodeParams& p, uint8_t* smem,
                                            float (&o)[8][NT][4], float (&m)[NT][2],
                                            float (&l)[NT][2], int b, int split, int hq0, int G,
                                            int warp, int lane, float out_scale) {
  constexpr int NWARP_GROUPS = kConsumerWarps;
  const int gq = lane >> 2;
  const int tq = lane & 3;
  // red[warp][h][d], red_m/red_l[warp][h], red_w[warp][h], fin[h][2]
  float* red = reinterpret_cast<float*>(smem);
  const int GH = NT * 8;
  float* red_m = red + NWARP_GROUPS * GH * kD;
  float* red_l = red_m + NWARP_GROUPS * GH;
  float* red_w = red_l + NWARP_GROUPS * GH;
  float* fin = red_w + NWARP_GROUPS * GH;
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float lv = l[nt][j];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        const int h = nt * 8 + 2 * tq + j;
        if (gq == 0) {
          red_m[warp * GH + h] = m[nt][j];
          red_l[warp * GH + h] = lv;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int e_lo = kPairRows ? 16 * mt + 2 * gq : 16 * mt + gq;
          const int e_hi = kPairRows ? e_lo + 1 : e_lo + 8;
          red[(warp * GH + h) * kD + e_lo] = o[mt][nt][j];
          red[(warp * GH + h) * kD + e_hi] = o[mt][nt][j + 2];
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWARP_GROUPS; ++w) M = fmaxf(M, red_m[w * GH + h]);
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP_GROUPS; ++w) {
      const float wt = (M == -INFINITY) ? 0.f : exp2f(red_m[w * GH + h] - M);
      red_w[w * GH + h] = wt;
      Ls += red_l[w * GH + h] * wt;
    }
    fin[2 * h] = M;
    fin[2 * h + 1] = Ls;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * (kD / 4); i += kThreads) {
    const int h = i / (kD / 4);
    const int e0 = (i % (kD / 4)) * 4;
    float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NWARP_GROUPS; ++w) {
      const float wt = red_w[w * GH + h];
      const float4 v = *reinterpret_cast<const float4*>(red + (w * GH + h) * kD + e0);
      acc4.x += wt * v.x;
      acc4.y += wt * v.y;
      acc4.z += wt * v.z;
      acc4.w += wt * v.w;
    }
    const float Ls = fin[2 * h + 1];
    const float inv = Ls > 0.f ? out_scale / Ls : 0.f;
    acc4.x *= inv;
    acc4.y *= inv;
    acc4.z *= inv;
    acc4.w *= inv;
    const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + hq0 + h;
    if (p.num_splits == 1) {
      *reinterpret_cast<uint2*>(p.out + row * kD + e0) =
          make_uint2(pack_bf16x2(acc4.x, acc4.y), pack_bf16x2(acc4.z, acc4.w));
    } else {
      const int64_t slot = row * p.num_splits + split;
      *reinterpret_cast<float4*>(p.ws_o + slot * kD + e0) = acc4;
      if (e0 == 0) p.ws_lse[slot] = Ls > 0.f ? fin[2 * h] + log2f(Ls) : -INFINITY;
    }
  }
}

template <int NT, bool kFp8>
pa_status launch_split_tc(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p,
                          dim3 grid, int G, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_raised{0};
  auto kern = paged_decode_split_tc_kernel<NT, kFp8>;
  constexpr int kSmem = TcLayout<kFp8>::kAlloc;
  if (!ensure_smem_limit(kern, kSmem, smem_raised)) return PA_ERR_CUDA;
  kern<<<grid, kThreads, kSmem, stream>>>(mk, mv, p, G);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

// ------------------------------------------------------- tensor maps --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load();
  if (f == nullptr) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn.store(f);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// [rows, H_KV, 128] bf16 viewed 3-D; box = 64 elements (one 128-byte half
// row) x 1 head x box_rows rows, landing 128-byte swizzled in shared memory.
bool make_kv_map_swizzled(CUtensorMap* map, const void* base, int64_t rows, int32_t num_kv_heads,
                          int32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes),
                                 static_cast<cuuint64_t>(kRowBytes) * num_kv_heads};
  const cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, H_KV, 128] e4m3 viewed 3-D as bytes; box = a whole 128-byte row x
// 1 head x box_rows rows, 128-byte swizzled.
bool make_kv_map_fp8(CUtensorMap* map, const void* base, int64_t rows, int32_t num_kv_heads,
                     int32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD),
                                 static_cast<cuuint64_t>(kD) * num_kv_heads};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), 1u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scratch of the allocation-free decode entry point.  Every GPU that loads
// this library holds these 16 MiB for the life of the process.  Host code
// must not use the name as an address: static_decode_scratch_address() asks
// the runtime for the device address.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_static_decode_scratch[kStaticScratchBytes];

size_t static_decode_scratch_bytes() { return kStaticScratchBytes; }

pa_status static_decode_scratch_address(void** ptr) {
  static std::atomic<void*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  const bool cacheable = dev >= 0 && dev < 64;
  if (cacheable) {
    void* p = cache[dev].load();
    if (p != nullptr) {
      *ptr = p;
      return PA_OK;
    }
  }
  // set-up, once per device, with that device current
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_decode_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  if (cacheable) cache[dev].store(p);
  *ptr = p;
  return PA_OK;
}

DecodePlan make_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len,
                            int32_t num_sms) {
  if (num_sms <= 0) num_sms = 148;
  if (max_context_len <= 0 || num_seqs <= 0 || num_kv_heads <= 0) return {1, kTile};
  const int64_t tiles_max = (static_cast<int64_t>(max_context_len) + kTile - 1) / kTile;
  const int64_t work = static_cast<int64_t>(num_seqs) * num_kv_heads;  // CTAs per split index
  const int64_t target = 32ll * num_sms;  // aim for ~32 CTAs per SM over the whole grid
  int64_t splits = (target + work - 1) / work;
  if (splits < 1) splits = 1;
  if (splits > tiles_max) splits = tiles_max;
  if (splits > 65535) splits = 65535;  // the grid's y extent
  const int64_t tiles_per_split = (tiles_max + splits - 1) / splits;
  splits = (tiles_max + tiles_per_split - 1) / tiles_per_split;
  return {static_cast<int32_t>(splits), static_cast<int32_t>(tiles_per_split * kTile)};
}

namespace {
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

// Workspace: [error word | pad to 256] [split counters: B*H_KV u32, padded]
//            [lse partials: B*H_Q*splits f32, padded] [output partials:
//            B*H_Q*splits*d f32].  One split needs the header only.
size_t decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_size, const DecodePlan& plan) {
  size_t bytes = kWorkspaceHeader;
  if (plan.num_splits > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * plan.num_splits;
    bytes += align256(static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(unsigned));
    bytes += align256(rows * sizeof(float));
    bytes += rows * static_cast<size_t>(head_size) * sizeof(float);
  }
  return bytes;
}

pa_status launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return PA_OK;
  const int32_t G = a.num_q_heads / a.num_kv_heads;
  const int64_t rows = a.num_blocks * a.block_size;
  const int32_t box_rows = a.block_size < kTile ? a.block_size : kTile;
  const bool fp8 = a.cache_dtype == PA_FP8_E4M3;
  CUtensorMap mk, mv;
  const bool maps_ok =
      fp8 ? make_kv_map_fp8(&mk, a.k_cache, rows, a.num_kv_heads, box_rows) &&
                make_kv_map_fp8(&mv, a.v_cache, rows, a.num_kv_heads, box_rows)
          : make_kv_map_swizzled(&mk, a.k_cache, rows, a.num_kv_heads, box_rows) &&
                make_kv_map_swizzled(&mv, a.v_cache, rows, a.num_kv_heads, box_rows);
  if (!maps_ok) return PA_ERR_CUDA;

  DecodeParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.err = a.error_word != nullptr ? a.error_word : reinterpret_cast<unsigned*>(ws);
  const size_t nrows = static_cast<size_t>(a.num_seqs) * a.num_q_heads * a.plan.num_splits;
  const size_t ctr_bytes = align256(static_cast<size_t>(a.num_seqs) * a.num_kv_heads * 4);
  p.counters = reinterpret_cast<unsigned*>(ws + kWorkspaceHeader);
  p.ws_lse = reinterpret_cast<float*>(ws + kWorkspaceHeader + ctr_bytes);
  p.ws_o = reinterpret_cast<float*>(ws + kWorkspaceHeader + ctr_bytes + align256(nrows * 4));
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  int lg = 0;
  while ((1 << lg) < a.block_size) ++lg;
  p.log2_bs = lg;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_splits = a.plan.num_splits;
  p.tokens_per_split = a.plan.tokens_per_split;
  p.scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.new_k = static_cast<const __nv_bfloat16*>(a.new_k);
  p.new_v = static_cast<const __nv_bfloat16*>(a.new_v);
  p.slot_mapping = a.slot_mapping;
  p.k_cache = const_cast<void*>(a.k_cache);
  p.v_cache = const_cast<void*>(a.v_cache);

  if (a.plan.num_splits > 65535 || a.num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(a.num_kv_heads), static_cast<unsigned>(a.plan.num_splits),
                  static_cast<unsigned>(a.num_seqs));
  pa_status st;
  switch (G) {
    case 1: case 2: case 4: case 8:
      st = fp8 ? launch_split_tc<1, true>(mk, mv, p, grid, G, stream)
               : launch_split_tc<1, false>(mk, mv, p, grid, G, stream);
      break;
    case 16:
      st = fp8 ? launch_split_tc<2, true>(mk, mv, p, grid, G, stream)
               : launch_split_tc<2, false>(mk, mv, p, grid, G, stream);
      break;
    default: return PA_ERR_UNSUPPORTED;
  }
  return st;
}

}  // namespace pa_detail
