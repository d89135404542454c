// prefill.cu -- causal varlen prefill attention over the paged cache.
//
// What is computed: sequence b has n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b]
// new tokens, the last n_b of its context_lens[b] = L_b cached tokens (the
// cache write has already stored their K/V).  New token j sits at position
// p = L_b - n_b + j and attends causally to tokens 0..p, read back from the
// paged cache along the block table (nano-vLLM walkthrough, section 2.6:
// attention reads the physical blocks via block_tables; the walkthrough names
// varlen flash prefill with cu_seqlens_q).  Query head h uses KV head
// h / G.  Output [total_new_tokens, H_Q, 128] bf16.
//
// How (sm_103a), FlashAttention-2 style on the tensor cores:
//  * grid = (query tile, kv head, sequence); a CTA owns 64 rows = 64/G new
//    tokens x the G query heads of one kv head, so every K/V byte it loads
//    serves G heads.  Tiles are issued heaviest (latest positions) first.
//  * one producer warp streams the key tiles 0..p_max of the sequence through
//    the same 128-byte-swizzled TMA ring as decode (64 keys per stage, one box
//    per block, K|V and half row, evict-first).
//  * four consumer warps own 16 rows each: S = Q.K^T with mma.sync
//    m16n8k16 (Q fragments in registers, K fragments by ldmatrix), causal and
//    validity masks, an fp32 online softmax (base 2, lazy rescale), and
//    O += P.V with P taken straight from the S accumulators (rounded to
//    bf16) and V fragments by ldmatrix.trans.
// Every mbarrier wait is bounded (2 s), as in decode.
#include <atomic>
#include <climits>

#include "pa_internal.cuh"

namespace pa_detail {
namespace {

using namespace pa;

constexpr int kD = 128;
constexpr int kTile = 64;          // keys per stage
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;  // 16 rows each
constexpr int kRows = 16 * kConsumerWarps;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHalfBytes = kTile * 128;          // [64 rows x 128 B] region
constexpr int kStageBytes = 4 * kHalfBytes;      // K_lo, K_hi, V_lo, V_hi
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kSmemBytes = kBarOffset + 3 * kStages * 8 + 16 + 1024;
constexpr float kRescaleLog2 = 8.0f;

struct PrefillParams {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  unsigned* err;
  int64_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t tokens_per_cta;  // kRows / group
  int32_t block_size;
  int32_t log2_bs;
  int32_t max_blocks_per_seq;
  float scale_log2;
};

__global__ void __launch_bounds__(kThreads, 2)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* tile_mask = empty + kStages;
  int* abort_ptr = reinterpret_cast<int*>(tile_mask + kStages);

  const int qtile = gridDim.x - 1 - blockIdx.x;  // latest positions first
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int bs = p.block_size;

  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int n = __ldg(p.cu_seqlens_q + b + 1) - q0;
  int L = __ldg(p.context_lens + b);
  const int Lcap = p.max_blocks_per_seq * bs;
  if (L > Lcap) {
    if (qtile == 0 && g == 0 && threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_CONTEXT_CLIPPED);
    L = Lcap;
  }
  const int qt0 = qtile * p.tokens_per_cta;
  if (qt0 >= n) return;
  const int ntok = min(p.tokens_per_cta, n - qt0);
  const int pos0 = L - n + qt0;         // position of the CTA's first token
  const int kend = min(L, pos0 + ntok);  // keys 0 .. kend-1 are needed
  const int ntiles = kend > 0 ? (kend + kTile - 1) / kTile : 0;

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
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      if (t >= kStages) {
        const bool w_ok = mbar_wait_bounded(&empty[stage], ((t / kStages) - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
      }
      const int tok0 = t * kTile;
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
      uint64_t bits = 0;
      if (valid) bits = (rows >= 64 ? ~0ull : ((1ull << rows) - 1ull)) << (lane * rpb);
      const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits));
      const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bits >> 32));
      const uint32_t vb = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) {
        tile_mask[stage] = (static_cast<uint64_t>(hi) << 32) | lo;
        mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(__popc(vb) * rpb * 256 * 2));
      }
      __syncwarp();
      if (valid) {
        const int32_t row = bid * bs + row0;
        uint8_t* st = smem + stage * kStageBytes + lane * rpb * 128;
        tma_load_3d(st + 0 * kHalfBytes, &tm_k, 0, g, row, &full[stage], pol);
        tma_load_3d(st + 1 * kHalfBytes, &tm_k, 64, g, row, &full[stage], pol);
        tma_load_3d(st + 2 * kHalfBytes, &tm_v, 0, g, row, &full[stage], pol);
        tma_load_3d(st + 3 * kHalfBytes, &tm_v, 64, g, row, &full[stage], pol);
      }
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
    __syncthreads();
    if (*abort_flag && lane == 0) {
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait_bounded(&full[t % kStages], (t / kStages) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gq = lane >> 2;
  const int tq = lane & 3;
  // this lane's two rows (gq and gq + 8 of the warp's 16): token, head, position
  int pos[2];
  bool rvalid[2];
  int64_t qrow[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = warp * 16 + gq + 8 * i;
    const int tok = r / G;
    rvalid[i] = tok < ntok;
    pos[i] = pos0 + tok;
    qrow[i] = (static_cast<int64_t>(q0 + qt0 + (rvalid[i] ? tok : 0)) * p.num_q_heads + g * G +
               r % G) * kD;
  }
  // Q as the A operand: a0/a2 row gq, a1/a3 row gq + 8; d = 16kk + 2tq (+8)
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(p.q + qrow[i]);
      qa[kk][i] = rvalid[i] ? __ldg(src + 8 * kk + tq) : 0u;
      qa[kk][i + 2] = rvalid[i] ? __ldg(src + 8 * kk + tq + 4) : 0u;
    }
  }
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nt][c] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  // the warp's smallest position: tiles entirely at or below it need no causal mask
  const int pos_min = __reduce_min_sync(0xffffffffu, rvalid[0] ? pos[0] : INT_MAX);
  const uint32_t smem_base = smem_u32(smem);
  const int sw = lane & 7;

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int stage = t % kStages;
    const bool w_ok = mbar_wait_bounded(&full[stage], (t / kStages) & 1, abort_flag);
    if (!__all_sync(0xffffffffu, w_ok)) {
      ok = false;
      break;
    }
    const uint64_t mask = tile_mask[stage];
    const int kt0 = t * kTile;
    const uint32_t st_base = smem_base + stage * kStageBytes;
    if (mask != ~0ull) {
      // keys without a cache row: zero their V rows (0 x NaN would poison P.V).
      // Every consumer warp reads every row, so each warp zeroes all of them
      // itself before reading: the writes agree, and no warp waits on another.
      uint8_t* vrow0 = smem + stage * kStageBytes + 2 * kHalfBytes;
      for (int idx = lane; idx < kTile * 16; idx += 32) {
        const int rr = idx >> 4, unit = idx & 15;
        if (!((mask >> rr) & 1ull))
          *reinterpret_cast<uint4*>(vrow0 + (unit >> 3) * kHalfBytes + rr * 128 + (unit & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
    // ---- S = Q . K^T over 64 keys (8 n-tiles of 8 keys)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[nt][c] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint32_t r[4];
        const int key = 16 * kp + (lane & 7) + 8 * (lane >> 4);
        const uint32_t u = static_cast<uint32_t>(((2 * kk) & 7) + ((lane >> 3) & 1));
        ldsm_x4(st_base + (kk >> 2) * kHalfBytes + key * 128 + ((u ^ sw) << 4), r);
        mma_bf16_16816(s[2 * kp], qa[kk], r[0], r[1]);
        mma_bf16_16816(s[2 * kp + 1], qa[kk], r[2], r[3]);
      }
    }
    // ---- masks, online softmax
    const bool full_tile = mask == ~0ull && kt0 + kTile - 1 <= pos_min;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = c >> 1;
        const int kl = 8 * nt + 2 * tq + (c & 1);
        float v = s[nt][c] * p.scale_log2;
        if (!full_tile) {
          const bool keep = rvalid[i] && ((mask >> kl) & 1ull) && kt0 + kl <= pos[i];
          v = keep ? v : -INFINITY;
        }
        s[nt][c] = v;
        mx[i] = fmaxf(mx[i], v);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      if (mx[i] > m[i] + kRescaleLog2) {  // new running max (always on the first)
        const float corr = exp2f(m[i] - mx[i]);
        l[i] *= corr;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][2 * i] *= corr;
          o[nt][2 * i + 1] *= corr;
        }
        m[i] = mx[i];
      }
    }
    // P in place of S, rounded to bf16 as the A operand of P.V
    uint32_t pa_[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float pv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = c >> 1;
        pv[c] = s[nt][c] == -INFINITY ? 0.f : exp2f(s[nt][c] - m[i]);
        l[i] += pv[c];
      }
      pa_[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(pv[0], pv[1]);
      pa_[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
    }
    // ---- O += P . V (16 n-tiles of 8 head elements, 4 k-steps of 16 keys)
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      // A fragment order a0..a3: (row gq, keys lo), (row gq+8, keys lo),
      // (row gq, keys hi), (row gq+8, keys hi)
      const uint32_t a[4] = {pa_[kp][0], pa_[kp][1], pa_[kp][2], pa_[kp][3]};
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t r[4];
        const int key = 16 * kp + (lane & 7) + 8 * ((lane >> 3) & 1);
        const uint32_t u = static_cast<uint32_t>(((2 * dp) & 7) + (lane >> 4));
        ldsm_x4_trans(st_base + (2 + (dp >> 2)) * kHalfBytes + key * 128 + ((u ^ sw) << 4), r);
        mma_bf16_16816(o[2 * dp], a, r[0], r[1]);
        mma_bf16_16816(o[2 * dp + 1], a, r[2], r[3]);
      }
    }
    if (mask != ~0ull) fence_proxy_async_smem();  // generic writes before the next TMA
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
  }
  __syncthreads();
  if (*abort_flag) return;

  // ------------------------------------------------------------ epilogue
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!rvalid[i]) continue;
    const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
    __nv_bfloat16* dst = p.out + qrow[i];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<uint32_t*>(dst + 8 * nt + 2 * tq) =
          pack_bf16x2(o[nt][2 * i] * inv, o[nt][2 * i + 1] * inv);
  }
}

}  // namespace

pa_status launch_paged_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.max_q_len == 0) return PA_OK;
  return launch_paged_prefill_tc(a, stream);
}

// the mma.sync kernel above (64-row tiles), kept for comparison
pa_status launch_paged_prefill_mma(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.max_q_len == 0) return PA_OK;
  const int32_t G = a.num_q_heads / a.num_kv_heads;
  const int64_t rows = a.num_blocks * a.block_size;
  const int32_t box_rows = a.block_size < kTile ? a.block_size : kTile;
  CUtensorMap mk, mv;
  if (!make_kv_map_swizzled(&mk, a.k_cache, rows, a.num_kv_heads, box_rows) ||
      !make_kv_map_swizzled(&mv, a.v_cache, rows, a.num_kv_heads, box_rows))
    return PA_ERR_CUDA;
  PrefillParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.cu_seqlens_q = a.cu_seqlens_q;
  p.context_lens = a.context_lens;
  p.err = a.error_word;
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = G;
  p.tokens_per_cta = kRows / G;
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
    if (cudaFuncSetAttribute(paged_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_set.store(true);
  }
  const dim3 grid(static_cast<unsigned>(qtiles), static_cast<unsigned>(a.num_kv_heads),
                  static_cast<unsigned>(a.num_seqs));
  paged_prefill_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
