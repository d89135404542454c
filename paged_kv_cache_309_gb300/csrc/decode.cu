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
//    looks up the tile's physical blocks in the block table and issues one
//    3-D TMA copy per (block, K|V) -- a [rows, 128] box of one KV head --
//    into a 3-stage shared-memory ring, signalling an mbarrier with the
//    byte count; a per-tile 64-bit mask marks the rows that exist (inside
//    the context and in a valid block).  The L2 policy is evict-first: the
//    K/V stream is read once.
//  * four consumer warps compute on CUDA cores in fp32.  A warp splits into
//    groups of LPT lanes, one token per group; a lane holds 128/LPT
//    elements of q (for all G heads, pre-multiplied by scale*log2(e)) and of
//    the output accumulator.  Scores are reduced across the group with
//    shuffles; the softmax is online in base 2 with a lazy rescale (the
//    running max moves only when a score exceeds it by more than 2^8, so the
//    accumulator is almost never rescaled); packed fp32x2 FMAs halve the
//    issue count of both products.
//  * epilogue: the groups' (max, sum, accumulator) are merged in shared
//    memory; one split writes bf16 directly, several splits write an fp32
//    partial and its log2-sum-exp to the workspace and a second kernel
//    merges them.
//
// Every mbarrier wait is bounded (2 s); a timeout sets an error bit in the
// workspace's error word, drains the copies already issued, and exits.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>

#include "pa_internal.cuh"

namespace pa_detail {
namespace {

constexpr int kD = 128;                 // head size handled by this kernel
constexpr int kTile = 64;               // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kStages = 3;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowBytes = kD * 2;       // one bf16 row of one KV head
constexpr int kTileBytes = kTile * kRowBytes;
constexpr float kRescaleLog2 = 8.0f;    // lazy-rescale threshold (base-2 units)
constexpr int kMergeWarps = 4;
constexpr size_t kWorkspaceHeader = 256;  // error word + padding

struct __align__(128) DecodeSmem {
  uint8_t kv[kStages][2][kTileBytes];  // [stage][K, V][64 rows x 256 B]
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t mask[kStages];
  int abort_flag;
};

struct DecodeParams {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_lse;
  float* ws_o;
  unsigned* err;
  int64_t num_blocks;
  int32_t num_q_heads;
  int32_t block_size;
  int32_t log2_bs;
  int32_t max_blocks_per_seq;
  int32_t num_splits;
  int32_t tokens_per_split;
  float scale_log2;
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

// lane's VEC-element slice `ld` of a bf16 row in shared memory -> fp32 pairs
template <int VEC>
__device__ __forceinline__ void lds_row_pairs(const uint8_t* row, int elem0, float2* out) {
  if constexpr (VEC == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + elem0 * 2);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      out[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
  } else {
    static_assert(VEC == 4, "VEC must be 4 or 8");
    const uint2 u = *reinterpret_cast<const uint2*>(row + elem0 * 2);
    out[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u));
    out[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  }
}

template <int G, int LPT>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using namespace pa;
  constexpr int EPL = kD / LPT;            // elements per lane
  constexpr int VEC = EPL < 8 ? EPL : 8;   // elements per shared-memory load
  constexpr int NLD = EPL / VEC;           // loads per row per lane
  constexpr int NP = EPL / 2;              // fp32 pairs per lane
  constexpr int PPL = VEC / 2;             // pairs per load
  constexpr int GPW = 32 / LPT;            // token groups per warp
  constexpr int NG = kConsumerWarps * GPW; // token groups per CTA
  constexpr int TPW = kTile / kConsumerWarps;
  constexpr int STEPS = TPW / GPW;
  static_assert(NG * G * (kD + 3) * 4 + 2 * G * 4 <= static_cast<int>(sizeof(DecodeSmem::kv)),
                "epilogue scratch must fit in the stage buffers");

  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);

  const int split = blockIdx.x;
  const int g = blockIdx.y;
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
    if (p.num_splits == 1) {  // empty context: a zero row per head
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
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    sm.abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  float m[G], l[G];
  float2 acc[G][NP];
  int issued = 0;
  const int grp = lane / LPT;
  const int j = lane % LPT;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int rpb = bs < kTile ? bs : kTile;  // rows per TMA box
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
        // every lane waits; the outcome is made warp-uniform before any
        // full-mask collective below
        const bool w_ok = mbar_wait_bounded(&sm.empty[stage], ((t / kStages) - 1) & 1, abort_flag);
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
        sm.mask[stage] = (static_cast<uint64_t>(hi) << 32) | lo;
        mbar_arrive_expect_tx(&sm.full[stage],
                              static_cast<uint32_t>(__popc(vb) * rpb * kRowBytes * 2));
      }
      __syncwarp();
      if (valid) {
        const int32_t row = bid * bs + row0;  // physical row index (< 2^31, checked on host)
        tma_load_3d(sm.kv[stage][0] + lane * rpb * kRowBytes, &tm_k, 0, g, row, &sm.full[stage],
                    pol);
        tma_load_3d(sm.kv[stage][1] + lane * rpb * kRowBytes, &tm_v, 0, g, row, &sm.full[stage],
                    pol);
      }
      issued = t + 1;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ consumers
    float2 q2[G][NP];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(
          p.q + (static_cast<int64_t>(b) * p.num_q_heads + hq0 + h) * kD);
#pragma unroll
      for (int ld = 0; ld < NLD; ++ld) {
        float2 t2[PPL];
        // q is tiny and read once per CTA: plain global loads
        if constexpr (VEC == 8) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(qrow + (j + LPT * ld) * VEC * 2));
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            t2[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
        } else {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(qrow + (j + LPT * ld) * VEC * 2));
          t2[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u));
          t2[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
        }
#pragma unroll
        for (int i = 0; i < PPL; ++i)
          q2[h][ld * PPL + i] = make_float2(t2[i].x * p.scale_log2, t2[i].y * p.scale_log2);
      }
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < NP; ++i) acc[h][i] = make_float2(0.f, 0.f);
    }

    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % kStages;
      const bool w_ok = mbar_wait_bounded(&sm.full[stage], (t / kStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w_ok)) {  // warp-uniform before the shuffles below
        ok = false;
        break;
      }
      const uint64_t mask = sm.mask[stage];
      const uint8_t* kb = sm.kv[stage][0];
      const uint8_t* vbuf = sm.kv[stage][1];
#pragma unroll 2
      for (int step = 0; step < STEPS; ++step) {
        const int r = warp * TPW + step * GPW + grp;
        const bool valid = (mask >> r) & 1ull;
        float2 kf[NP];
#pragma unroll
        for (int ld = 0; ld < NLD; ++ld)
          lds_row_pairs<VEC>(kb + r * kRowBytes, (j + LPT * ld) * VEC, kf + ld * PPL);
        float s[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < NP; i += 2) {
            a0 = __ffma2_rn(q2[h][i], kf[i], a0);
            if (i + 1 < NP) a1 = __ffma2_rn(q2[h][i + 1], kf[i + 1], a1);
          }
          s[h] = (a0.x + a0.y) + (a1.x + a1.y);
        }
#pragma unroll
        for (int off = LPT / 2; off >= 1; off >>= 1) {
#pragma unroll
          for (int h = 0; h < G; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], off);
        }
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float sv = valid ? s[h] : -INFINITY;
          if (sv > m[h] + kRescaleLog2) {  // new running max (always taken first)
            const float corr = exp2f(m[h] - sv);
            l[h] *= corr;
#pragma unroll
            for (int i = 0; i < NP; ++i) {
              acc[h][i].x *= corr;
              acc[h][i].y *= corr;
            }
            m[h] = sv;
          }
          pr[h] = valid ? exp2f(sv - m[h]) : 0.f;
          l[h] += pr[h];
        }
        if (valid) {
          float2 vf[NP];
#pragma unroll
          for (int ld = 0; ld < NLD; ++ld)
            lds_row_pairs<VEC>(vbuf + r * kRowBytes, (j + LPT * ld) * VEC, vf + ld * PPL);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float2 pp = make_float2(pr[h], pr[h]);
#pragma unroll
            for (int i = 0; i < NP; ++i) acc[h][i] = __ffma2_rn(pp, vf[i], acc[h][i]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) atomicOr(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }
  }

  __syncthreads();
  if (sm.abort_flag) {
    // wait (bounded) for copies already in flight before the CTA retires
    if (warp == kConsumerWarps && lane == 0) {
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait_bounded(&sm.full[t % kStages], (t / kStages) & 1, nullptr);
    }
    return;
  }

  // ------------------------------------------------------------ epilogue
  float* red = reinterpret_cast<float*>(&sm.kv[0][0][0]);  // [NG][G][kD]
  float* red_m = red + NG * G * kD;                         // [NG][G]
  float* red_l = red_m + NG * G;                            // [NG][G]
  float* red_w = red_l + NG * G;                            // [NG][G]
  float* fin = red_w + NG * G;                              // [G][2]
  if (warp < kConsumerWarps) {
    const int gid = warp * GPW + grp;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* dst = red + (gid * G + h) * kD;
#pragma unroll
      for (int ld = 0; ld < NLD; ++ld) {
        const int e0 = (j + LPT * ld) * VEC;
#pragma unroll
        for (int i = 0; i < PPL; i += 2) {
          const float2 a = acc[h][ld * PPL + i];
          const float2 c = acc[h][ld * PPL + i + 1];
          *reinterpret_cast<float4*>(dst + e0 + 2 * i) = make_float4(a.x, a.y, c.x, c.y);
        }
      }
      if (j == 0) {
        red_m[gid * G + h] = m[h];
        red_l[gid * G + h] = l[h];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = -INFINITY;
#pragma unroll 4
    for (int gg = 0; gg < NG; ++gg) M = fmaxf(M, red_m[gg * G + h]);
    float Ls = 0.f;
    for (int gg = 0; gg < NG; ++gg) {
      const float w = (M == -INFINITY) ? 0.f : exp2f(red_m[gg * G + h] - M);
      red_w[gg * G + h] = w;
      Ls += red_l[gg * G + h] * w;
    }
    fin[2 * h] = M;
    fin[2 * h + 1] = Ls;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * (kD / 4); i += kThreads) {
    const int h = i / (kD / 4);
    const int e0 = (i % (kD / 4)) * 4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int gg = 0; gg < NG; ++gg) {
      const float w = red_w[gg * G + h];
      const float4 v = *reinterpret_cast<const float4*>(red + (gg * G + h) * kD + e0);
      o.x += w * v.x;
      o.y += w * v.y;
      o.z += w * v.z;
      o.w += w * v.w;
    }
    const float Ls = fin[2 * h + 1];
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
    const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + hq0 + h;
    if (p.num_splits == 1) {
      const uint32_t w0 = __bfloat16_as_ushort(__float2bfloat16_rn(o.x)) |
                          (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o.y))) << 16);
      const uint32_t w1 = __bfloat16_as_ushort(__float2bfloat16_rn(o.z)) |
                          (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o.w))) << 16);
      *reinterpret_cast<uint2*>(p.out + row * kD + e0) = make_uint2(w0, w1);
    } else {
      const int64_t slot = row * p.num_splits + split;
      *reinterpret_cast<float4*>(p.ws_o + slot * kD + e0) = o;
      if (e0 == 0) p.ws_lse[slot] = Ls > 0.f ? fin[2 * h] + log2f(Ls) : -INFINITY;
    }
  }
}

// One warp per (sequence, query head): weights 2^(lse_s - max) over the
// splits that hold tokens, out = sum_s w_s o_s / sum_s w_s, rounded to bf16.
__global__ void __launch_bounds__(kMergeWarps * 32)
    paged_decode_merge_kernel(const DecodeParams p, int32_t num_seqs) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t bh = static_cast<int64_t>(blockIdx.x) * kMergeWarps + warp;
  if (bh >= static_cast<int64_t>(num_seqs) * p.num_q_heads) return;
  const int b = static_cast<int>(bh / p.num_q_heads);
  bool clipped;
  const int L = effective_len(p, b, &clipped);
  const int n = (L + p.tokens_per_split - 1) / p.tokens_per_split;
  const float* lse = p.ws_lse + bh * p.num_splits;
  const float* o = p.ws_o + bh * p.num_splits * kD;

  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < n; s0 += 32) {
      const int my = s0 + lane;
      const float wl = my < n ? exp2f(lse[my] - M) : 0.f;
      const int cnt = min(32, n - s0);
      int k = 0;
      for (; k + 4 <= cnt; k += 4) {
        float4 v[4];
        float w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          v[u] = *reinterpret_cast<const float4*>(o + static_cast<int64_t>(s0 + k + u) * kD + lane * 4);
          w[u] = __shfl_sync(0xffffffffu, wl, k + u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          W += w[u];
          acc.x += w[u] * v[u].x;
          acc.y += w[u] * v[u].y;
          acc.z += w[u] * v[u].z;
          acc.w += w[u] * v[u].w;
        }
      }
      for (; k < cnt; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(o + static_cast<int64_t>(s0 + k) * kD + lane * 4);
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
  const uint32_t w0 = __bfloat16_as_ushort(__float2bfloat16_rn(acc.x * inv)) |
                      (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y * inv))) << 16);
  const uint32_t w1 = __bfloat16_as_ushort(__float2bfloat16_rn(acc.z * inv)) |
                      (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w * inv))) << 16);
  *reinterpret_cast<uint2*>(p.out + bh * kD + lane * 4) = make_uint2(w0, w1);
}

// ---------------------------------------------------------------- host --
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

bool make_kv_map(CUtensorMap* map, const void* base, int64_t rows, int32_t num_kv_heads,
                 int32_t box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kRowBytes),
                                 static_cast<cuuint64_t>(kRowBytes) * num_kv_heads};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), 1u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G, int LPT>
pa_status launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& p,
                       dim3 grid, cudaStream_t stream) {
  static std::atomic<bool> attr_set{false};
  auto kern = paged_decode_split_kernel<G, LPT>;
  if (!attr_set.load()) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(DecodeSmem))) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_set.store(true);
  }
  kern<<<grid, kThreads, sizeof(DecodeSmem), stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

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
  const int64_t tiles_per_split = (tiles_max + splits - 1) / splits;
  splits = (tiles_max + tiles_per_split - 1) / tiles_per_split;
  return {static_cast<int32_t>(splits), static_cast<int32_t>(tiles_per_split * kTile)};
}

size_t decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                              const DecodePlan& plan) {
  size_t bytes = kWorkspaceHeader;
  if (plan.num_splits > 1) {
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * plan.num_splits;
    bytes += (rows * sizeof(float) + 255) / 256 * 256;         // lse partials
    bytes += rows * static_cast<size_t>(head_size) * sizeof(float);  // output partials
  }
  return bytes;
}

pa_status launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return PA_OK;
  const int32_t G = a.num_q_heads / a.num_kv_heads;
  const int64_t rows = a.num_blocks * a.block_size;
  const int32_t box_rows = a.block_size < kTile ? a.block_size : kTile;
  CUtensorMap mk, mv;
  if (!make_kv_map(&mk, a.k_cache, rows, a.num_kv_heads, box_rows) ||
      !make_kv_map(&mv, a.v_cache, rows, a.num_kv_heads, box_rows))
    return PA_ERR_CUDA;

  DecodeParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.err = a.error_word != nullptr ? a.error_word : reinterpret_cast<unsigned*>(ws);
  const size_t nrows = static_cast<size_t>(a.num_seqs) * a.num_q_heads * a.plan.num_splits;
  p.ws_lse = reinterpret_cast<float*>(ws + kWorkspaceHeader);
  p.ws_o = reinterpret_cast<float*>(ws + kWorkspaceHeader + (nrows * sizeof(float) + 255) / 256 * 256);
  p.num_blocks = a.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.block_size = a.block_size;
  int lg = 0;
  while ((1 << lg) < a.block_size) ++lg;
  p.log2_bs = lg;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_splits = a.plan.num_splits;
  p.tokens_per_split = a.plan.tokens_per_split;
  p.scale_log2 = a.scale * 1.4426950408889634f;  // log2(e)

  const dim3 grid(static_cast<unsigned>(a.plan.num_splits), static_cast<unsigned>(a.num_kv_heads),
                  static_cast<unsigned>(a.num_seqs));
  pa_status st;
  switch (G) {
    case 1: st = launch_split<1, 8>(mk, mv, p, grid, stream); break;
    case 2: st = launch_split<2, 8>(mk, mv, p, grid, stream); break;
    case 4: st = launch_split<4, 8>(mk, mv, p, grid, stream); break;
    case 8: st = launch_split<8, 16>(mk, mv, p, grid, stream); break;
    case 16: st = launch_split<16, 32>(mk, mv, p, grid, stream); break;
    default: return PA_ERR_UNSUPPORTED;
  }
  if (st != PA_OK || a.plan.num_splits == 1) return st;
  const int64_t bh = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  const int64_t blocks = (bh + kMergeWarps - 1) / kMergeWarps;
  paged_decode_merge_kernel<<<static_cast<unsigned>(blocks), kMergeWarps * 32, 0, stream>>>(
      p, a.num_seqs);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_detail
