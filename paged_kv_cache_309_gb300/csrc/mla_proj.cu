// mla_proj.cu -- the two per-head products that put MLA decode in its
// absorbed form (PagedAttention-principle post, MLA section: K and V of head
// h are c_kv W_UK_h and c_kv W_UV_h with W_UK, W_UV: [d_c, H * d_h] and
// head h owning columns h*d_h .. (h+1)*d_h - 1):
//   absorb:  q_lat[b, h, c]  = sum_i q_nope[b, h, i] * W_UK[c, h*d_h + i]   (c < d_c)
//            q_lat[b, h, d_c + r] = q_pe[b, h, r]
//   project: out[b, h, i]    = sum_c o_lat[b, h, c] * W_UV[c, h*d_v + i]
// Both are Y_h = X_h . W_h per head, bf16 in, fp32 accumulate, bf16 out, on
// the tensor cores (mma.sync m16n8k16).  A CTA owns 64 rows (sequences) of
// one head and a group of 64-column output chunks; it walks its (column
// chunk, 64-wide K chunk) steps through a 3-stage cp.async ring of 64 x 64
// operand tiles (16 bytes of padding per row, so the eight rows of an
// ldmatrix phase hit eight different bank groups), accumulating a 64 x 64
// chunk in four warps of 16 rows.  At decode batch sizes the weights are the
// bytes that matter: every weight element is read once per 64 sequences, and
// two column groups per head make one wave of CTAs.
// W_UK_h is read with rows = outputs (ldmatrix), W_UV_h with rows = the
// reduction index (ldmatrix.trans).
#include <atomic>

#include "pa_internal.cuh"

namespace pa_detail {
namespace {

using namespace pa;

constexpr int kTM = 64, kTN = 64, kTK = 64;   // CTA rows, column chunk, K chunk
constexpr int kPad = 72;                       // elements per staged row (64 + 8)
constexpr int kTileBytes = 64 * kPad * 2;      // one staged 64 x 64 tile: 9 KB
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kTileBytes;    // X tile, then W tile
constexpr int kSmem = kStages * kStageBytes;   // 54 KB
constexpr int kThreads = 128;
constexpr int kGroups = 2;                     // column groups per head

struct ProjParams {
  __nv_bfloat16* y;        // [M, H, ldy], columns 0..N-1 written
  const __nv_bfloat16* x;  // [M, H, K]
  const __nv_bfloat16* w;
  const __nv_bfloat16* extra;  // absorb: q_pe [M, H, extra_dim] copied to y columns N..
  int32_t M, H, K, N, ldy, extra_dim;
  int32_t chunks_per_group;  // 64-column chunks per CTA
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t"
      "@p cp.async.cg.shared.global [%0], [%1], 16;\n\t"
      "@!p st.shared.v4.u32 [%0], {0, 0, 0, 0};\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

// kTransB = false: W(k, n) = w[n, h*K + k]   (absorb, rows = outputs)
// kTransB = true:  W(k, n) = w[k, h*N + n]   (project, rows = reduction index)
template <bool kTransB>
__global__ void __launch_bounds__(kThreads) mla_head_gemm_kernel(const ProjParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  const int h = blockIdx.y;
  const int m0 = blockIdx.z * kTM;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int64_t xrow = static_cast<int64_t>(p.H) * p.K;
  const int nk = p.K / kTK;
  const int c_first = blockIdx.x * p.chunks_per_group;
  const int c_count = min(p.chunks_per_group, p.N / kTN - c_first);
  const int steps = c_count > 0 ? c_count * nk : 0;

  // step s: column chunk c_first + s / nk, K chunk s % nk; 512 16-byte units
  // per tile, four per thread
  auto load_step = [&](int s) {
    uint8_t* st = dyn + (s % kStages) * kStageBytes;
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(st);
    __nv_bfloat16* ws = reinterpret_cast<__nv_bfloat16*>(st + kTileBytes);
    const int n0 = (c_first + s / nk) * kTN, k0 = (s % nk) * kTK;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = threadIdx.x + kThreads * j;
      const int r = i >> 3, u = i & 7;
      const bool ok = m0 + r < p.M;
      cp_async16(xs + r * kPad + 8 * u,
                 p.x + (ok ? (m0 + r) * xrow : 0) + static_cast<int64_t>(h) * p.K + k0 + 8 * u, ok);
      if constexpr (kTransB)
        cp_async16(ws + r * kPad + 8 * u,
                   p.w + static_cast<int64_t>(k0 + r) * p.H * p.N + static_cast<int64_t>(h) * p.N +
                       n0 + 8 * u,
                   true);
      else
        cp_async16(ws + r * kPad + 8 * u,
                   p.w + static_cast<int64_t>(n0 + r) * p.H * p.K + static_cast<int64_t>(h) * p.K +
                       k0 + 8 * u,
                   true);
    }
  };
  // one commit group per step (empty ones past the end), so that at step s
  // exactly one newer group may still be pending
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < steps) load_step(s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  float acc[kTN / 8][4];
#pragma unroll
  for (int nt = 0; nt < kTN / 8; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
  for (int s = 0; s < steps; ++s) {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();  // step s is in shared memory for all; step s - 1's stage is free
    if (s + kStages - 1 < steps) load_step(s + kStages - 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const uint32_t xs_base = smem_u32(dyn + (s % kStages) * kStageBytes);
    const uint32_t ws_base = xs_base + kTileBytes;
#pragma unroll
    for (int kk = 0; kk < kTK / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(xs_base + static_cast<uint32_t>(((16 * warp + (lane & 15)) * kPad + 16 * kk +
                                              8 * (lane >> 4)) * 2), a);
#pragma unroll
      for (int np = 0; np < kTN / 16; ++np) {
        uint32_t bb[4];
        if constexpr (kTransB) {
          // rows = k: lanes 0-7 k 0-7, 8-15 k 8-15 (n 0-7), 16-31 the same for n 8-15
          const int kr = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x4_trans(ws_base + static_cast<uint32_t>((kr * kPad + 16 * np + 8 * (lane >> 4)) * 2), bb);
        } else {
          // rows = n: lanes 0-7 n 0-7 k 0-7, 8-15 n 0-7 k 8-15, 16-31 the same for n 8-15
          const int nr = 16 * np + (lane & 7) + 8 * (lane >> 4);
          ldsm_x4(ws_base + static_cast<uint32_t>((nr * kPad + 16 * kk + 8 * ((lane >> 3) & 1)) * 2), bb);
        }
        mma_bf16_16816(acc[2 * np], a, bb[0], bb[1]);
        mma_bf16_16816(acc[2 * np + 1], a, bb[2], bb[3]);
      }
    }
    if (s % nk == nk - 1) {
      // the column chunk is complete: write it and start the next
      const int n0 = (c_first + s / nk) * kTN;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int m = m0 + 16 * warp + gq + 8 * r;
        if (m >= p.M) continue;
        __nv_bfloat16* dst = p.y + (static_cast<int64_t>(m) * p.H + h) * p.ldy + n0 + 2 * tq;
#pragma unroll
        for (int nt = 0; nt < kTN / 8; ++nt)
          *reinterpret_cast<uint32_t*>(dst + 8 * nt) =
              pack_bf16x2(acc[nt][2 * r], acc[nt][2 * r + 1]);
      }
#pragma unroll
      for (int nt = 0; nt < kTN / 8; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // absorb: the rope part of the query is copied behind the latent part
  if (p.extra != nullptr && blockIdx.x == 0) {
    const int units = p.extra_dim / 8;
    for (int i = threadIdx.x; i < kTM * units; i += kThreads) {
      const int r = i / units, u = i % units;
      if (m0 + r >= p.M) continue;
      const int64_t row = static_cast<int64_t>(m0 + r) * p.H + h;
      *reinterpret_cast<uint4*>(p.y + row * p.ldy + p.N + 8 * u) =
          __ldg(reinterpret_cast<const uint4*>(p.extra + row * p.extra_dim) + u);
    }
  }
}

template <bool kTransB>
pa_status launch_gemm(ProjParams p, cudaStream_t stream) {
  const int chunks = p.N / kTN;
  const int groups = chunks < kGroups ? chunks : kGroups;
  p.chunks_per_group = (chunks + groups - 1) / groups;
  const dim3 grid(static_cast<unsigned>(groups), static_cast<unsigned>(p.H),
                  static_cast<unsigned>((p.M + kTM - 1) / kTM));
  static std::atomic<uint64_t> smem_raised{0};
  if (!ensure_smem_limit(mla_head_gemm_kernel<kTransB>, kSmem, smem_raised)) return PA_ERR_CUDA;
  mla_head_gemm_kernel<kTransB><<<grid, kThreads, kSmem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

pa_status launch_mla_absorb_q(void* q_latent, const void* q_nope, const void* q_pe,
                              const void* w_uk, int32_t num_seqs, int32_t num_heads,
                              int32_t nope_dim, int32_t rope_dim, int32_t latent_dim,
                              cudaStream_t stream) {
  if (num_seqs == 0) return PA_OK;
  ProjParams p;
  p.y = static_cast<__nv_bfloat16*>(q_latent);
  p.x = static_cast<const __nv_bfloat16*>(q_nope);
  p.w = static_cast<const __nv_bfloat16*>(w_uk);
  p.extra = static_cast<const __nv_bfloat16*>(q_pe);
  p.M = num_seqs;
  p.H = num_heads;
  p.K = nope_dim;
  p.N = latent_dim;
  p.ldy = latent_dim + rope_dim;
  p.extra_dim = rope_dim;
  return launch_gemm<false>(p, stream);
}

pa_status launch_mla_project_out(void* out, const void* out_latent, const void* w_uv,
                                 int32_t num_seqs, int32_t num_heads, int32_t latent_dim,
                                 int32_t v_head_dim, cudaStream_t stream) {
  if (num_seqs == 0) return PA_OK;
  ProjParams p;
  p.y = static_cast<__nv_bfloat16*>(out);
  p.x = static_cast<const __nv_bfloat16*>(out_latent);
  p.w = static_cast<const __nv_bfloat16*>(w_uv);
  p.extra = nullptr;
  p.M = num_seqs;
  p.H = num_heads;
  p.K = latent_dim;
  p.N = v_head_dim;
  p.ldy = v_head_dim;
  p.extra_dim = 0;
  return launch_gemm<true>(p, stream);
}

}  // namespace pa_detail
