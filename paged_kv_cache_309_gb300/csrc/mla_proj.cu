// mla_proj.cu -- the two per-head products that put MLA decode in its
// absorbed form (PagedAttention-principle post, MLA section: K and V of head
// h are c_kv W_UK_h and c_kv W_UV_h with W_UK, W_UV: [d_c, H * d_h] and
// head h owning columns h*d_h .. (h+1)*d_h - 1):
//   absorb:  q_lat[b, h, c]  = sum_i q_nope[b, h, i] * W_UK[c, h*d_h + i]   (c < d_c)
//            q_lat[b, h, d_c + r] = q_pe[b, h, r]
//   project: out[b, h, i]    = sum_c o_lat[b, h, c] * W_UV[c, h*d_v + i]
// Both are Y_h = X_h . W_h per head, bf16 in, fp32 accumulate, bf16 out, on
// the tensor cores (mma.sync m16n8k16).  At decode batch sizes the weights
// are the bytes that matter (16.8 MB per call at 128 heads against ~2 MB of
// activations), read once per 64 sequences, so the kernels are built to keep
// the most weight bytes in flight.
//
// mla_head_gemm_tc_kernel (the benchmark shapes: d_h = d_v = 128, d_c =
// 512, up to 64 sequences): both products on tcgen05, described at its
// definition.  With L2 flushed, B = 64, 128 heads: absorb 13.8 -> 12.4 us,
// project 12.4 -> 10.7 us against the two kernels below.
//
// mla_head_gemm_tma_kernel (K = 128, N a multiple of 128: the absorb
// product at d_h = 128): a CTA owns 64 rows (sequences) of one head and 128
// output columns over the whole reduction.  One thread issues every load of
// the CTA up front -- six 8 KB TMA boxes (64 rows x 128 bytes, 128-byte
// swizzled), two mbarriers, one per 64-wide half of K -- so all 48 KB are in
// flight before any math; 512 CTAs at four per SM make one wave at 128
// heads.  The rope rows of the query are read into registers meanwhile.
// Four warps of 16 rows multiply each half as it lands (ldmatrix on the
// swizzled tiles); the bf16 results go through shared memory and leave as
// full 256-byte rows.  A per-CTA timeline showed the late q_pe copy and
// narrow 8-byte stores dominating an earlier fp32-staged epilogue.  A version
// for larger K split the reduction over clusters of CTAs and summed the fp32
// partials through distributed shared memory; it measured slower than the
// ring kernel below (16.6 against 12.6 us for the output projection at B =
// 64, 128 heads), so that shape stays on the ring kernel.
//
// mla_head_gemm_kernel (every other shape): a CTA owns 64 rows of one head
// and a group of 64-column output chunks, walking its (column chunk, 64-wide
// K chunk) steps through a 3-stage cp.async ring of 64 x 64 operand tiles
// (16 bytes of padding per row, so the eight rows of an ldmatrix phase hit
// eight different bank groups).
// W_UK_h is read with rows = outputs (ldmatrix), W_UV_h with rows = the
// reduction index (ldmatrix.trans).
#include <cudaTypedefs.h>

#include <atomic>

#include "pa_internal.cuh"
#include "tc_ops.cuh"

namespace pa_detail {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();  // decode.cu

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

// ---------------------------------------------------------- TMA path --
constexpr int kBM = 64;                   // sequences per CTA
constexpr int kBN = 128;                  // output columns per CTA
constexpr int kBK = 128;                  // reduction slice per CTA
constexpr int kBox = 64 * 64 * 2;         // one TMA box: 64 rows x 128 bytes
constexpr int kTmaData = 6 * kBox;        // X (2 k halves) + W (2 n halves x 2 k halves)
constexpr int kTmaSmem = kTmaData + 1024 + 64;  // + alignment slack + barriers
constexpr int kPeRegs = 4;                // 16-byte units of q_pe held per thread

struct TmaProjParams {
  __nv_bfloat16* y;            // [M, H, ldy]: columns 0..N-1 written
  const __nv_bfloat16* extra;  // absorb: q_pe [M, H, extra_dim] copied to y columns N..
  int32_t M, H, K, N, ldy, extra_dim;
};

// kTransB = false: W(k, n) = w[n, h*K + k]   (absorb, rows = outputs)
// kTransB = true:  W(k, n) = w[k, h*N + n]   (project, rows = reduction index)
// mx: X [M, H, K] as 3-D {K, H, M}, box {64, 1, 64}; mw: w as 2-D, box {64, 64}.
template <bool kTransB>
__global__ void __launch_bounds__(kThreads) mla_head_gemm_tma_kernel(
    const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
    const TmaProjParams p) {
  extern __shared__ uint8_t dyn_raw[];
  // 128-byte swizzled boxes want 1024-byte aligned destinations
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + kTmaData);
  const int nchunks = p.N / kBN;
  const int h = blockIdx.y / nchunks, nc = blockIdx.y % nchunks;
  const int n0 = nc * kBN, k0 = 0, m0 = blockIdx.z * kBM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  if (tid == 0) {
    prefetch_tensormap(&mx);
    prefetch_tensormap(&mw);
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) {
    // every load of the CTA, issued at once: half kh of the slice is X box
    // kh and the two W boxes of that half (24 KB on bar[kh])
    const uint64_t pol_w = l2_policy_evict_first();   // weights: read once
    const uint64_t pol_x = l2_policy_evict_normal();  // X: shared by the column blocks
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      mbar_arrive_expect_tx(&bar[kh], 3 * kBox);
      tma_load_3d(base + kh * kBox, &mx, k0 + 64 * kh, h, m0, &bar[kh], pol_x);
#pragma unroll
      for (int nh = 0; nh < 2; ++nh) {
        uint8_t* dst = base + (2 + 2 * nh + kh) * kBox;
        if constexpr (kTransB)
          tma_load_2d(dst, &mw, h * p.N + n0 + 64 * nh, k0 + 64 * kh, &bar[kh], pol_w);
        else
          tma_load_2d(dst, &mw, h * p.K + k0 + 64 * kh, n0 + 64 * nh, &bar[kh], pol_w);
      }
    }
  }

  // absorb: the rope part of the query rides behind the latent part; its
  // rows (up to kPeRegs 16-byte units per thread) are read now, while the
  // tiles are in flight, and stored at the end
  const bool copy_pe = p.extra != nullptr && nc == 0;
  const int pe_units = p.extra_dim / 8;
  const bool pe_in_regs = pe_units * kBM <= kPeRegs * kThreads;
  uint4 pe[kPeRegs];
  if (copy_pe && pe_in_regs) {
#pragma unroll
    for (int j = 0; j < kPeRegs; ++j) {
      const int i = tid + kThreads * j;
      const int r = i / pe_units, u = i - (i / pe_units) * pe_units;
      pe[j] = (i < kBM * pe_units && m0 + r < p.M)
                  ? __ldg(reinterpret_cast<const uint4*>(
                              p.extra + (static_cast<int64_t>(m0 + r) * p.H + h) * p.extra_dim) + u)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  }

  float acc[kBN / 8][4];
#pragma unroll
  for (int nt = 0; nt < kBN / 8; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
  bool ok = true;
#pragma unroll
  for (int kh = 0; kh < 2; ++kh) {
    ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(&bar[kh], 0, nullptr));
    if (!ok) break;
    const uint32_t xs = smem_u32(base + kh * kBox);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      const int row = 16 * warp + (lane & 15);
      const int ua = 2 * kk + (lane >> 4);
      ldsm_x4(xs + static_cast<uint32_t>(row * 128 + ((ua ^ (row & 7)) << 4)), a);
#pragma unroll
      for (int np = 0; np < kBN / 16; ++np) {
        const uint32_t ws = smem_u32(base + (2 + 2 * (np >> 2) + kh) * kBox);
        uint32_t bb[4];
        if constexpr (kTransB) {
          // rows = k: lanes 0-7 k 0-7, 8-15 k 8-15 (n 0-7), 16-31 the same for n 8-15
          const int kr = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ub = 2 * (np & 3) + (lane >> 4);
          ldsm_x4_trans(ws + static_cast<uint32_t>(kr * 128 + ((ub ^ (kr & 7)) << 4)), bb);
        } else {
          // rows = n: lanes 0-7 n 0-7 k 0-7, 8-15 n 0-7 k 8-15, 16-31 the same for n 8-15
          const int nr = 16 * (np & 3) + (lane & 7) + 8 * (lane >> 4);
          const int ub = 2 * kk + ((lane >> 3) & 1);
          ldsm_x4(ws + static_cast<uint32_t>(nr * 128 + ((ub ^ (nr & 7)) << 4)), bb);
        }
        mma_bf16_16816(acc[2 * np], a, bb[0], bb[1]);
        mma_bf16_16816(acc[2 * np + 1], a, bb[2], bb[3]);
      }
    }
  }
  if (!ok) {
    // a load never landed (never expected): wait once more, bounded, for the
    // copies still in flight into this CTA's shared memory; the CTA's
    // outputs become NaN
    if (tid == 0) {
      mbar_wait_bounded(&bar[0], 0, nullptr);
      mbar_wait_bounded(&bar[1], 0, nullptr);
    }
  }
  __syncthreads();  // every warp is done with the input tiles

  const float bad = __int_as_float(0x7fc00000);
  // bf16 rows staged in shared memory (Y[64][128], 16-byte chunk c of row r
  // at chunk c ^ (r & 7), so a warp's eight rows hit eight bank groups),
  // then stored as full 256-byte rows
  uint8_t* Y = base;
#pragma unroll
  for (int nt = 0; nt < kBN / 8; ++nt)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = 16 * warp + gq + 8 * r;
      const uint32_t v = ok ? pack_bf16x2(acc[nt][2 * r], acc[nt][2 * r + 1])
                            : pack_bf16x2(bad, bad);
      *reinterpret_cast<uint32_t*>(Y + row * 256 + ((nt ^ (row & 7)) << 4) + tq * 4) = v;
    }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kBM * 16 / kThreads; ++j) {
    const int idx = tid + kThreads * j;
    const int row = idx >> 4, c = idx & 15;
    const int m = m0 + row;
    if (m < p.M)
      *reinterpret_cast<uint4*>(p.y + (static_cast<int64_t>(m) * p.H + h) * p.ldy + n0 + 8 * c) =
          *reinterpret_cast<const uint4*>(Y + row * 256 + ((c ^ (row & 7)) << 4));
  }
  if (copy_pe) {
    if (pe_in_regs) {
#pragma unroll
      for (int j = 0; j < kPeRegs; ++j) {
        const int i = tid + kThreads * j;
        const int r = i / pe_units, u = i - (i / pe_units) * pe_units;
        if (i < kBM * pe_units && m0 + r < p.M)
          *reinterpret_cast<uint4*>(p.y + (static_cast<int64_t>(m0 + r) * p.H + h) * p.ldy + p.N +
                                    8 * u) = pe[j];
      }
    } else {
      for (int i = tid; i < kBM * pe_units; i += kThreads) {
        const int r = i / pe_units, u = i % pe_units;
        if (m0 + r >= p.M) continue;
        const int64_t row = static_cast<int64_t>(m0 + r) * p.H + h;
        *reinterpret_cast<uint4*>(p.y + row * p.ldy + p.N + 8 * u) =
            __ldg(reinterpret_cast<const uint4*>(p.extra + row * p.extra_dim) + u);
      }
    }
  }
}

// ------------------------------------------------------------ tcgen05 path --
// The two products of the benchmark shapes (d_h = d_v = 128, d_c = 512, up to
// 64 sequences) on the 5th-generation tensor cores, with the head's outputs
// on M and the sequences on N (N = 64, rows past M read as zero):
//   absorb:  D[c, b] = sum_i W_UK[c, h*128 + i] X[b, h, i]  A = the weight
//            rows (K-major: i is contiguous), B = q_nope rows; a CTA owns one
//            head and half of the 512 outputs (two M blocks of 128): 64 KB of
//            weights + 16 KB of q_nope, two CTAs per SM, 256 CTAs;
//   project: D[i, b] = sum_c W_UV[c, h*128 + i] X[b, h, c]  A = the weight
//            read MN-major (i is contiguous within a row c), B = o_lat rows;
//            a CTA owns one head: 128 KB of weights + 64 KB of o_lat, 128 CTAs.
// Every load of the CTA is issued up front by one thread (128-byte swizzled
// TMA boxes on a few mbarriers), one thread issues the products as their
// operands land, and the four warps read D from TMEM (lane = output, column
// = sequence), stage it as bf16 rows in shared memory and store whole rows.
namespace tcp {
constexpr int kB = 64;                 // sequences per CTA: N of the products
constexpr int kWBox = 128 * 128;       // a weight box: 128 rows x 64 elements (16 KB)
constexpr int kXBox = kB * 128;        // an activation box: 64 rows x 64 elements (8 KB)
// absorb: weight boxes [M block j][K half kh], then the two q_nope halves
constexpr int kAbsW = 4 * kWBox, kAbsX = 2 * kXBox;
constexpr int kAbsSmem = kAbsW + kAbsX + 1024 + 128;
// project: weight boxes [c quarter q][i half ih], then eight o_lat chunks
constexpr int kPrjW = 8 * kWBox, kPrjX = 8 * kXBox;
constexpr int kPrjSmem = kPrjW + kPrjX + 1024 + 128;
static_assert(kPrjSmem <= 227 * 1024, "shared memory");
constexpr int kThreads = 128;
constexpr uint32_t kIdescAbs = tc::instr_desc(128, kB, false);
constexpr uint32_t kIdescPrj = tc::instr_desc(128, kB, false, true);
}  // namespace tcp

struct TcProjParams {
  __nv_bfloat16* y;            // absorb: q_lat [M, H, ldy]; project: out [M, H, 128]
  const __nv_bfloat16* extra;  // absorb: q_pe [M, H, extra_dim], copied to columns 512..
  int32_t M, H, ldy, extra_dim;
};

// mx: the activations [M, H, K] as 3-D {K, H, M}, box {64, 1, 64};
// mw: the weights [d_c, H * 128] as 2-D, box {64, 128}.
template <bool kProject>
__global__ void __launch_bounds__(tcp::kThreads, 1)
    mla_head_gemm_tc_kernel(const __grid_constant__ CUtensorMap mx,
                            const __grid_constant__ CUtensorMap mw, const TcProjParams p) {
  using namespace tcp;
  using namespace tc;
  constexpr int kWBytes = kProject ? kPrjW : kAbsW;
  constexpr int kXBytes = kProject ? kPrjX : kAbsX;
  constexpr int kNBar = kProject ? 4 : 2;  // load groups: c quarters / K halves
  constexpr int kMBlocks = kProject ? 1 : 2;
  constexpr uint32_t kCols = kProject ? 64 : 128;  // TMEM columns: one N = 64 block per M block
  extern __shared__ uint8_t dyn_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* wsm = base;
  uint8_t* xsm = base + kWBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + kWBytes + kXBytes);  // [kNBar] loads, [kNBar] done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kNBar + 1);
  const int h = kProject ? blockIdx.x : blockIdx.x >> 1;
  const int v = kProject ? 0 : blockIdx.x & 1;  // absorb: outputs 256 v ..
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    prefetch_tensormap(&mx);
    prefetch_tensormap(&mw);
    for (int i = 0; i <= kNBar; ++i) mbar_init(&bar[i], 1);
    mbar_init_fence();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tslot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  uint64_t* done = &bar[kNBar];

  if (tid == 0) {
    // every load of the CTA at once
    const uint64_t pol_w = l2_policy_evict_first();   // weights: read once
    const uint64_t pol_x = l2_policy_evict_normal();  // activations: shared by the CTAs of a head
    if constexpr (kProject) {
      // group q: weight rows c 128 q .. (both i halves) and o_lat chunks 2q, 2q + 1
      for (int q = 0; q < 4; ++q) {
        mbar_arrive_expect_tx(&bar[q], 2 * kWBox + 2 * kXBox);
        for (int ih = 0; ih < 2; ++ih)
          tma_load_2d(wsm + (2 * q + ih) * kWBox, &mw, h * 128 + 64 * ih, 128 * q, &bar[q], pol_w);
        for (int k2 = 0; k2 < 2; ++k2)
          tma_load_3d(xsm + (2 * q + k2) * kXBox, &mx, 64 * (2 * q + k2), h, 0, &bar[q], pol_x);
      }
    } else {
      // group kh: the two weight blocks' K half kh and q_nope half kh
      for (int kh = 0; kh < 2; ++kh) {
        mbar_arrive_expect_tx(&bar[kh], 2 * kWBox + kXBox);
        for (int j = 0; j < 2; ++j)
          tma_load_2d(wsm + (2 * j + kh) * kWBox, &mw, h * 128 + 64 * kh, 256 * v + 128 * j,
                      &bar[kh], pol_w);
        tma_load_3d(xsm + kh * kXBox, &mx, 64 * kh, h, 0, &bar[kh], pol_x);
      }
    }
  }

  // absorb: the rope part of the query rides behind the latent part (the
  // first CTA of each head copies it); its rows are read now
  const bool copy_pe = !kProject && p.extra != nullptr && v == 0;
  const int pe_units = p.extra_dim / 8;
  uint4 pe[4];
  if (copy_pe) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + tcp::kThreads * j;
      const int r = pe_units > 0 ? i / pe_units : 0, u = i - r * pe_units;
      pe[j] = (pe_units > 0 && i < kB * pe_units && r < p.M)
                  ? __ldg(reinterpret_cast<const uint4*>(
                              p.extra + (static_cast<int64_t>(r) * p.H + h) * p.extra_dim) + u)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  }

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      const uint32_t w0 = smem_u32(wsm), x0 = smem_u32(xsm);
      for (int g = 0; g < kNBar && ok; ++g) {
        ok = mbar_wait_bounded(&bar[g], 0, nullptr);
        if (!ok) break;
        tc_fence_after();
        if constexpr (kProject) {
          // 128 rows c of group g: A = both i halves (leading offset 16 KB),
          // 16 rows c per k-step (2 KB); B = o_lat chunk 2g + c / 64
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_ss(tmem, smem_desc(w0 + (2 * g) * kWBox + kk * 2048, kWBox, 1024),
                      smem_desc(x0 + (2 * g + (kk >> 2)) * kXBox + 32 * (kk & 3), 16, 1024),
                      kIdescPrj, (g > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int j = 0; j < kMBlocks; ++j)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_ss(tmem + kB * j, smem_desc(w0 + (2 * j + g) * kWBox + 32 * kk, 16, 1024),
                        smem_desc(x0 + g * kXBox + 32 * kk, 16, 1024), kIdescAbs,
                        (g > 0 || kk > 0) ? 1u : 0u);
        }
      }
      tc_commit(done);  // also after a timeout: every product issued completes first
    }
    __syncwarp();
  }
  // the products are done (their operands are no longer read)
  ok = __syncthreads_and(ok && mbar_wait_bounded(done, 0, nullptr));
  if (!ok) {
    // a load never landed (never expected): wait once more, bounded, for the
    // copies still in flight into the shared memory staged below; the CTA's
    // outputs become NaN
    if (tid == 0)
      for (int g = 0; g < kNBar; ++g) mbar_wait_bounded(&bar[g], 0, nullptr);
    __syncthreads();
  }
  tc_fence_after();

  // D: lane = output (32 per warp and M block), 64 columns = sequences; staged
  // as bf16 rows Y[b][outputs of the CTA] in the weight region, then stored
  // as whole rows
  constexpr int kOut = 128 * kMBlocks;  // outputs per CTA
  uint8_t* Y = wsm;
  const float bad = __int_as_float(0x7fc00000);
#pragma unroll
  for (int j = 0; j < kMBlocks; ++j) {
    float d[kB];
    tc_ld32_nowait(tmem + (static_cast<uint32_t>(32 * warp) << 16) + kB * j, &d[0]);
    tc_ld32_nowait(tmem + (static_cast<uint32_t>(32 * warp) << 16) + kB * j + 32, &d[32]);
    tc_wait_ld();
    const int o = 128 * j + 32 * warp + lane;
#pragma unroll
    for (int b = 0; b < kB; ++b)
      *reinterpret_cast<__nv_bfloat16*>(Y + (b * kOut + o) * 2) =
          __float2bfloat16_rn(ok ? d[b] : bad);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
  constexpr int kRowUnits = kOut / 8;  // 16-byte units per staged row
  const int col0 = kProject ? 0 : 256 * v;
  for (int idx = tid; idx < kB * kRowUnits; idx += tcp::kThreads) {
    const int b = idx / kRowUnits, u = idx % kRowUnits;
    if (b < p.M)
      *reinterpret_cast<uint4*>(p.y + (static_cast<int64_t>(b) * p.H + h) * p.ldy + col0 + 8 * u) =
          *reinterpret_cast<const uint4*>(Y + (b * kOut + 8 * u) * 2);
  }
  if (copy_pe) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + tcp::kThreads * j;
      const int r = pe_units > 0 ? i / pe_units : 0, u = i - r * pe_units;
      if (pe_units > 0 && i < kB * pe_units && r < p.M)
        *reinterpret_cast<uint4*>(p.y + (static_cast<int64_t>(r) * p.H + h) * p.ldy + 512 +
                                  8 * u) = pe[j];
    }
  }
}

// 2-D map over w [rows, cols] bf16, boxes of 64 elements x box_rows rows,
// 128-byte swizzle.
bool make_weight_map(CUtensorMap* map, const void* w, int64_t rows, int64_t cols,
                     uint32_t box_rows = 64) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t es[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over x [M, H, K] bf16 as {K, H, M}, boxes of 64 elements x 1 head x
// 64 rows (rows past M read as zero), 128-byte swizzle.
bool make_rows_map(CUtensorMap* map, const void* x, int32_t M, int32_t H, int32_t K) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2,
                                 static_cast<cuuint64_t>(K) * 2 * static_cast<cuuint64_t>(H)};
  const cuuint32_t box[3] = {64u, 1u, 64u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The TMA path covers K = 128 (the absorb product at d_h = 128) and N a
// multiple of 128.
bool tma_path_fits(const ProjParams& p) { return p.K == kBK && p.N % kBN == 0; }


template <bool kTransB>
pa_status launch_gemm_tma(const ProjParams& q, cudaStream_t stream) {
  CUtensorMap mx, mw;
  const bool maps = make_rows_map(&mx, q.x, q.M, q.H, q.K) &&
                    (kTransB ? make_weight_map(&mw, q.w, q.K, static_cast<int64_t>(q.H) * q.N)
                             : make_weight_map(&mw, q.w, q.N, static_cast<int64_t>(q.H) * q.K));
  if (!maps) return PA_ERR_CUDA;
  TmaProjParams p;
  p.y = q.y;
  p.extra = q.extra;
  p.M = q.M;
  p.H = q.H;
  p.K = q.K;
  p.N = q.N;
  p.ldy = q.ldy;
  p.extra_dim = q.extra_dim;
  static std::atomic<uint64_t> smem_raised{0};
  auto kern = mla_head_gemm_tma_kernel<kTransB>;
  if (!ensure_smem_limit(kern, kTmaSmem, smem_raised)) return PA_ERR_CUDA;
  const dim3 grid(1u, static_cast<unsigned>(q.H * (q.N / kBN)),
                  static_cast<unsigned>((q.M + kBM - 1) / kBM));
  kern<<<grid, kThreads, kTmaSmem, stream>>>(mx, mw, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// The tcgen05 path: absorb with d_h = 128, d_c = 512, a rope part of at most
// 64 elements; project with d_c = 512, d_v = 128; up to 64 sequences.
bool tc_path_fits(const ProjParams& p, bool project) {
  return p.M <= tcp::kB &&
         (project ? (p.K == 512 && p.N == 128)
                  : (p.K == 128 && p.N == 512 && p.extra_dim <= 64 && p.extra_dim % 8 == 0));
}

template <bool kProject>
pa_status launch_gemm_tc(const ProjParams& q, cudaStream_t stream) {
  CUtensorMap mx, mw;
  // weights [d_c, H * 128] in both products (rows = outputs for absorb, the
  // reduction index for project), boxes of 128 rows
  const int64_t wrows = kProject ? q.K : q.N;
  const int64_t wcols = static_cast<int64_t>(q.H) * (kProject ? q.N : q.K);
  if (!make_rows_map(&mx, q.x, q.M, q.H, q.K) || !make_weight_map(&mw, q.w, wrows, wcols, 128))
    return PA_ERR_CUDA;
  TcProjParams p;
  p.y = q.y;
  p.extra = q.extra;
  p.M = q.M;
  p.H = q.H;
  p.ldy = q.ldy;
  p.extra_dim = q.extra_dim;
  static std::atomic<uint64_t> smem_raised{0};
  auto kern = mla_head_gemm_tc_kernel<kProject>;
  constexpr int kSmemTc = kProject ? tcp::kPrjSmem : tcp::kAbsSmem;
  if (!ensure_smem_limit(kern, kSmemTc, smem_raised)) return PA_ERR_CUDA;
  const dim3 grid(static_cast<unsigned>(kProject ? q.H : 2 * q.H), 1u, 1u);
  kern<<<grid, tcp::kThreads, kSmemTc, stream>>>(mx, mw, p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <bool kTransB>
pa_status launch_gemm(ProjParams p, cudaStream_t stream) {
  if (tc_path_fits(p, kTransB)) return launch_gemm_tc<kTransB>(p, stream);
  if (tma_path_fits(p)) return launch_gemm_tma<kTransB>(p, stream);
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
