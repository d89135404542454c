// pa_internal.cuh -- shared device helpers of the sm_103a paged-KV library.
//
// Element vectors (8 elements per 16-byte-class access), round-to-nearest
// casts through CUDA's conversion intrinsics, and the mbarrier / TMA
// primitives of the decode pipeline (inline PTX).  Every wait on an mbarrier
// is bounded by %globaltimer so that a lost transfer turns into an error
// word on the host side instead of a hung GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------- dtypes --
using bf16 = __nv_bfloat16;
using f16 = __half;
struct e4m3 {  // storage-only tag type for fp8 E4M3
  uint8_t bits;
};

template <typename T>
struct Vec8;  // eight elements, raw
template <>
struct Vec8<bf16> { uint4 u; };
template <>
struct Vec8<f16> { uint4 u; };
template <>
struct Vec8<float> { uint4 u[2]; };
template <>
struct Vec8<e4m3> { uint2 u; };

// read-only, streamed loads (the source rows are read exactly once)
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <typename T>
__device__ __forceinline__ Vec8<T> load8(const T* p);
template <>
__device__ __forceinline__ Vec8<bf16> load8(const bf16* p) { return {ld_stream16(p)}; }
template <>
__device__ __forceinline__ Vec8<f16> load8(const f16* p) { return {ld_stream16(p)}; }
template <>
__device__ __forceinline__ Vec8<float> load8(const float* p) {
  Vec8<float> v;
  v.u[0] = ld_stream16(p);
  v.u[1] = ld_stream16(p + 4);
  return v;
}

template <typename T>
__device__ __forceinline__ void store8(T* p, const Vec8<T>& v);
template <>
__device__ __forceinline__ void store8(bf16* p, const Vec8<bf16>& v) {
  *reinterpret_cast<uint4*>(p) = v.u;
}
template <>
__device__ __forceinline__ void store8(f16* p, const Vec8<f16>& v) {
  *reinterpret_cast<uint4*>(p) = v.u;
}
template <>
__device__ __forceinline__ void store8(float* p, const Vec8<float>& v) {
  reinterpret_cast<uint4*>(p)[0] = v.u[0];
  reinterpret_cast<uint4*>(p)[1] = v.u[1];
}
template <>
__device__ __forceinline__ void store8(e4m3* p, const Vec8<e4m3>& v) {
  *reinterpret_cast<uint2*>(p) = v.u;
}

// widen eight elements to fp32 (exact for every source type)
__device__ __forceinline__ void to_f32(const Vec8<bf16>& v, float f[8]) {
  const uint32_t w[4] = {v.u.x, v.u.y, v.u.z, v.u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void to_f32(const Vec8<f16>& v, float f[8]) {
  const uint32_t w[4] = {v.u.x, v.u.y, v.u.z, v.u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 t = __half22float2(h);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void to_f32(const Vec8<float>& v, float f[8]) {
  const uint32_t w[8] = {v.u[0].x, v.u[0].y, v.u[0].z, v.u[0].w,
                         v.u[1].x, v.u[1].y, v.u[1].z, v.u[1].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(w[i]);
}
// the same, negated (-x: the sign bit flipped in the source format, exact)
__device__ __forceinline__ void to_f32_neg(const Vec8<bf16>& v, float f[8]) {
  const uint32_t w[4] = {v.u.x, v.u.y, v.u.z, v.u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float((w[i] << 16) ^ 0x80000000u);
    f[2 * i + 1] = __uint_as_float((w[i] & 0xFFFF0000u) ^ 0x80000000u);
  }
}
__device__ __forceinline__ void to_f32_neg(const Vec8<f16>& v, float f[8]) {
  Vec8<f16> n;
  n.u = make_uint4(v.u.x ^ 0x80008000u, v.u.y ^ 0x80008000u, v.u.z ^ 0x80008000u,
                   v.u.w ^ 0x80008000u);
  to_f32(n, f);
}
__device__ __forceinline__ void to_f32_neg(const Vec8<float>& v, float f[8]) {
  const uint32_t w[8] = {v.u[0].x, v.u[0].y, v.u[0].z, v.u[0].w,
                         v.u[1].x, v.u[1].y, v.u[1].z, v.u[1].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(w[i] ^ 0x80000000u);
}

// narrow eight fp32 values, round to nearest even (E4M3: saturating)
template <typename T>
__device__ __forceinline__ Vec8<T> from_f32(const float f[8]);
template <>
__device__ __forceinline__ Vec8<bf16> from_f32(const float f[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i]));
    uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i + 1]));
    w[i] = lo | (hi << 16);
  }
  return {make_uint4(w[0], w[1], w[2], w[3])};
}
template <>
__device__ __forceinline__ Vec8<f16> from_f32(const float f[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo = __half_as_ushort(__float2half_rn(f[2 * i]));
    uint32_t hi = __half_as_ushort(__float2half_rn(f[2 * i + 1]));
    w[i] = lo | (hi << 16);
  }
  return {make_uint4(w[0], w[1], w[2], w[3])};
}
template <>
__device__ __forceinline__ Vec8<float> from_f32(const float f[8]) {
  Vec8<float> v;
  v.u[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  v.u[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                      __float_as_uint(f[7]));
  return v;
}
template <>
__device__ __forceinline__ Vec8<e4m3> from_f32(const float f[8]) {
  // four codes per register: two paired conversions (the first value of a
  // pair in the low byte) joined as the register's 16-bit halves
  uint32_t w[2];
#pragma unroll
  for (int i = 0; i < 2; ++i)
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(w[i])
        : "f"(f[4 * i]), "f"(f[4 * i + 1]), "f"(f[4 * i + 2]), "f"(f[4 * i + 3]));
  return {make_uint2(w[0], w[1])};
}

// ------------------------------------------------------------- division --
// x / s rounded to nearest (IEEE), for one divisor s shared by many x.
// r = RN(1/s) is computed once; then two residual corrections
//     q0 = RN(x r),  q1 = RN(q0 + RN(x - s q0) r),  q2 = RN(q1 + RN(x - s q1) r)
// where each residual x - s q is exact with an FMA.  q1 is within one ulp of
// x/s, and Markstein's theorem (division with a fused multiply-add: r within
// half an ulp of 1/s and q within one ulp of x/s give RN(q + (x - s q) r) =
// RN(x/s)) makes q2 the correctly rounded quotient, provided nothing under-
// or overflows.  Outside the ranges that guarantee that (and for zeros,
// infinities and NaN) the library's IEEE division is used.
struct Divisor {
  float s, r;
  bool fast;
};
__device__ __forceinline__ Divisor make_divisor(float s) {
  Divisor d;
  d.s = s;
  d.r = __frcp_rn(s);
  const float as = fabsf(s);
  d.fast = s > 0.f && as >= 0x1p-30f && as <= 0x1p30f;  // false for NaN
  return d;
}
// Chunk of eight quotients by the library division (kept out of line: the
// rare path of div8_for_e4m3).
struct F8 {
  float v[8];
};
static __device__ __noinline__ F8 div8_library(F8 x, float s) {
#pragma unroll
  for (int e = 0; e < 8; ++e) x.v[e] = __fdiv_rn(x.v[e], s);
  return x;
}

// The same operations on pairs (one instruction for two lanes of work on
// sm_100 and later; each lane rounds exactly as the scalar operation does).
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
  return d;
}

// Eight quotients x / s (x: the eight source elements of v) that only feed
// a round-to-nearest cast to E4M3.  Such a cast depends on the fp32 quotient
// only where |x / s| lies in [2^-11, 480]: smaller values become +-0, larger
// ones saturate.  With the divisor in [2^-30, 2^30] (d.fast), every quotient
// in that band has |x| >= 2^-41, where the two residual corrections of
// div_rn are exact, so no per-value range test is needed -- only that x * r
// cannot overflow (the chunk's largest |x| at most xmax; NaN passes through
// as NaN).  Other chunks use the library.
// The corrections run on n = -x, which the widening gives at no extra cost:
//     y0 = RN(n (-r)),  y' = RN(y + RN(s y + n) (-r)).
// Round-to-nearest is symmetric in sign, so RN(s y + n) = -RN(x - s y) and
// every step equals the one of div_rn for a nonzero quotient; for a zero one
// the signed-zero sums give the sign of x (x = -0: RN(-0 + +0) = +0, then
// RN(+0 (-r) + -0) = -0), with no separate sign fix-up.
template <typename S>
__device__ __forceinline__ void div8_for_e4m3(const Vec8<S>& v, float (&f)[8], const Divisor& d,
                                              float xmax) {
  float n[8];
  to_f32_neg(v, n);
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; e += 2) amax = max3_abs(amax, n[e], n[e + 1]);
  if (d.fast && amax <= xmax) {
    const float2 nr2 = make_float2(-d.r, -d.r), s2 = make_float2(d.s, d.s);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 ne = make_float2(n[e], n[e + 1]);
      float2 y = mul2_rn(ne, nr2);
      y = fma2_rn(fma2_rn(s2, y, ne), nr2, y);
      y = fma2_rn(fma2_rn(s2, y, ne), nr2, y);
      f[e] = y.x;
      f[e + 1] = y.y;
    }
  } else {
    F8 t;
#pragma unroll
    for (int e = 0; e < 8; ++e) t.v[e] = -n[e];
    t = div8_library(t, d.s);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = t.v[e];
  }
}

__device__ __forceinline__ float div_rn(float x, const Divisor& d) {
  const float ax = fabsf(x);
  if (d.fast && ax >= 0x1p-60f && ax <= 0x1p60f) {
    float q = __fmul_rn(x, d.r);
    q = __fmaf_rn(__fmaf_rn(-d.s, q, x), d.r, q);
    return __fmaf_rn(__fmaf_rn(-d.s, q, x), d.r, q);
  }
  return __fdiv_rn(x, d.s);
}

// ------------------------------------------------------- mbarrier / TMA --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// make barrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with `parity` to complete.  Gives up (returns false)
// after `timeout_ns` of wall time, or early once *abort_flag is set by
// another warp of the CTA.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
    }
  }
}

// As mbar_wait_bounded, for waits that are usually long (a whole pipeline
// step): each try_wait may keep the thread suspended for up to `hint_ns`
// (it resumes as soon as the phase completes), so a waiting warp re-polls
// rarely and leaves the issue slots of its SM sub-partition to the warps
// that compute.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded_long(uint64_t* bar, uint32_t parity,
                                                       volatile int* abort_flag) {
  constexpr uint32_t kHintNs = 20000;
  if (mbar_try_wait_hint(bar, parity, kHintNs)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, kHintNs)) return true;
    if (abort_flag && *abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
// L2 hint: the K/V stream is read once, evict it first.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, uint64_t* bar,
                                            uint64_t l2_policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(l2_policy)
      : "memory");
}

// 2-D tiled TMA load global -> shared with an L2 hint, completion on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, uint64_t* bar, uint64_t l2_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(l2_policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Barrier `id` over `nthreads` threads (a multiple of 32) that also returns
// whether `pred` held in every participating thread.
__device__ __forceinline__ bool named_barrier_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------ tensor-core fragments (mma.sync) --
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two floats rounded to nearest-even f16, lo in bits 0-15 (one instruction).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// four e4m3 codes (low byte first) -> two f16x2 (codes 0,1 and 2,3), exact;
// the register's 16-bit halves feed the conversions directly (no shifts or
// masks)
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_codes, uint32_t& lo,
                                                  uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four_codes));
}
// Two floats rounded to nearest-even bf16, lo in bits 0-15: one conversion
// instruction for the pair (two scalar conversions plus a merge cost several
// times more issue time in the softmax loops).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Global data written by ordinary stores (this or other CTAs, already
// acquired) made visible to the copy engine before a bulk copy reads it.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Untiled bulk copy global -> this CTA's shared memory, completion counted
// in bytes on `bar`; both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace pa

// ------------------------------------------------- internal host launchers --
namespace pa_detail {

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute is per device, and `raised` (one per
// call site) holds a bit for each device already done.
template <typename Kernel>
inline bool ensure_smem_limit(Kernel kernel, int bytes, std::atomic<uint64_t>& raised) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0ull && (raised.load() & bit) != 0ull) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  raised.fetch_or(bit);
  return true;
}


int num_sms_current_device();  // cached per device; 0 if no device

// TMA maps over a [rows, H_KV, 128] cache (rows = num_blocks * block_size):
// bf16 in 64-element half-row boxes, e4m3 in whole 128-byte rows; box_rows
// rows of one kv head per copy, 128-byte swizzled in shared memory.
bool make_kv_map_swizzled(CUtensorMap* map, const void* base, int64_t rows, int32_t num_kv_heads,
                          int32_t box_rows);
bool make_kv_map_fp8(CUtensorMap* map, const void* base, int64_t rows, int32_t num_kv_heads,
                     int32_t box_rows);

struct ReshapeArgs {
  const void* key;
  const void* value;
  void* key_cache;
  void* value_cache;
  const int64_t* slot_mapping;
  const int64_t* swa;
  const float* k_scale;
  const float* v_scale;
  int64_t swa_len;
  int64_t num_tokens;
  int64_t key_stride;
  int64_t value_stride;
  int64_t block_stride;
  int64_t num_slots;
  int32_t row_chunks;  // (num_heads * head_size) / 8
  int32_t block_size;
  int32_t groups;      // chunk groups (warps) per token
  // two-source rows (pa_concat_and_cache_mla): chunks >= key_chunks of a
  // row come from key2 (null: every chunk from key)
  const void* key2;
  int64_t key2_stride;
  int32_t key_chunks;
};
pa_status launch_reshape_and_cache(const ReshapeArgs& a, pa_dtype src, pa_dtype dst,
                                   cudaStream_t stream);

struct ConcatArgs {
  void* k;
  const void* k_nope;
  const void* k_rope;
  int64_t num_tokens;
  int64_t k_stride0, k_stride1, nope_stride0, nope_stride1, rope_stride0;
  int32_t num_heads;
  int32_t nope_chunks;  // nope_dim / 8
  int32_t rope_chunks;  // rope_dim / 8
};
pa_status launch_concat_mla_k(const ConcatArgs& a, pa_dtype src, pa_dtype dst,
                              cudaStream_t stream);

struct DecodePlan {
  int32_t num_splits;
  int32_t tokens_per_split;
};
DecodePlan make_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len,
                            int32_t num_sms);
size_t decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_size, const DecodePlan& plan);

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* workspace;
  unsigned* error_word;  // nullptr: the workspace's own error word
  int32_t num_seqs, num_q_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq;
  int64_t num_blocks;
  float scale;
  DecodePlan plan;
  pa_dtype cache_dtype;    // PA_BF16 or PA_FP8_E4M3
  const float* k_scale;    // e4m3 cache: device scalars (null = 1)
  const float* v_scale;
  const void* new_k;       // fused decode step: [B, H_KV, d] bf16 (else null)
  const void* new_v;
  const int64_t* slot_mapping;
};
pa_status launch_paged_decode(const DecodeArgs& a, cudaStream_t stream);

struct PrefillArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  unsigned* error_word;
  int32_t num_seqs, num_q_heads, num_kv_heads, block_size, max_blocks_per_seq, max_q_len;
  int64_t num_blocks;
  float scale;
};
pa_status launch_paged_prefill(const PrefillArgs& a, cudaStream_t stream);  // prefill_tc.cu

struct MlaDecodeArgs {
  void* out_latent;          // [B, H, 512] bf16
  const void* q_latent;      // [B, H, 576] bf16
  const void* latent_cache;  // [num_blocks, block_size, 576] bf16
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* workspace;
  int32_t num_seqs, num_heads, block_size, max_blocks_per_seq;
  int64_t num_blocks;
  float scale;
  DecodePlan plan;
};
int mla_head_tile(int32_t num_heads);  // 64 when num_heads % 64 == 0, else 16
DecodePlan make_mla_plan(int32_t num_seqs, int32_t num_heads, int32_t max_context_len,
                         int32_t num_sms);
size_t mla_workspace_bytes(int32_t num_seqs, int32_t num_heads, const DecodePlan& plan);
pa_status launch_mla_decode(const MlaDecodeArgs& a, cudaStream_t stream);
pa_status launch_mla_absorb_q(void* q_latent, const void* q_nope, const void* q_pe,
                              const void* w_uk, int32_t num_seqs, int32_t num_heads,
                              int32_t nope_dim, int32_t rope_dim, int32_t latent_dim,
                              cudaStream_t stream);
pa_status launch_mla_project_out(void* out, const void* out_latent, const void* w_uv,
                                 int32_t num_seqs, int32_t num_heads, int32_t latent_dim,
                                 int32_t v_head_dim, cudaStream_t stream);

// Library-owned decode scratch (a file-scope __device__ array in decode.cu)
// for callers that cannot allocate: its size, and its device address on the
// current device (looked up once per device).
size_t static_decode_scratch_bytes();
pa_status static_decode_scratch_address(void** ptr);

}  // namespace pa_detail
