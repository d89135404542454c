/*
 * oracle.c -- plain, slow, CPU reference for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against.  It is called from the test suite, from the package's
 * smoke check and from the benchmark's CPU-baseline leg, and from nowhere
 * else.  It includes no CUDA header and shares no code, table or constant
 * with the CUDA library; the two agree only because both follow the pages
 * cited below.
 *
 * Everything is nested loops in the order the definitions state them:
 *   - number formats (bf16, fp16, fp8 e4m3) are built from their bit-field
 *     definitions; encoding is "nearest representable value, ties to the
 *     even code", found by search in a table of every finite value;
 *   - the cache write follows sglang cache_ops.py, reshape_and_cache_flash
 *     (its "slot mapping", "optional scale" and "target layout" blocks) and
 *     the nano-vLLM walkthrough, section 2.6 Attention (store_kvcache_kernel);
 *   - the MLA K assembly follows sglang cache_ops.py,
 *     concat_and_cast_mha_k_kernel and its wrapper's shape checks;
 *   - decode attention is dense softmax attention of one query row over the
 *     context gathered, in logical order, through the block table
 *     (PagedAttention-principle post, section "paged attention原理": blocks
 *     may be scattered, a table keeps their order; walkthrough section 2.6:
 *     decode reads the cache back along block_tables).  Arithmetic in double;
 *   - MLA decode keeps one latent row per token (PagedAttention-principle
 *     post, MLA section: c_kv = x W_DKV is what is cached; K and V of a head
 *     are c_kv W_UK and c_kv W_UV; the rope part of K rides beside it).  It
 *     is written here twice, head by head, with plain loops: in the pages'
 *     own form (or_mla_decode_explicit: K and V rebuilt from the latent,
 *     then plain attention) and in the absorbed form the three library calls
 *     take (or_mla_absorb_q, or_mla_decode_row, or_mla_project_out).
 *
 * Error returns are negative integers (see the OR_E* codes); nothing here
 * aborts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- dtype codes of this oracle (its own numbering) --------------------- */
#define OR_BF16 0
#define OR_FP16 1
#define OR_FP32 2
#define OR_E4M3 3
#define OR_FP64 4 /* read-only: inputs already in double (MLA functions) */

#define OR_OK 0
#define OR_EINVAL (-1)      /* bad argument                                  */
#define OR_EDUPSLOT (-2)    /* two tokens resolve to the same cache slot     */
#define OR_ENOMEM (-3)

/* ======================================================================== */
/* Number formats from their definitions                                    */
/* ======================================================================== */

/* A binary floating-point format with e exponent bits, m stored mantissa
 * bits and exponent bias `bias`.  Code layout: sign | exponent | mantissa.
 * has_inf: IEEE style (exponent all ones = inf/NaN).  Without it (OCP FP8
 * E4M3), only the all-ones exponent with all-ones mantissa is NaN and the
 * other all-ones-exponent codes are finite normals. */
typedef struct {
  int e, m, bias, has_inf;
  uint32_t max_finite_code; /* largest non-negative finite code */
  uint32_t inf_code;        /* has_inf only                      */
  uint32_t nan_code;        /* quiet NaN, sign bit clear         */
  double *val;              /* val[c] for c = 0..max_finite_code */
} or_fmt;

static or_fmt F_BF16 = {8, 7, 127, 1, 0x7F7Fu, 0x7F80u, 0x7FC0u, NULL};
static or_fmt F_FP16 = {5, 10, 15, 1, 0x7BFFu, 0x7C00u, 0x7E00u, NULL};
static or_fmt F_E4M3 = {4, 3, 7, 0, 0x7Eu, 0u, 0x7Fu, NULL};

/* Value of a non-negative code with a finite meaning. */
static double fmt_code_value(const or_fmt *f, uint32_t c) {
  uint32_t mant = c & ((1u << f->m) - 1u);
  uint32_t ex = c >> f->m;
  if (ex == 0) /* subnormal: 0.mant * 2^(1-bias) */
    return ldexp((double)mant, 1 - f->bias - f->m);
  /* normal: 1.mant * 2^(ex-bias) */
  return ldexp((double)((1u << f->m) + mant), (int)ex - f->bias - f->m);
}

static int fmt_ready(or_fmt *f) {
  if (f->val) return 1;
  double *v = (double *)malloc(sizeof(double) * (f->max_finite_code + 1u));
  if (!v) return 0;
  for (uint32_t c = 0; c <= f->max_finite_code; ++c) v[c] = fmt_code_value(f, c);
  f->val = v;
  return 1;
}

static or_fmt *fmt_of(int dtype) {
  switch (dtype) {
    case OR_BF16: return &F_BF16;
    case OR_FP16: return &F_FP16;
    case OR_E4M3: return &F_E4M3;
    default: return NULL;
  }
}

/* Decode a code of format f to double (NaN and inf included). */
static double fmt_decode(or_fmt *f, uint32_t code) {
  uint32_t nbits = 1u + (uint32_t)f->e + (uint32_t)f->m;
  uint32_t sign = (code >> (nbits - 1u)) & 1u;
  uint32_t mag = code & ((1u << (nbits - 1u)) - 1u);
  double r;
  uint32_t exp_all_ones = ((1u << f->e) - 1u);
  if (f->has_inf && (mag >> f->m) == exp_all_ones) {
    r = (mag & ((1u << f->m) - 1u)) ? NAN : INFINITY;
  } else if (!f->has_inf && mag > f->max_finite_code) {
    r = NAN;
  } else {
    r = fmt_code_value(f, mag);
  }
  return sign ? -r : r;
}

/* Encode y: nearest representable value, ties to the even code.  Formats
 * with infinities round past the top like IEEE 754 (a value at or beyond
 * the midpoint between the largest finite value and 2^(emax+1) becomes
 * inf); E4M3 saturates to its largest finite value (+-448), inf included.
 * NaN becomes the quiet NaN code. */
static uint32_t fmt_encode(or_fmt *f, double y) {
  uint32_t nbits = 1u + (uint32_t)f->e + (uint32_t)f->m;
  uint32_t sign_bit = 1u << (nbits - 1u);
  if (isnan(y)) return f->nan_code;
  uint32_t sign = signbit(y) ? sign_bit : 0u;
  double a = fabs(y);
  const double *v = f->val;
  uint32_t top = f->max_finite_code;
  uint32_t code;
  if (a >= v[top]) {
    if (!f->has_inf) {
      code = top; /* saturate */
    } else {
      /* the next step above the largest finite value is 2^(emax+1); its
       * code is the inf code, whose mantissa is zero (even) */
      double next = 2.0 * ldexp(1.0, (int)((1u << f->e) - 2u) - f->bias);
      double mid = 0.5 * (v[top] + next);
      if (a < mid) code = top;
      else if (a > mid) code = f->inf_code;
      else code = (top & 1u) ? f->inf_code : top;
    }
  } else {
    /* binary search: v[lo] <= a < v[lo+1] */
    uint32_t lo = 0, hi = top;
    while (hi - lo > 1u) {
      uint32_t mid_c = lo + (hi - lo) / 2u;
      if (v[mid_c] <= a) lo = mid_c; else hi = mid_c;
    }
    double mid = 0.5 * (v[lo] + v[lo + 1u]);
    if (a < mid) code = lo;
    else if (a > mid) code = lo + 1u;
    else code = (lo & 1u) ? lo + 1u : lo;
  }
  return sign | code;
}

static int dtype_size(int dtype) {
  switch (dtype) {
    case OR_BF16: case OR_FP16: return 2;
    case OR_FP32: return 4;
    case OR_E4M3: return 1;
    default: return 0;
  }
}

/* element i of an array of `dtype` as a double */
static double load_elem(int dtype, const void *base, int64_t i) {
  if (dtype == OR_FP64) return ((const double *)base)[i];
  if (dtype == OR_FP32) return (double)((const float *)base)[i];
  if (dtype == OR_E4M3) return fmt_decode(&F_E4M3, ((const uint8_t *)base)[i]);
  return fmt_decode(fmt_of(dtype), ((const uint16_t *)base)[i]);
}

/* store float y into element i of an array of `dtype` */
static void store_elem(int dtype, void *base, int64_t i, float y) {
  if (dtype == OR_FP32) { ((float *)base)[i] = y; return; }
  if (dtype == OR_E4M3) { ((uint8_t *)base)[i] = (uint8_t)fmt_encode(&F_E4M3, (double)y); return; }
  ((uint16_t *)base)[i] = (uint16_t)fmt_encode(fmt_of(dtype), (double)y);
}

/* copy element i of `src` to element j of `dst`, both of `dtype`, bit for bit
 * (a cast to the same format changes nothing; NaN payloads included) */
static void copy_elem(int dtype, void *dst, int64_t j, const void *src, int64_t i) {
  int sz = dtype_size(dtype);
  memcpy((uint8_t *)dst + j * sz, (const uint8_t *)src + i * sz, (size_t)sz);
}

static int formats_ready(void) {
  return fmt_ready(&F_BF16) && fmt_ready(&F_FP16) && fmt_ready(&F_E4M3);
}

/* ---- exported codec entry points (used by the tests' pins) ------------- */
int or_encode_array(int dtype, const float *y, int64_t n, void *out) {
  if (!formats_ready() || dtype_size(dtype) == 0) return OR_EINVAL;
  for (int64_t i = 0; i < n; ++i) store_elem(dtype, out, i, y[i]);
  return OR_OK;
}

int or_decode_array(int dtype, const void *codes, int64_t n, double *out) {
  if (!formats_ready() || dtype_size(dtype) == 0) return OR_EINVAL;
  for (int64_t i = 0; i < n; ++i) out[i] = load_elem(dtype, codes, i);
  return OR_OK;
}

/* number of non-negative finite values of a format, and the largest one */
int or_format_info(int dtype, int64_t *n_nonneg_finite, double *max_finite) {
  or_fmt *f = fmt_of(dtype);
  if (!f || !formats_ready()) return OR_EINVAL;
  *n_nonneg_finite = (int64_t)f->max_finite_code + 1;
  *max_finite = f->val[f->max_finite_code];
  return OR_OK;
}

/* ======================================================================== */
/* Cache write                                                              */
/* sglang cache_ops.py, reshape_and_cache_flash + launch wrapper; nano-vLLM */
/* walkthrough section 2.6 (store_kvcache_kernel, -1 slots skipped).        */
/* ======================================================================== */

/* Resolve token t's slot: the mapping, then the optional SWA second-stage
 * table; any negative value, an SWA index outside the table, or a slot past
 * the pool means "skip" (returns -1). */
static int64_t resolve_slot(const int64_t *slot_mapping, const int64_t *swa,
                            int64_t swa_len, int64_t num_slots, int64_t t) {
  int64_t s = slot_mapping[t];
  if (s < 0) return -1;
  if (swa) {
    if (s >= swa_len) return -1;
    s = swa[s];
    if (s < 0) return -1;
  }
  if (s >= num_slots) return -1;
  return s;
}

/* Returns the number of tokens written (>= 0) or an OR_E* code.
 * key/value: [num_tokens, num_heads, head_size] with key_stride/value_stride
 * elements between tokens.  value may be NULL (K-only cache; then
 * value_cache must be NULL too).  Caches: [num_blocks, block_size,
 * num_heads, head_size] with block_stride elements between blocks.
 * k_scale/v_scale: both NULL or both set (host scalars here). */
int64_t or_reshape_and_cache(const void *key, const void *value, int src_dtype,
                             int64_t num_tokens, int32_t num_heads, int32_t head_size,
                             int64_t key_stride, int64_t value_stride,
                             void *key_cache, void *value_cache, int cache_dtype,
                             int64_t num_blocks, int32_t block_size, int64_t block_stride,
                             const int64_t *slot_mapping, const int64_t *swa_slot_mapping,
                             int64_t swa_len, const float *k_scale, const float *v_scale) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!key || !key_cache || !slot_mapping) return OR_EINVAL;
  if ((value == NULL) != (value_cache == NULL)) return OR_EINVAL;
  if ((k_scale == NULL) != (v_scale == NULL)) return OR_EINVAL;
  if (num_tokens < 0 || num_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
    return OR_EINVAL;
  if (dtype_size(src_dtype) == 0 || src_dtype == OR_E4M3 || dtype_size(cache_dtype) == 0)
    return OR_EINVAL;
  const int64_t num_slots = num_blocks * (int64_t)block_size;
  const int64_t row = (int64_t)num_heads * head_size; /* elements of one token */

  /* the pages leave duplicate targets undefined; the oracle refuses them */
  uint8_t *seen = (uint8_t *)calloc((size_t)(num_slots > 0 ? num_slots : 1), 1);
  if (!seen) return OR_ENOMEM;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t s = resolve_slot(slot_mapping, swa_slot_mapping, swa_len, num_slots, t);
    if (s < 0) continue;
    if (seen[s]) { free(seen); return OR_EDUPSLOT; }
    seen[s] = 1;
  }
  free(seen);

  const int raw = (src_dtype == cache_dtype) && k_scale == NULL;
  int64_t written = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t s = resolve_slot(slot_mapping, swa_slot_mapping, swa_len, num_slots, t);
    if (s < 0) continue;
    int64_t block_idx = s / block_size;
    int64_t block_offset = s % block_size;
    for (int32_t h = 0; h < num_heads; ++h) {
      for (int32_t i = 0; i < head_size; ++i) {
        /* source: token t, head h, element i */
        int64_t kin = t * key_stride + (int64_t)h * head_size + i;
        /* target: [block_idx, block_offset, h, i] */
        int64_t dst = block_idx * block_stride + block_offset * row + (int64_t)h * head_size + i;
        int64_t vin = t * value_stride + (int64_t)h * head_size + i;
        if (raw) { /* same format, no scale: a plain copy */
          copy_elem(src_dtype, key_cache, dst, key, kin);
          if (value) copy_elem(src_dtype, value_cache, dst, value, vin);
          continue;
        }
        float kx = (float)load_elem(src_dtype, key, kin);
        if (k_scale) kx = kx / *k_scale; /* IEEE single-precision division */
        store_elem(cache_dtype, key_cache, dst, kx);
        if (value) {
          float vx = (float)load_elem(src_dtype, value, vin);
          if (v_scale) vx = vx / *v_scale;
          store_elem(cache_dtype, value_cache, dst, vx);
        }
      }
    }
    ++written;
  }
  return written;
}

/* ======================================================================== */
/* MLA K assembly                                                           */
/* sglang cache_ops.py, concat_and_cast_mha_k_kernel and                    */
/* concat_and_cast_mha_k_triton (shape checks; implicit cast to k's dtype). */
/* ======================================================================== */
/* k[n, h, 0:nope] = k_nope[n, h, :];  k[n, h, nope:nope+rope] = k_rope[n, 0, :]
 * Strides in elements; the last dimension of every tensor is contiguous. */
int or_concat_mla_k(void *k, int k_dtype, const void *k_nope, const void *k_rope, int src_dtype,
                    int64_t num_tokens, int32_t num_heads, int32_t nope_dim, int32_t rope_dim,
                    int64_t k_stride0, int64_t k_stride1, int64_t nope_stride0,
                    int64_t nope_stride1, int64_t rope_stride0) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!k || !k_nope || !k_rope) return OR_EINVAL;
  if (num_tokens < 0 || num_heads <= 0 || nope_dim <= 0 || rope_dim <= 0) return OR_EINVAL;
  if (dtype_size(k_dtype) == 0 || dtype_size(src_dtype) == 0 || src_dtype == OR_E4M3)
    return OR_EINVAL;
  const int raw = (k_dtype == src_dtype);
  for (int64_t n = 0; n < num_tokens; ++n) {
    for (int32_t h = 0; h < num_heads; ++h) {
      for (int32_t i = 0; i < nope_dim; ++i) {
        int64_t from = n * nope_stride0 + (int64_t)h * nope_stride1 + i;
        int64_t to = n * k_stride0 + (int64_t)h * k_stride1 + i;
        if (raw) copy_elem(k_dtype, k, to, k_nope, from);
        else store_elem(k_dtype, k, to, (float)load_elem(src_dtype, k_nope, from));
      }
      for (int32_t i = 0; i < rope_dim; ++i) {
        int64_t from = n * rope_stride0 + i;
        int64_t to = n * k_stride0 + (int64_t)h * k_stride1 + nope_dim + i;
        if (raw) copy_elem(k_dtype, k, to, k_rope, from);
        else store_elem(k_dtype, k, to, (float)load_elem(src_dtype, k_rope, from));
      }
    }
  }
  return OR_OK;
}

/* ======================================================================== */
/* Decode attention                                                         */
/* ======================================================================== */

/* Dense attention of one query q[0:d] over L contiguous rows K[j], V[j]
 * (row j at K + j*k_row_stride elements):
 *   s_j = scale * sum_i q_i K_ji
 *   p_j = exp(s_j - max s) / sum_j' exp(s_j' - max s)
 *   out_i = sum_j p_j V_ji,   lse = max s + log sum_j exp(s_j - max s)
 * psum (optional) receives sum_j p_j.  L == 0 gives out = 0, lse = -inf. */
int or_dense_attention_row(double *out, double *lse, double *psum, const double *q,
                           const double *K, int64_t k_row_stride, const double *V,
                           int64_t v_row_stride, int64_t L, int32_t d, double scale) {
  if (!out || !q || d <= 0 || L < 0) return OR_EINVAL;
  for (int32_t i = 0; i < d; ++i) out[i] = 0.0;
  if (L == 0) {
    if (lse) *lse = -INFINITY;
    if (psum) *psum = 0.0;
    return OR_OK;
  }
  double *s = (double *)malloc(sizeof(double) * (size_t)L);
  if (!s) return OR_ENOMEM;
  double smax = -INFINITY;
  for (int64_t j = 0; j < L; ++j) {
    double dot = 0.0;
    for (int32_t i = 0; i < d; ++i) dot += q[i] * K[j * k_row_stride + i];
    s[j] = scale * dot;
    if (s[j] > smax) smax = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < L; ++j) l += exp(s[j] - smax);
  double ps = 0.0;
  for (int64_t j = 0; j < L; ++j) {
    double p = exp(s[j] - smax) / l;
    ps += p;
    for (int32_t i = 0; i < d; ++i) out[i] += p * V[j * v_row_stride + i];
  }
  if (lse) *lse = smax + log(l);
  if (psum) *psum = ps;
  free(s);
  return OR_OK;
}

/* One output row (sequence b, query head h) of paged GQA decode attention.
 * q: [B, H_Q, d]; caches: [num_blocks, block_size, H_KV, d], contiguous;
 * block_tables: [B, max_blocks_per_seq]; context_lens: [B].
 * Query head h reads KV head h / (H_Q / H_KV) (consecutive grouping).
 * Logical token j of sequence b lives in physical block
 * block_tables[b][j / block_size], row j % block_size.  A token whose block
 * id is outside [0, num_blocks) is left out of the softmax (the library never
 * dereferences such ids either).  The context is gathered in logical order
 * and handed to the dense definition above. */
/* With a quantised cache (sglang cache_ops.py, reshape_and_cache_flash,
 * "optional scale": the cache holds x / k_scale and x / v_scale), the value a
 * code stands for is code * scale: K rows are multiplied by k_scale and V rows
 * by v_scale after decoding (in double).  Unquantised caches use 1. */
int or_paged_decode_row_scaled(double *out, double *lse, double *psum, const void *q,
                               int q_dtype, const void *k_cache, const void *v_cache,
                               int cache_dtype, const int32_t *block_tables,
                               const int32_t *context_lens, int32_t b, int32_t h,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                               int32_t block_size, int32_t max_blocks_per_seq,
                               int64_t num_blocks, float scale, float k_scale, float v_scale);

int or_paged_decode_row(double *out, double *lse, double *psum, const void *q, int q_dtype,
                        const void *k_cache, const void *v_cache, int cache_dtype,
                        const int32_t *block_tables, const int32_t *context_lens, int32_t b,
                        int32_t h, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                        int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks,
                        float scale) {
  return or_paged_decode_row_scaled(out, lse, psum, q, q_dtype, k_cache, v_cache, cache_dtype,
                                    block_tables, context_lens, b, h, num_q_heads, num_kv_heads,
                                    head_size, block_size, max_blocks_per_seq, num_blocks, scale,
                                    1.0f, 1.0f);
}

int or_paged_decode_row_scaled(double *out, double *lse, double *psum, const void *q,
                               int q_dtype, const void *k_cache, const void *v_cache,
                               int cache_dtype, const int32_t *block_tables,
                               const int32_t *context_lens, int32_t b, int32_t h,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                               int32_t block_size, int32_t max_blocks_per_seq,
                               int64_t num_blocks, float scale, float k_scale, float v_scale) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return OR_EINVAL;
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return OR_EINVAL;
  if (head_size <= 0 || block_size <= 0 || max_blocks_per_seq < 0) return OR_EINVAL;
  if (h < 0 || h >= num_q_heads || b < 0) return OR_EINVAL;
  const int32_t group = num_q_heads / num_kv_heads;
  const int32_t g = h / group;
  const int64_t L = context_lens[b];
  if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) return OR_EINVAL;
  const int32_t d = head_size;

  double *qd = (double *)malloc(sizeof(double) * (size_t)d);
  double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)d);
  double *V = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)d);
  if (!qd || !K || !V) { free(qd); free(K); free(V); return OR_ENOMEM; }
  for (int32_t i = 0; i < d; ++i)
    qd[i] = load_elem(q_dtype, q, ((int64_t)b * num_q_heads + h) * d + i);

  int64_t n = 0; /* gathered rows */
  for (int64_t j = 0; j < L; ++j) {
    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
    if (blk < 0 || blk >= num_blocks) continue;
    int64_t phys_row = blk * block_size + j % block_size;
    int64_t base = (phys_row * num_kv_heads + g) * d;
    for (int32_t i = 0; i < d; ++i) {
      K[n * d + i] = load_elem(cache_dtype, k_cache, base + i) * (double)k_scale;
      V[n * d + i] = load_elem(cache_dtype, v_cache, base + i) * (double)v_scale;
    }
    ++n;
  }
  int rc = or_dense_attention_row(out, lse, psum, qd, K, d, V, d, n, d, (double)scale);
  free(qd); free(K); free(V);
  return rc;
}

/* All rows: out [B, H_Q, d] as float (the double result rounded once),
 * lse [B, H_Q] (nullable). */
int or_paged_decode(float *out, double *lse, const void *q, int q_dtype, const void *k_cache,
                    const void *v_cache, int cache_dtype, const int32_t *block_tables,
                    const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                    int32_t max_blocks_per_seq, int64_t num_blocks, float scale) {
  if (num_seqs < 0 || head_size <= 0) return OR_EINVAL;
  double *row = (double *)malloc(sizeof(double) * (size_t)head_size);
  if (!row) return OR_ENOMEM;
  for (int32_t b = 0; b < num_seqs; ++b) {
    for (int32_t h = 0; h < num_q_heads; ++h) {
      double l;
      int rc = or_paged_decode_row(row, &l, NULL, q, q_dtype, k_cache, v_cache, cache_dtype,
                                   block_tables, context_lens, b, h, num_q_heads, num_kv_heads,
                                   head_size, block_size, max_blocks_per_seq, num_blocks, scale);
      if (rc != OR_OK) { free(row); return rc; }
      for (int32_t i = 0; i < head_size; ++i)
        out[((int64_t)b * num_q_heads + h) * head_size + i] = (float)row[i];
      if (lse) lse[(int64_t)b * num_q_heads + h] = l;
    }
  }
  free(row);
  return OR_OK;
}

/* ======================================================================== */
/* MLA decode over the latent cache                                          */
/* PagedAttention-principle post, MLA section ("MLA 不直接缓存 k 和 v"): per  */
/* token only c_kv ([d_c]) is cached; k_raw = c_kv W_UK and v_raw = c_kv     */
/* W_UV with W_UK, W_UV: [d_c, H * d_h], reshaped to [H, d_h]; the rope part  */
/* of K is added separately (same post, closing remark of the section).       */
/* ======================================================================== */
/* Cache row of a token: [c_kv (d_c) | k_pe (d_r)], one row per slot, the    */
/* layout [num_blocks, block_size, 1, d_c + d_r].                             */
/*                                                                            */
/* Absorbed form (a reading: associativity of the two products, not printed  */
/* on the pages).  For head h with W_UK_h = W_UK[:, h d_h : (h+1) d_h]:       */
/*   q_nope_h . (c W_UK_h) = (W_UK_h q_nope_h) . c                            */
/*   sum_j p_j (c_j W_UV_h) = (sum_j p_j c_j) W_UV_h                          */
/* so decode is one MQA over the latent rows:                                 */
/*   q_lat[h] = [W_UK_h q_nope_h | q_pe_h]              (d_c + d_r)           */
/*   o_lat[h] = sum_j softmax_j(scale q_lat[h] . row_j) row_j[0:d_c]          */
/*   out[h]   = o_lat[h] W_UV_h                          (d_v)                */

/* q_lat [B, H, d_c + d_r] in double from q_nope [B, H, d_h], q_pe [B, H, d_r]
 * and W_UK [d_c, H * d_h] (row-major), all of in_dtype / w_dtype. */
int or_mla_absorb_q(double *q_lat, const void *q_nope, const void *q_pe, int in_dtype,
                    const void *w_uk, int w_dtype, int32_t num_seqs, int32_t num_heads,
                    int32_t d_h, int32_t d_r, int32_t d_c) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!q_lat || !q_nope || !w_uk || (d_r > 0 && !q_pe)) return OR_EINVAL;
  if (num_seqs < 0 || num_heads <= 0 || d_h <= 0 || d_r < 0 || d_c <= 0) return OR_EINVAL;
  const int64_t row = (int64_t)d_c + d_r;
  const int64_t wcols = (int64_t)num_heads * d_h;
  for (int32_t b = 0; b < num_seqs; ++b) {
    for (int32_t h = 0; h < num_heads; ++h) {
      double *dst = q_lat + ((int64_t)b * num_heads + h) * row;
      const int64_t qn = ((int64_t)b * num_heads + h) * d_h;
      for (int32_t c = 0; c < d_c; ++c) {
        double acc = 0.0;
        for (int32_t i = 0; i < d_h; ++i)
          acc += load_elem(w_dtype, w_uk, (int64_t)c * wcols + (int64_t)h * d_h + i) *
                 load_elem(in_dtype, q_nope, qn + i);
        dst[c] = acc;
      }
      for (int32_t r = 0; r < d_r; ++r)
        dst[d_c + r] = load_elem(in_dtype, q_pe, ((int64_t)b * num_heads + h) * d_r + r);
    }
  }
  return OR_OK;
}

/* One output row (sequence b, head h) of MLA decode over the paged latent
 * cache: scores over all d_c + d_r elements of each row, values = the first
 * d_c.  q_lat [B, H, d_c + d_r] of q_dtype; latent_cache [num_blocks,
 * block_size, d_c + d_r] of cache_dtype.  Tokens are gathered in logical
 * order along the block table; a token whose block id is outside
 * [0, num_blocks) is left out, as in or_paged_decode_row.
 * out [d_c]; lse = log sum exp of the scaled scores (nullable); abs_out
 * [d_c] (nullable) = sum_j p_j |row_j[i]|, the scale of the error a rounding
 * of the weights p_j can cause in out[i]. */
int or_mla_decode_row(double *out, double *lse, double *abs_out, const void *q_lat, int q_dtype,
                      const void *latent_cache, int cache_dtype, const int32_t *block_tables,
                      const int32_t *context_lens, int32_t b, int32_t h, int32_t num_heads,
                      int32_t d_c, int32_t d_r, int32_t block_size, int32_t max_blocks_per_seq,
                      int64_t num_blocks, float scale) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!out || !q_lat || !latent_cache || !block_tables || !context_lens) return OR_EINVAL;
  if (num_heads <= 0 || d_c <= 0 || d_r < 0 || block_size <= 0 || max_blocks_per_seq < 0)
    return OR_EINVAL;
  if (b < 0 || h < 0 || h >= num_heads) return OR_EINVAL;
  const int64_t L = context_lens[b];
  if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) return OR_EINVAL;
  const int32_t dk = d_c + d_r;

  double *qd = (double *)malloc(sizeof(double) * (size_t)dk);
  double *R = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)dk);
  double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  if (!qd || !R || !s) { free(qd); free(R); free(s); return OR_ENOMEM; }
  for (int32_t i = 0; i < dk; ++i)
    qd[i] = load_elem(q_dtype, q_lat, ((int64_t)b * num_heads + h) * dk + i);

  /* gather the context's latent rows in logical order */
  int64_t n = 0;
  for (int64_t j = 0; j < L; ++j) {
    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
    if (blk < 0 || blk >= num_blocks) continue;
    int64_t base = (blk * block_size + j % block_size) * dk;
    for (int32_t i = 0; i < dk; ++i) R[n * dk + i] = load_elem(cache_dtype, latent_cache, base + i);
    ++n;
  }

  for (int32_t i = 0; i < d_c; ++i) {
    out[i] = 0.0;
    if (abs_out) abs_out[i] = 0.0;
  }
  if (n == 0) {
    if (lse) *lse = -INFINITY;
    free(qd); free(R); free(s);
    return OR_OK;
  }
  /* scores over the whole row, then the softmax, then the weighted sum of
   * the first d_c elements */
  double smax = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int32_t i = 0; i < dk; ++i) dot += qd[i] * R[j * dk + i];
    s[j] = (double)scale * dot;
    if (s[j] > smax) smax = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) l += exp(s[j] - smax);
  for (int64_t j = 0; j < n; ++j) {
    double p = exp(s[j] - smax) / l;
    for (int32_t i = 0; i < d_c; ++i) {
      out[i] += p * R[j * dk + i];
      if (abs_out) abs_out[i] += p * fabs(R[j * dk + i]);
    }
  }
  if (lse) *lse = smax + log(l);
  free(qd); free(R); free(s);
  return OR_OK;
}

/* out [B, H, d_v] in double = o_lat[b, h, :] W_UV_h, with o_lat [B, H, d_c]
 * of in_dtype and W_UV [d_c, H * d_v] (row-major) of w_dtype. */
int or_mla_project_out(double *out, const void *o_lat, int in_dtype, const void *w_uv,
                       int w_dtype, int32_t num_seqs, int32_t num_heads, int32_t d_c,
                       int32_t d_v) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!out || !o_lat || !w_uv) return OR_EINVAL;
  if (num_seqs < 0 || num_heads <= 0 || d_c <= 0 || d_v <= 0) return OR_EINVAL;
  const int64_t wcols = (int64_t)num_heads * d_v;
  for (int32_t b = 0; b < num_seqs; ++b) {
    for (int32_t h = 0; h < num_heads; ++h) {
      const int64_t src = ((int64_t)b * num_heads + h) * d_c;
      for (int32_t i = 0; i < d_v; ++i) {
        double acc = 0.0;
        for (int32_t c = 0; c < d_c; ++c)
          acc += load_elem(in_dtype, o_lat, src + c) *
                 load_elem(w_dtype, w_uv, (int64_t)c * wcols + (int64_t)h * d_v + i);
        out[((int64_t)b * num_heads + h) * d_v + i] = acc;
      }
    }
  }
  return OR_OK;
}

/* MLA decode of one (sequence b, head h) row in the pages' own form, with
 * no absorption (PagedAttention-principle post, MLA section): for every
 * context token j, gathered in logical order along the block table, rebuild
 *   K_j = [c_kv_j W_UK_h | k_pe_j]          (d_h + d_r)
 *   V_j =  c_kv_j W_UV_h                     (d_v)
 * from its cached row [c_kv_j | k_pe_j], then plain softmax attention of
 *   q = [q_nope[b, h] | q_pe[b, h]]:  s_j = scale q . K_j,
 *   out = sum_j softmax_j(s) V_j.
 * W_UK [d_c, H * d_h] and W_UV [d_c, H * d_v] row-major, head h owning
 * columns h*d_h .. (h+1)*d_h - 1 (resp. d_v).  q_nope [B, H, d_h], q_pe
 * [B, H, d_r] of q_dtype; latent_cache [num_blocks, block_size, d_c + d_r]
 * of cache_dtype; weights of w_dtype.  out [d_v]; lse nullable.  A token
 * whose block id is outside [0, num_blocks) is left out. */
int or_mla_decode_explicit(double *out, double *lse, const void *q_nope, const void *q_pe,
                           int q_dtype, const void *latent_cache, int cache_dtype,
                           const void *w_uk, const void *w_uv, int w_dtype,
                           const int32_t *block_tables, const int32_t *context_lens, int32_t b,
                           int32_t h, int32_t num_heads, int32_t d_h, int32_t d_r, int32_t d_c,
                           int32_t d_v, int32_t block_size, int32_t max_blocks_per_seq,
                           int64_t num_blocks, float scale) {
  if (!formats_ready()) return OR_ENOMEM;
  if (!out || !q_nope || (d_r > 0 && !q_pe) || !latent_cache || !w_uk || !w_uv ||
      !block_tables || !context_lens)
    return OR_EINVAL;
  if (num_heads <= 0 || d_h <= 0 || d_r < 0 || d_c <= 0 || d_v <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0 || b < 0 || h < 0 || h >= num_heads)
    return OR_EINVAL;
  const int64_t L = context_lens[b];
  if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) return OR_EINVAL;
  const int32_t row = d_c + d_r;
  const int32_t dk = d_h + d_r;

  double *q = (double *)malloc(sizeof(double) * (size_t)dk);
  double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)dk);
  double *V = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)d_v);
  double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  double *c = (double *)malloc(sizeof(double) * (size_t)row);
  /* head h's weight columns, decoded once: wk[i][k] = W_UK[k, h d_h + i],
   * wv[i][k] = W_UV[k, h d_v + i] */
  double *wk = (double *)malloc(sizeof(double) * (size_t)d_h * (size_t)d_c);
  double *wv = (double *)malloc(sizeof(double) * (size_t)d_v * (size_t)d_c);
  if (!q || !K || !V || !s || !c || !wk || !wv) {
    free(q); free(K); free(V); free(s); free(c); free(wk); free(wv);
    return OR_ENOMEM;
  }
  for (int32_t k = 0; k < d_c; ++k) {
    for (int32_t i = 0; i < d_h; ++i)
      wk[(int64_t)i * d_c + k] =
          load_elem(w_dtype, w_uk, (int64_t)k * num_heads * d_h + (int64_t)h * d_h + i);
    for (int32_t i = 0; i < d_v; ++i)
      wv[(int64_t)i * d_c + k] =
          load_elem(w_dtype, w_uv, (int64_t)k * num_heads * d_v + (int64_t)h * d_v + i);
  }
  for (int32_t i = 0; i < d_h; ++i)
    q[i] = load_elem(q_dtype, q_nope, ((int64_t)b * num_heads + h) * d_h + i);
  for (int32_t r = 0; r < d_r; ++r)
    q[d_h + r] = load_elem(q_dtype, q_pe, ((int64_t)b * num_heads + h) * d_r + r);

  /* rebuild K and V of head h for every context token */
  int64_t n = 0;
  for (int64_t j = 0; j < L; ++j) {
    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
    if (blk < 0 || blk >= num_blocks) continue;
    int64_t base = (blk * block_size + j % block_size) * row;
    for (int32_t i = 0; i < row; ++i) c[i] = load_elem(cache_dtype, latent_cache, base + i);
    for (int32_t i = 0; i < d_h; ++i) { /* K_j[i] = sum_k c_kv_j[k] W_UK[k, h d_h + i] */
      double acc = 0.0;
      for (int32_t k = 0; k < d_c; ++k) acc += c[k] * wk[(int64_t)i * d_c + k];
      K[n * dk + i] = acc;
    }
    for (int32_t r = 0; r < d_r; ++r) K[n * dk + d_h + r] = c[d_c + r];
    for (int32_t i = 0; i < d_v; ++i) { /* V_j[i] = sum_k c_kv_j[k] W_UV[k, h d_v + i] */
      double acc = 0.0;
      for (int32_t k = 0; k < d_c; ++k) acc += c[k] * wv[(int64_t)i * d_c + k];
      V[n * d_v + i] = acc;
    }
    ++n;
  }

  for (int32_t i = 0; i < d_v; ++i) out[i] = 0.0;
  if (n == 0) {
    if (lse) *lse = -INFINITY;
  } else {
    /* plain softmax attention over the rebuilt K and V */
    double smax = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      double dot = 0.0;
      for (int32_t i = 0; i < dk; ++i) dot += q[i] * K[j * dk + i];
      s[j] = (double)scale * dot;
      if (s[j] > smax) smax = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += exp(s[j] - smax);
    for (int64_t j = 0; j < n; ++j) {
      double p = exp(s[j] - smax) / l;
      for (int32_t i = 0; i < d_v; ++i) out[i] += p * V[j * d_v + i];
    }
    if (lse) *lse = smax + log(l);
  }
  free(q); free(K); free(V); free(s); free(c); free(wk); free(wv);
  return OR_OK;
}
