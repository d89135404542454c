"""CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product path (the
CUDA library and its binding) never imports this package, and this package
imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, double precision, nested
loops); this module compiles it with gcc on first use and wraps it with
ctypes.  Arrays are numpy; half-width formats travel as their raw integer
codes (bf16/fp16 as uint16, fp8 e4m3 as uint8).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# dtype codes of the oracle's own enumeration
BF16, FP16, FP32, E4M3 = 0, 1, 2, 3
FP64 = 4  # read-only input format (plain float64 arrays) of the MLA functions
_NP_CODE_TYPE = {BF16: np.uint16, FP16: np.uint16, FP32: np.float32, E4M3: np.uint8,
                 FP64: np.float64}
DTYPE_NAMES = {"bf16": BF16, "fp16": FP16, "fp32": FP32, "e4m3": E4M3}

ERRORS = {-1: "invalid argument", -2: "duplicate target slot", -3: "out of memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math,
    no FMA contraction) and return the library path."""
    with _lock:
        fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
        if force or not fresh:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                   "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P, I32, I64, F32, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    C_INT = ctypes.c_int
    lib.or_encode_array.argtypes = [C_INT, P, I64, P]
    lib.or_encode_array.restype = C_INT
    lib.or_decode_array.argtypes = [C_INT, P, I64, P]
    lib.or_decode_array.restype = C_INT
    lib.or_format_info.argtypes = [C_INT, P, P]
    lib.or_format_info.restype = C_INT
    lib.or_reshape_and_cache.argtypes = [P, P, C_INT, I64, I32, I32, I64, I64, P, P, C_INT,
                                         I64, I32, I64, P, P, I64, P, P]
    lib.or_reshape_and_cache.restype = I64
    lib.or_concat_mla_k.argtypes = [P, C_INT, P, P, C_INT, I64, I32, I32, I32, I64, I64, I64,
                                    I64, I64]
    lib.or_concat_mla_k.restype = C_INT
    lib.or_dense_attention_row.argtypes = [P, P, P, P, P, I64, P, I64, I64, I32, D]
    lib.or_dense_attention_row.restype = C_INT
    lib.or_paged_decode_row.argtypes = [P, P, P, P, C_INT, P, P, C_INT, P, P, I32, I32, I32,
                                        I32, I32, I32, I32, I64, F32]
    lib.or_paged_decode_row.restype = C_INT
    lib.or_paged_decode_row_scaled.argtypes = [P, P, P, P, C_INT, P, P, C_INT, P, P, I32, I32,
                                               I32, I32, I32, I32, I32, I64, F32, F32, F32]
    lib.or_paged_decode_row_scaled.restype = C_INT
    lib.or_paged_decode.argtypes = [P, P, P, C_INT, P, P, C_INT, P, P, I32, I32, I32, I32, I32,
                                    I32, I64, F32]
    lib.or_paged_decode.restype = C_INT
    lib.or_mla_absorb_q.argtypes = [P, P, P, C_INT, P, C_INT, I32, I32, I32, I32, I32]
    lib.or_mla_absorb_q.restype = C_INT
    lib.or_mla_decode_row.argtypes = [P, P, P, P, C_INT, P, C_INT, P, P, I32, I32, I32, I32,
                                      I32, I32, I32, I64, F32]
    lib.or_mla_decode_row.restype = C_INT
    lib.or_mla_project_out.argtypes = [P, P, C_INT, P, C_INT, I32, I32, I32, I32]
    lib.or_mla_project_out.restype = C_INT
    lib.or_mla_decode_explicit.argtypes = [P, P, P, P, C_INT, P, C_INT, P, P, C_INT, P, P, I32,
                                           I32, I32, I32, I32, I32, I32, I32, I32, I64, F32]
    lib.or_mla_decode_explicit.restype = C_INT
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc < 0:
        raise OracleError(ERRORS.get(int(rc), f"error {rc}"))
    return rc


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats --
def encode(dtype: int, y) -> np.ndarray:
    """float32 values -> codes of `dtype` (nearest, ties to even; e4m3
    saturates to +-448; NaN -> quiet NaN)."""
    y = _c(y, np.float32)
    out = np.empty(y.shape, dtype=_NP_CODE_TYPE[dtype])
    _check(_load().or_encode_array(dtype, _ptr(y), y.size, _ptr(out)))
    return out


def decode(dtype: int, codes) -> np.ndarray:
    """codes of `dtype` -> float64 values."""
    codes = _c(codes, _NP_CODE_TYPE[dtype])
    out = np.empty(codes.shape, dtype=np.float64)
    _check(_load().or_decode_array(dtype, _ptr(codes), codes.size, _ptr(out)))
    return out


def format_info(dtype: int):
    """(number of non-negative finite values, largest finite value)."""
    n = ctypes.c_int64()
    m = ctypes.c_double()
    _check(_load().or_format_info(dtype, ctypes.byref(n), ctypes.byref(m)))
    return n.value, m.value


# ------------------------------------------------------------ cache write --
def reshape_and_cache(key, value, src_dtype, key_cache, value_cache, cache_dtype,
                      slot_mapping, swa_slot_mapping=None, k_scale=None, v_scale=None,
                      key_stride=None, value_stride=None, block_stride=None,
                      num_heads=None, head_size=None):
    """Scatter key/value [N, H, d] into the caches [num_blocks, bs, H, d]
    IN PLACE (the cache arrays are modified).  Returns the number of tokens
    written.  key/value may be 2-D [N, row] views with explicit strides when
    num_heads/head_size are given."""
    if num_heads is None:
        _, num_heads, head_size = key.shape
    num_tokens = key.shape[0]
    if key_stride is None:
        key_stride = key.strides[0] // key.itemsize
    if value is not None and value_stride is None:
        value_stride = value.strides[0] // value.itemsize
    if value_stride is None:
        value_stride = 0
    num_blocks, block_size = key_cache.shape[0], key_cache.shape[1]
    if block_stride is None:
        block_stride = key_cache.strides[0] // key_cache.itemsize
    slot_mapping = _c(slot_mapping, np.int64)
    swa = None if swa_slot_mapping is None else _c(swa_slot_mapping, np.int64)
    ks = None if k_scale is None else np.array([k_scale], dtype=np.float32)
    vs = None if v_scale is None else np.array([v_scale], dtype=np.float32)
    rc = _load().or_reshape_and_cache(
        _ptr(key), _ptr(value), src_dtype, num_tokens, num_heads, head_size, key_stride,
        value_stride, _ptr(key_cache), _ptr(value_cache), cache_dtype, num_blocks, block_size,
        block_stride, _ptr(slot_mapping), _ptr(swa), 0 if swa is None else swa.size,
        _ptr(ks), _ptr(vs))
    return _check(rc)


# ------------------------------------------------------------- MLA concat --
def concat_mla_k(k, k_dtype, k_nope, k_rope, src_dtype):
    """k[n, h, :nope] = k_nope[n, h, :]; k[n, h, nope:] = k_rope[n, 0, :]
    (k modified in place; all arrays 3-D with a contiguous last axis)."""
    n, h, nope = k_nope.shape
    rope = k_rope.shape[2]
    es = lambda a, i: a.strides[i] // a.itemsize
    _check(_load().or_concat_mla_k(
        _ptr(k), k_dtype, _ptr(k_nope), _ptr(k_rope), src_dtype, n, h, nope, rope,
        es(k, 0), es(k, 1), es(k_nope, 0), es(k_nope, 1), es(k_rope, 0)))
    return k


# -------------------------------------------------------- decode attention --
def dense_attention_row(q, K, V, scale):
    """Dense softmax attention of one query over contiguous rows.
    Returns (out[d] float64, lse, sum of the softmax weights)."""
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    L, d = K.shape
    out = np.empty(d, dtype=np.float64)
    lse = ctypes.c_double()
    ps = ctypes.c_double()
    _check(_load().or_dense_attention_row(_ptr(out), ctypes.byref(lse), ctypes.byref(ps),
                                          _ptr(q), _ptr(K), d, _ptr(V), d, L, d, float(scale)))
    return out, lse.value, ps.value


def paged_decode_row(q, k_cache, v_cache, block_tables, context_lens, b, h, scale,
                     q_dtype=BF16, cache_dtype=BF16, k_scale=1.0, v_scale=1.0):
    """One (sequence, query head) row of paged GQA decode attention.
    q [B, H_Q, d] codes; caches [num_blocks, bs, H_KV, d] codes; a quantised
    cache's codes stand for code * k_scale (K) and code * v_scale (V).
    Returns (out[d] float64, lse, sum of softmax weights)."""
    B, HQ, d = q.shape
    nb, bs, HKV, d2 = k_cache.shape
    assert d == d2
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.empty(d, dtype=np.float64)
    lse = ctypes.c_double()
    ps = ctypes.c_double()
    _check(_load().or_paged_decode_row_scaled(
        _ptr(out), ctypes.byref(lse), ctypes.byref(ps), _ptr(_c(q, q.dtype)), q_dtype,
        _ptr(_c(k_cache, k_cache.dtype)), _ptr(_c(v_cache, v_cache.dtype)), cache_dtype,
        _ptr(bt), _ptr(cl), b, h, HQ, HKV, d, bs, bt.shape[1], nb, float(scale), float(k_scale),
        float(v_scale)))
    return out, lse.value, ps.value


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                 q_dtype=BF16, cache_dtype=BF16):
    """Every row: returns (out [B, H_Q, d] float32, lse [B, H_Q] float64)."""
    B, HQ, d = q.shape
    nb, bs, HKV, _ = k_cache.shape
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.empty((B, HQ, d), dtype=np.float32)
    lse = np.empty((B, HQ), dtype=np.float64)
    _check(_load().or_paged_decode(
        _ptr(out), _ptr(lse), _ptr(_c(q, q.dtype)), q_dtype, _ptr(_c(k_cache, k_cache.dtype)),
        _ptr(_c(v_cache, v_cache.dtype)), cache_dtype, _ptr(bt), _ptr(cl), B, HQ, HKV, d, bs,
        bt.shape[1], nb, float(scale)))
    return out, lse


def paged_prefill_row(q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens, b, j, h,
                      scale, q_dtype=BF16, cache_dtype=BF16):
    """Causal prefill attention of one new token: sequence b's j-th new token
    (of n = cu_seqlens_q[b+1] - cu_seqlens_q[b]) sits at position
    p = context_lens[b] - n + j and attends to the cached tokens 0..p, i.e.
    decode attention over a context of p + 1 tokens.  q is [total, H_Q, d].
    Returns (out[d] float64, lse, sum of softmax weights)."""
    n = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
    p = int(context_lens[b]) - n + j
    row = int(cu_seqlens_q[b]) + j
    lens = np.zeros(np.asarray(context_lens).shape, np.int32)
    lens[b] = max(p + 1, 0)
    qrow = np.zeros((len(lens),) + tuple(q.shape[1:]), dtype=q.dtype)
    qrow[b] = q[row]
    return paged_decode_row(qrow, k_cache, v_cache, block_tables, lens, b, h, scale,
                            q_dtype=q_dtype, cache_dtype=cache_dtype)


# ------------------------------------------------------------- MLA decode --
def mla_absorb_q(q_nope, q_pe, w_uk, in_dtype=BF16, w_dtype=BF16):
    """q_lat [B, H, d_c + d_r] float64: [W_UK_h q_nope[b, h] | q_pe[b, h]],
    with W_UK [d_c, H * d_h] and W_UK_h its columns h*d_h .. (h+1)*d_h - 1."""
    B, H, dh = q_nope.shape
    dr = q_pe.shape[2]
    dc = w_uk.shape[0]
    assert w_uk.shape[1] == H * dh and q_pe.shape[:2] == (B, H)
    out = np.empty((B, H, dc + dr), dtype=np.float64)
    _check(_load().or_mla_absorb_q(_ptr(out), _ptr(_c(q_nope, q_nope.dtype)),
                                   _ptr(_c(q_pe, q_pe.dtype)), in_dtype,
                                   _ptr(_c(w_uk, w_uk.dtype)), w_dtype, B, H, dh, dr, dc))
    return out


def mla_decode_row(q_lat, latent_cache, block_tables, context_lens, b, h, scale, d_c,
                   q_dtype=BF16, cache_dtype=BF16):
    """One (sequence, head) row of MLA decode over the paged latent cache.
    q_lat [B, H, d_c + d_r]; latent_cache [num_blocks, bs, (1,) d_c + d_r].
    Returns (o_lat[d_c] float64, lse, abs_out[d_c]) where abs_out[i] =
    sum_j p_j |row_j[i]|."""
    B, H, dk = q_lat.shape
    nb, bs = latent_cache.shape[0], latent_cache.shape[1]
    assert latent_cache.shape[-1] == dk and latent_cache.size == nb * bs * dk
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.empty(d_c, dtype=np.float64)
    ab = np.empty(d_c, dtype=np.float64)
    lse = ctypes.c_double()
    _check(_load().or_mla_decode_row(
        _ptr(out), ctypes.byref(lse), _ptr(ab), _ptr(_c(q_lat, q_lat.dtype)), q_dtype,
        _ptr(_c(latent_cache, latent_cache.dtype)), cache_dtype, _ptr(bt), _ptr(cl), b, h, H,
        d_c, dk - d_c, bs, bt.shape[1], nb, float(scale)))
    return out, lse.value, ab


def mla_project_out(o_lat, w_uv, in_dtype=BF16, w_dtype=BF16):
    """out [B, H, d_v] float64 = o_lat[b, h, :] W_UV_h with W_UV [d_c, H * d_v]."""
    B, H, dc = o_lat.shape
    assert w_uv.shape[0] == dc and w_uv.shape[1] % H == 0
    dv = w_uv.shape[1] // H
    out = np.empty((B, H, dv), dtype=np.float64)
    _check(_load().or_mla_project_out(_ptr(out), _ptr(_c(o_lat, o_lat.dtype)), in_dtype,
                                      _ptr(_c(w_uv, w_uv.dtype)), w_dtype, B, H, dc, dv))
    return out


def mla_decode_explicit_row(q_nope, q_pe, latent_cache, w_uk, w_uv, block_tables, context_lens,
                            b, h, scale, d_c, q_dtype=BF16, cache_dtype=BF16, w_dtype=BF16):
    """One (sequence, head) row of MLA decode in the pages' form: rebuild
    K_j = [c_kv_j W_UK_h | k_pe_j] and V_j = c_kv_j W_UV_h for every context
    token, then softmax attention of [q_nope | q_pe].  q_nope [B, H, d_h],
    q_pe [B, H, d_r], latent_cache [num_blocks, bs, (1,) d_c + d_r], w_uk
    [d_c, H * d_h], w_uv [d_c, H * d_v].  Returns (out[d_v] float64, lse)."""
    B, H, dh = q_nope.shape
    dr = q_pe.shape[2]
    nb, bs = latent_cache.shape[0], latent_cache.shape[1]
    assert latent_cache.shape[-1] == d_c + dr and latent_cache.size == nb * bs * (d_c + dr)
    assert w_uk.shape == (d_c, H * dh) and w_uv.shape[0] == d_c and w_uv.shape[1] % H == 0
    dv = w_uv.shape[1] // H
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.empty(dv, dtype=np.float64)
    lse = ctypes.c_double()
    _check(_load().or_mla_decode_explicit(
        _ptr(out), ctypes.byref(lse), _ptr(_c(q_nope, q_nope.dtype)), _ptr(_c(q_pe, q_pe.dtype)),
        q_dtype, _ptr(_c(latent_cache, latent_cache.dtype)), cache_dtype,
        _ptr(_c(w_uk, w_uk.dtype)), _ptr(_c(w_uv, w_uv.dtype)), w_dtype, _ptr(bt), _ptr(cl), b,
        h, H, dh, dr, d_c, dv, bs, bt.shape[1], nb, float(scale)))
    return out, lse.value
