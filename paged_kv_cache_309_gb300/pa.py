"""Thin ctypes binding of libpa.so, same names as the C ABI (include/pa.h).

Argument marshalling only: each function turns torch tensors into device
pointers, sizes and strides, passes the current (or given) CUDA stream and
raises ``PAError`` on a non-OK status.  All computation happens in the CUDA
library; there is no fallback: if ``libpa.so`` is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pa.h")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_ALIGN, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(6)
PA_BF16, PA_FP16, PA_FP32, PA_FP8_E4M3 = range(4)
PA_DEVERR_WAIT_TIMEOUT = 0x1
PA_DEVERR_CONTEXT_CLIPPED = 0x2
PA_DEVERR_SLOT_MISMATCH = 0x4

_TORCH_DTYPE = {torch.bfloat16: PA_BF16, torch.float16: PA_FP16, torch.float32: PA_FP32,
                torch.float8_e4m3fn: PA_FP8_E4M3}

_lib = None


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _load().pa_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg}")


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                           "(paged_kv_cache_309_gb300.build.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    E = ctypes.c_int  # enums
    lib.pa_status_string.argtypes = [E]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_reshape_and_cache.argtypes = [P, P, E, I64, I32, I32, I64, I64, P, P, E, I64, I32, I64,
                                         P, P, I64, P, P, P]
    lib.pa_reshape_and_cache.restype = E
    lib.pa_concat_mla_k.argtypes = [P, E, P, P, E, I64, I32, I32, I32, I64, I64, I64, I64, I64, P]
    lib.pa_concat_mla_k.restype = E
    lib.pa_concat_and_cache_mla.argtypes = [P, P, E, I64, I32, I32, I64, I64, P, E, I64, I32,
                                            I64, P, P, P]
    lib.pa_concat_and_cache_mla.restype = E
    lib.pa_paged_decode_workspace_size.argtypes = [I32, I32, I32, I32, I32]
    lib.pa_paged_decode_workspace_size.restype = SZ
    lib.pa_paged_decode_attention.argtypes = [P, P, P, P, E, P, P, I32, I32, I32, I32, I32, I32,
                                              I64, F32, I32, P, SZ, P]
    lib.pa_paged_decode_attention.restype = E
    lib.pa_paged_decode_attention_fp8.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I32, I32,
                                                  I32, I32, I64, F32, I32, P, SZ, P]
    lib.pa_paged_decode_attention_fp8.restype = E
    lib.pa_paged_decode_step.argtypes = [P, P, P, P, P, P, P, E, P, P, P, P, I32, I32, I32, I32,
                                         I32, I32, I64, F32, I32, P, SZ, P]
    lib.pa_paged_decode_step.restype = E
    lib.pa_paged_prefill_attention.argtypes = [P, P, P, P, E, P, P, P, I32, I32, I32, I32, I32,
                                               I32, I64, F32, I32, P, P]
    lib.pa_paged_prefill_attention.restype = E
    lib.pa_paged_decode_attention_static.argtypes = [P, P, P, P, E, P, P, I32, I32, I32, I32,
                                                     I32, I32, I64, F32, I32, P, P]
    lib.pa_paged_decode_attention_static.restype = E
    lib.pa_paged_decode_plan.argtypes = [I32, I32, I32, I32, ctypes.POINTER(I32),
                                         ctypes.POINTER(I32)]
    lib.pa_paged_decode_plan.restype = E
    lib.pa_mla_absorb_q.argtypes = [P, P, P, P, I32, I32, I32, I32, I32, P]
    lib.pa_mla_absorb_q.restype = E
    lib.pa_mla_decode_workspace_size.argtypes = [I32, I32, I32]
    lib.pa_mla_decode_workspace_size.restype = SZ
    lib.pa_mla_decode_attention.argtypes = [P, P, P, P, P, I32, I32, I32, I32, I32, I32, I64,
                                            ctypes.c_float, I32, P, SZ, P]
    lib.pa_mla_decode_attention.restype = E
    lib.pa_mla_project_out.argtypes = [P, P, P, I32, I32, I32, I32, P]
    lib.pa_mla_project_out.restype = E
    lib.pa_selftest_bounded_wait.argtypes = [P, P]
    lib.pa_selftest_bounded_wait.restype = E
    _lib = lib
    return lib


def library():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def declared_functions():
    """Names of the functions include/pa.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def _check(status, where):
    if status != PA_OK:
        raise PAError(status, where)


def _on_device(**tensors):
    """Refuse, before anything is launched, a tensor the kernels cannot use:
    every tensor passed (None is skipped) must be a CUDA tensor on the
    current CUDA device, because the library takes its pointers as device
    addresses of that device (a host or another GPU's pointer would be
    dereferenced as one)."""
    cur = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name} must be a torch tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (it is on {t.device})")
        if cur is None:
            cur = torch.cuda.current_device()
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur}")


def _word(t, name):
    """A device word the kernels OR 4-byte error bits into: int32, at least
    one element, on the current device."""
    if t is None:
        return
    _on_device(**{name: t})
    if t.dtype != torch.int32 or t.numel() < 1:
        raise ValueError(f"{name} must be an int32 tensor with at least one element")


def _scales(k_scale, v_scale):
    """k_scale/v_scale: both None, or both one-element float32 device tensors."""
    if (k_scale is None) != (v_scale is None):
        raise ValueError("give both k_scale and v_scale, or neither")
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is None:
            continue
        _on_device(**{name: t})
        if t.dtype != torch.float32 or t.numel() < 1:
            raise ValueError(f"{name} must be a float32 tensor with at least one element")


def _workspace(t):
    """A decode workspace: a uint8 device tensor on the current device."""
    _on_device(workspace=t)
    if not t.is_contiguous():
        raise ValueError("workspace must be contiguous")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    if stream is not None and s.device.index != torch.cuda.current_device():
        raise ValueError(f"stream belongs to {s.device}, not the current device")
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t):
    try:
        return _TORCH_DTYPE[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


def pa_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                         swa_slot_mapping=None, k_scale=None, v_scale=None, stream=None):
    """key/value [N, H, d] (token stride free), caches [num_blocks, bs, H, d]
    (block stride free), slot_mapping [N] int64, optional swa table int64,
    optional k_scale/v_scale one-element float32 device tensors."""
    _on_device(key=key, value=value, key_cache=key_cache, value_cache=value_cache,
               slot_mapping=slot_mapping, swa_slot_mapping=swa_slot_mapping)
    _scales(k_scale, v_scale)
    lib = _load()
    N, H, d = key.shape
    if key.stride(2) != 1 or key.stride(1) != d:
        raise ValueError("key: heads and elements must be contiguous")
    if value is not None and (value.shape != key.shape or value.stride(2) != 1
                              or value.stride(1) != d):
        raise ValueError("value must match key and be contiguous per token")
    nb, bs, Hc, dc = key_cache.shape
    if (Hc, dc) != (H, d) or key_cache.stride(3) != 1 or key_cache.stride(2) != d \
            or key_cache.stride(1) != H * d:
        raise ValueError("key_cache must be [num_blocks, bs, H, d], contiguous inside a block")
    if value_cache is not None and (value_cache.shape != key_cache.shape
                                    or value_cache.stride() != key_cache.stride()
                                    or value_cache.dtype != key_cache.dtype):
        raise ValueError("value_cache must match key_cache")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != N:
        raise ValueError("slot_mapping must be int64 [N]")
    swa_len = 0
    if swa_slot_mapping is not None:
        if swa_slot_mapping.dtype != torch.int64:
            raise ValueError("swa_slot_mapping must be int64")
        swa_len = swa_slot_mapping.numel()
    st = lib.pa_reshape_and_cache(
        _ptr(key), _ptr(value), _dtype(key), N, H, d, key.stride(0),
        0 if value is None else value.stride(0), _ptr(key_cache), _ptr(value_cache),
        _dtype(key_cache), nb, bs, key_cache.stride(0), _ptr(slot_mapping),
        _ptr(swa_slot_mapping), swa_len, _ptr(k_scale), _ptr(v_scale), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_concat_mla_k(k, k_nope, k_rope, stream=None):
    """k [N, H, nope+rope] <- k_nope [N, H, nope] | k_rope [N, 1, rope]."""
    _on_device(k=k, k_nope=k_nope, k_rope=k_rope)
    lib = _load()
    N, H, nope = k_nope.shape
    rope = k_rope.shape[2]
    for t in (k, k_nope, k_rope):
        if t.stride(2) != 1:
            raise ValueError("last dimension must be contiguous")
    if k.shape != (N, H, nope + rope) or k_rope.shape[:2] != (N, 1):
        raise ValueError("shape mismatch")
    if k_rope.dtype != k_nope.dtype:
        raise ValueError("k_nope and k_rope must share a dtype")
    st = lib.pa_concat_mla_k(_ptr(k), _dtype(k), _ptr(k_nope), _ptr(k_rope), _dtype(k_nope), N, H,
                             nope, rope, k.stride(0), k.stride(1), k_nope.stride(0),
                             k_nope.stride(1), k_rope.stride(0), _stream(stream))
    _check(st, "pa_concat_mla_k")


def pa_concat_and_cache_mla(kv_c, k_pe, latent_cache, slot_mapping, scale=None, stream=None):
    """latent_cache [num_blocks, bs, (1,) d_c + d_r] <- [kv_c[t] | k_pe[t]] at
    slot_mapping[t] (int64 [N]; negative or out-of-pool slots skipped);
    kv_c [N, d_c] and k_pe [N, d_r] (token stride free, rows contiguous);
    optional scale: one-element float32 device tensor (x / scale before the
    cast)."""
    _on_device(kv_c=kv_c, k_pe=k_pe, latent_cache=latent_cache, slot_mapping=slot_mapping)
    if scale is not None:
        _on_device(scale=scale)
        if scale.dtype != torch.float32 or scale.numel() < 1:
            raise ValueError("scale must be a float32 tensor with at least one element")
    lib = _load()
    kc = kv_c.view(kv_c.shape[0], -1) if kv_c.dim() == 3 else kv_c
    kp = k_pe.view(k_pe.shape[0], -1) if k_pe.dim() == 3 else k_pe
    N, dc = kc.shape
    dr = kp.shape[1]
    if kp.shape[0] != N or kc.stride(1) != 1 or kp.stride(1) != 1:
        raise ValueError("kv_c [N, d_c] and k_pe [N, d_r] with contiguous rows expected")
    if kp.dtype != kc.dtype:
        raise ValueError("kv_c and k_pe must share a dtype")
    nb, bs = latent_cache.shape[0], latent_cache.shape[1]
    if latent_cache.shape[-1] != dc + dr or latent_cache.numel() != nb * bs * (dc + dr) \
            or not latent_cache.is_contiguous():
        raise ValueError("latent_cache must be [num_blocks, bs, (1,) d_c + d_r], contiguous")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != N:
        raise ValueError("slot_mapping must be int64 [N]")
    st = lib.pa_concat_and_cache_mla(
        _ptr(kc), _ptr(kp), _dtype(kc), N, dc, dr, kc.stride(0), kp.stride(0),
        _ptr(latent_cache), _dtype(latent_cache), nb, bs, bs * (dc + dr), _ptr(slot_mapping),
        _ptr(scale), _stream(stream))
    _check(st, "pa_concat_and_cache_mla")


def pa_paged_decode_plan(num_seqs, num_kv_heads, max_context_len, num_sms=0):
    """(num_splits, tokens_per_split) of the decode split plan."""
    lib = _load()
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.pa_paged_decode_plan(num_seqs, num_kv_heads, max_context_len, num_sms,
                                    ctypes.byref(a), ctypes.byref(b)), "pa_paged_decode_plan")
    return a.value, b.value


def pa_paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                   max_context_len):
    return int(_load().pa_paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                      head_size, max_context_len))


def decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_size, max_context_len,
                     device=None):
    """A zeroed device workspace of the required size (allocated by torch)."""
    n = pa_paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                       max_context_len)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def read_device_error(workspace) -> int:
    """The sticky device-side error word (first 4 bytes of the workspace)."""
    return int(workspace[:4].view(torch.int32).item())


def pa_paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                              max_context_len, workspace, stream=None, k_scale=None,
                              v_scale=None):
    """out/q [B, H_Q, d] bf16; caches [num_blocks, bs, H_KV, d] bf16 or
    float8_e4m3fn, contiguous; block_tables [B, max_blocks_per_seq] int32;
    context_lens [B] int32.  With k_scale/v_scale (one-element float32 device
    tensors) the e4m3 cache goes through pa_paged_decode_attention_fp8."""
    _on_device(out=out, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               context_lens=context_lens)
    _workspace(workspace)
    _scales(k_scale, v_scale)
    lib = _load()
    B, HQ, d = q.shape
    nb, bs, HKV, dc = k_cache.shape
    for t, name in ((q, "q"), (out, "out"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                    (block_tables, "block_tables"), (context_lens, "context_lens")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out.shape != q.shape or v_cache.shape != k_cache.shape or dc != d:
        raise ValueError("shape mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks_per_seq], context_lens [B]")
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("q and out must be bf16")
    if k_scale is not None or v_scale is not None:
        if k_cache.dtype != torch.float8_e4m3fn:
            raise ValueError("k_scale/v_scale apply to an e4m3 cache")
        st = lib.pa_paged_decode_attention_fp8(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_tables), _ptr(context_lens), B, HQ, HKV, d, bs, block_tables.shape[1], nb,
            float(scale), int(max_context_len), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
        _check(st, "pa_paged_decode_attention_fp8")
        return
    st = lib.pa_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype(k_cache), _ptr(block_tables),
        _ptr(context_lens), B, HQ, HKV, d, bs, block_tables.shape[1], nb, float(scale),
        int(max_context_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st, "pa_paged_decode_attention")


def pa_paged_decode_attention_static(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                     max_context_len, error_word=None, stream=None):
    """Decode attention without a caller workspace: the split-K partials go
    to the library's own 16 MiB device scratch (for callers that cannot
    allocate device memory).  error_word: None or a one-element int32 device
    tensor that receives the device-side error bits.  Calls sharing the
    scratch must be ordered on one stream."""
    _on_device(out=out, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               context_lens=context_lens)
    _word(error_word, "error_word")
    lib = _load()
    B, HQ, d = q.shape
    nb, bs, HKV, dc = k_cache.shape
    for t, name in ((q, "q"), (out, "out"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                    (block_tables, "block_tables"), (context_lens, "context_lens")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out.shape != q.shape or v_cache.shape != k_cache.shape or dc != d:
        raise ValueError("shape mismatch")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    st = lib.pa_paged_decode_attention_static(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype(k_cache), _ptr(block_tables),
        _ptr(context_lens), B, HQ, HKV, d, bs, block_tables.shape[1], nb, float(scale),
        int(max_context_len), _ptr(error_word), _stream(stream))
    _check(st, "pa_paged_decode_attention_static")


def pa_paged_decode_step(out, q, new_k, new_v, slot_mapping, k_cache, v_cache, block_tables,
                         context_lens, scale, max_context_len, workspace, k_scale=None,
                         v_scale=None, stream=None):
    """One decode step in one launch: new_k/new_v [B, H_KV, d] bf16 are
    written at slot_mapping [B] int64 (bf16 cache, or e4m3 cache with
    k_scale/v_scale), then attention over the cache as in
    pa_paged_decode_attention."""
    _on_device(out=out, q=q, new_k=new_k, new_v=new_v, slot_mapping=slot_mapping,
               k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               context_lens=context_lens)
    _workspace(workspace)
    _scales(k_scale, v_scale)
    lib = _load()
    B, HQ, d = q.shape
    nb, bs, HKV, dc = k_cache.shape
    for t, name in ((q, "q"), (out, "out"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                    (new_k, "new_k"), (new_v, "new_v"), (block_tables, "block_tables"),
                    (context_lens, "context_lens"), (slot_mapping, "slot_mapping")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if new_k.shape != (B, HKV, d) or new_v.shape != (B, HKV, d) or new_k.dtype != torch.bfloat16:
        raise ValueError("new_k/new_v must be bf16 [B, H_KV, d]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != B:
        raise ValueError("slot_mapping must be int64 [B]")
    st = lib.pa_paged_decode_step(
        _ptr(out), _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), _dtype(k_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
        _ptr(context_lens), B, HQ, HKV, d, bs, block_tables.shape[1], nb, float(scale),
        int(max_context_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(st, "pa_paged_decode_step")


def pa_paged_prefill_attention(out, q, k_cache, v_cache, block_tables, cu_seqlens_q,
                               context_lens, scale, max_q_len, error_word, stream=None):
    """Causal varlen prefill: q/out [total_new, H_Q, d] bf16, caches
    [num_blocks, bs, H_KV, d] bf16, cu_seqlens_q [B+1] int32, context_lens [B]
    int32 (tokens including the new ones), error_word one int32 on the device."""
    if error_word is None:
        raise ValueError("error_word is required")
    _on_device(out=out, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
               cu_seqlens_q=cu_seqlens_q, context_lens=context_lens)
    _word(error_word, "error_word")
    lib = _load()
    T, HQ, d = q.shape
    nb, bs, HKV, dc = k_cache.shape
    B = context_lens.numel()
    for t, name in ((q, "q"), (out, "out"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                    (block_tables, "block_tables"), (cu_seqlens_q, "cu_seqlens_q"),
                    (context_lens, "context_lens")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out.shape != q.shape or cu_seqlens_q.numel() != B + 1 or dc != d:
        raise ValueError("shape mismatch")
    if cu_seqlens_q.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("cu_seqlens_q and context_lens must be int32")
    st = lib.pa_paged_prefill_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype(k_cache), _ptr(block_tables),
        _ptr(cu_seqlens_q), _ptr(context_lens), B, HQ, HKV, d, bs, block_tables.shape[1], nb,
        float(scale), int(max_q_len), _ptr(error_word), _stream(stream))
    _check(st, "pa_paged_prefill_attention")


def pa_selftest_bounded_wait(error_word, stream=None):
    """Diagnostic: one CTA's bounded wait on a barrier nothing completes runs
    out (2 s) and sets PA_DEVERR_WAIT_TIMEOUT (1) in error_word, a one-element
    int32 device tensor the caller cleared."""
    if error_word is None:
        raise ValueError("error_word is required")
    _word(error_word, "error_word")
    st = _load().pa_selftest_bounded_wait(_ptr(error_word), _stream(stream))
    _check(st, "pa_selftest_bounded_wait")


# ------------------------------------------------------------- MLA decode --
def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def pa_mla_absorb_q(q_latent, q_nope, q_pe, w_uk, stream=None):
    """q_latent [B, H, d_c + d_r] <- [W_UK_h q_nope[b, h] | q_pe[b, h]];
    q_nope [B, H, d_h], q_pe [B, H, d_r], w_uk [d_c, H * d_h], all bf16."""
    _on_device(q_latent=q_latent, q_nope=q_nope, q_pe=q_pe, w_uk=w_uk)
    B, H, dh = q_nope.shape
    dr = q_pe.shape[2]
    dc = w_uk.shape[0]
    for t in (q_latent, q_nope, q_pe, w_uk):
        _need(t.is_contiguous() and t.dtype == torch.bfloat16, "bf16 contiguous tensors expected")
    _need(q_latent.shape == (B, H, dc + dr) and q_pe.shape[:2] == (B, H)
          and w_uk.shape == (dc, H * dh), "shape mismatch")
    _check(_load().pa_mla_absorb_q(_ptr(q_latent), _ptr(q_nope), _ptr(q_pe), _ptr(w_uk), B, H,
                                   dh, dr, dc, _stream(stream)), "pa_mla_absorb_q")


def pa_mla_decode_workspace_size(num_seqs, num_heads, max_context_len):
    return int(_load().pa_mla_decode_workspace_size(num_seqs, num_heads, max_context_len))


def mla_decode_workspace(num_seqs, num_heads, max_context_len, device=None):
    """A zeroed device workspace for pa_mla_decode_attention (allocated by torch)."""
    n = pa_mla_decode_workspace_size(num_seqs, num_heads, max_context_len)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def pa_mla_decode_attention(out_latent, q_latent, latent_cache, block_tables, context_lens,
                            scale, max_context_len, workspace, latent_dim=512, stream=None):
    """out_latent [B, H, d_c] bf16; q_latent [B, H, d_c + d_r] bf16;
    latent_cache [num_blocks, bs, (1,) d_c + d_r] bf16; block_tables
    [B, max_blocks_per_seq] int32; context_lens [B] int32."""
    _on_device(out_latent=out_latent, q_latent=q_latent, latent_cache=latent_cache,
               block_tables=block_tables, context_lens=context_lens)
    _workspace(workspace)
    B, H, dk = q_latent.shape
    nb, bs = latent_cache.shape[0], latent_cache.shape[1]
    for t, name in ((out_latent, "out_latent"), (q_latent, "q_latent"),
                    (latent_cache, "latent_cache"), (block_tables, "block_tables"),
                    (context_lens, "context_lens")):
        _need(t.is_contiguous(), f"{name} must be contiguous")
    _need(latent_cache.shape[-1] == dk and latent_cache.numel() == nb * bs * dk,
          "latent_cache must be [num_blocks, bs, (1,) d_c + d_r]")
    _need(out_latent.shape == (B, H, latent_dim), "out_latent must be [B, H, d_c]")
    _need(q_latent.dtype == torch.bfloat16 and out_latent.dtype == torch.bfloat16
          and latent_cache.dtype == torch.bfloat16, "bf16 tensors expected")
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
          "block_tables and context_lens must be int32")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == B and context_lens.numel() == B,
          "block_tables must be [B, max_blocks_per_seq], context_lens [B]")
    st = _load().pa_mla_decode_attention(
        _ptr(out_latent), _ptr(q_latent), _ptr(latent_cache), _ptr(block_tables),
        _ptr(context_lens), B, H, latent_dim, dk - latent_dim, bs, block_tables.shape[1], nb,
        float(scale), int(max_context_len), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_mla_decode_attention")


def pa_mla_project_out(out, out_latent, w_uv, stream=None):
    """out [B, H, d_v] <- out_latent[b, h, :] W_UV_h; out_latent [B, H, d_c],
    w_uv [d_c, H * d_v], all bf16."""
    _on_device(out=out, out_latent=out_latent, w_uv=w_uv)
    B, H, dc = out_latent.shape
    dv = out.shape[2]
    for t in (out, out_latent, w_uv):
        _need(t.is_contiguous() and t.dtype == torch.bfloat16, "bf16 contiguous tensors expected")
    _need(out.shape[:2] == (B, H) and w_uv.shape == (dc, H * dv), "shape mismatch")
    _check(_load().pa_mla_project_out(_ptr(out), _ptr(out_latent), _ptr(w_uv), B, H, dc, dv,
                                      _stream(stream)), "pa_mla_project_out")
