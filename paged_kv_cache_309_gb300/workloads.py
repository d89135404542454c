"""Seeded synthetic inputs for the paged KV-cache hot path.

This module only builds inputs: random bf16 tensors, block pools, block
tables, context lengths and slot mappings.  It holds none of the kernels'
arithmetic (no cache write, no encoder, no attention) and is shared by the
CUDA-side tests, the oracle-side tests and the benchmark, so that both sides
see identical bytes.

Conventions (nano-vLLM walkthrough section 2.6; sglang cache_ops.py,
reshape_and_cache_flash docstring; PagedAttention-principle post, section
"paged attention原理"):
  * a cache is [num_blocks, block_size, H_KV, d_h];
  * slot = physical_block * block_size + row_in_block; -1 means "skip";
  * a sequence of L tokens owns ceil(L / block_size) blocks, listed in
    logical order in its block-table row; physically they are a random
    subset of the pool (random permutation).

Values are N(0, 1) drawn in float32 from ``torch.Generator().manual_seed``
and rounded to bf16; unused cache rows are poisoned with bf16 NaN (0x7FC0)
or fp8 NaN (0x7F) so that a stray read shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
_CHUNK = 1 << 25  # draw very large tensors in fixed-size pieces


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def randn_bf16(gen: torch.Generator, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) values rounded to bf16, returned as uint16 codes."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        x = torch.randn(hi - lo, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        out[lo:hi] = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out.reshape(shape)


def randperm(gen: torch.Generator, n: int) -> np.ndarray:
    return torch.randperm(n, generator=gen).numpy().astype(np.int64)


def blocks_needed(length: int, block_size: int) -> int:
    """A sequence of `length` tokens occupies ceil(length / block_size) blocks
    (PagedAttention-principle post: 68 tokens at block size 32 take 3)."""
    return -(-int(length) // int(block_size))


# --------------------------------------------------------------- decode ---
@dataclass
class DecodeWorkload:
    """One decode step of one layer: write each sequence's newest token
    (position context_lens[b] - 1) into the cache, then attend over all
    context_lens[b] tokens."""
    name: str
    q: np.ndarray             # [B, H_Q, d] bf16 codes
    k_cache: np.ndarray       # [num_blocks, bs, H_KV, d] bf16 codes (history only)
    v_cache: np.ndarray
    block_tables: np.ndarray  # [B, max_blocks_per_seq] int32, -1 past the end
    context_lens: np.ndarray  # [B] int32, including the new token
    new_k: np.ndarray         # [B, H_KV, d] bf16 codes
    new_v: np.ndarray
    slot_mapping: np.ndarray  # [B] int64, slot of each new token
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self): return self.q.shape[0]
    @property
    def num_q_heads(self): return self.q.shape[1]
    @property
    def head_size(self): return self.q.shape[2]
    @property
    def num_blocks(self): return self.k_cache.shape[0]
    @property
    def block_size(self): return self.k_cache.shape[1]
    @property
    def num_kv_heads(self): return self.k_cache.shape[2]
    @property
    def max_blocks_per_seq(self): return self.block_tables.shape[1]
    @property
    def max_context_len(self): return int(self.context_lens.max()) if self.context_lens.size else 0


def make_decode(name, seed, num_seqs, ctx_lo, ctx_hi, num_q_heads, num_kv_heads, head_size,
                block_size, pool_blocks=None, pool_factor=1.1, q_std=1.0,
                context_lens=None) -> DecodeWorkload:
    """Seeded decode-step workload.

    context_lens ~ U{ctx_lo..ctx_hi} (unless given).  The pool holds
    `pool_blocks` blocks (default: ceil(pool_factor * blocks needed)); each
    sequence draws its blocks from one random permutation of the pool.
    Cache rows holding history are N(0,1) bf16; every other row (the new
    token's row, rows past the end, unused blocks) is bf16 NaN."""
    g = _gen(seed)
    B, HQ, HKV, d, bs = num_seqs, num_q_heads, num_kv_heads, head_size, block_size
    if context_lens is None:
        context_lens = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g).numpy()
    context_lens = np.asarray(context_lens, dtype=np.int32)
    nblk = [blocks_needed(L, bs) for L in context_lens]
    need = int(sum(nblk))
    if pool_blocks is None:
        pool_blocks = max(1, math.ceil(pool_factor * need))
    assert pool_blocks >= need, "pool too small"
    mbps = max(1, max(nblk) if nblk else 1)
    perm = randperm(g, pool_blocks)
    block_tables = np.full((B, mbps), -1, dtype=np.int32)
    used = np.zeros(pool_blocks, dtype=bool)
    cur = 0
    for b in range(B):
        block_tables[b, :nblk[b]] = perm[cur:cur + nblk[b]]
        used[perm[cur:cur + nblk[b]]] = True
        cur += nblk[b]
    q = randn_bf16(g, (B, HQ, d), std=q_std)
    new_k = randn_bf16(g, (B, HKV, d))
    new_v = randn_bf16(g, (B, HKV, d))
    # history: fill used blocks with random values, unused ones with NaN
    k_cache = np.full((pool_blocks, bs, HKV, d), BF16_NAN, dtype=np.uint16)
    v_cache = np.full((pool_blocks, bs, HKV, d), BF16_NAN, dtype=np.uint16)
    used_ids = np.nonzero(used)[0]
    k_cache[used_ids] = randn_bf16(g, (used_ids.size, bs, HKV, d))
    v_cache[used_ids] = randn_bf16(g, (used_ids.size, bs, HKV, d))
    slot_mapping = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        L = int(context_lens[b])
        if L == 0:
            continue
        last_blk = int(block_tables[b, nblk[b] - 1])
        first_unused_row = (L - 1) - (nblk[b] - 1) * bs  # row of position L-1
        # poison the new token's row and everything after it in the last block
        k_cache[last_blk, first_unused_row:] = BF16_NAN
        v_cache[last_blk, first_unused_row:] = BF16_NAN
        slot_mapping[b] = last_blk * bs + first_unused_row
    return DecodeWorkload(name=name, q=q, k_cache=k_cache, v_cache=v_cache,
                          block_tables=block_tables, context_lens=context_lens, new_k=new_k,
                          new_v=new_v, slot_mapping=slot_mapping,
                          scale=1.0 / math.sqrt(d),
                          meta=dict(seed=seed, ctx_lo=ctx_lo, ctx_hi=ctx_hi, pool_blocks=pool_blocks))


def random_e4m3_codes(gen: torch.Generator, shape, exp_lo=4, exp_hi=11) -> np.ndarray:
    """Random finite e4m3 codes: random sign and mantissa, exponent field
    uniform in [exp_lo, exp_hi] (values 2^(exp_lo-7) .. 2^(exp_hi-6))."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)
    combos = 2 * 8 * (exp_hi - exp_lo + 1)  # sign x mantissa x exponent
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        c = torch.randint(0, combos, (hi - lo,), generator=gen, dtype=torch.int16).numpy()
        c = c.astype(np.uint16)
        sign, man, ex = c & 1, (c >> 1) & 7, exp_lo + (c >> 4)
        out[lo:hi] = ((sign << 7) | (ex << 3) | man).astype(np.uint8)
    return out.reshape(shape)


def as_fp8_history(w: DecodeWorkload, seed: int, k_scale=0.05, v_scale=0.05) -> DecodeWorkload:
    """The same sequences, block tables and new tokens with an e4m3 cache:
    history rows are random finite codes, every other row the e4m3 NaN code
    (0x7F).  The new tokens stay bf16; the decode step writes them with the
    scales."""
    g = _gen(seed)
    hist = w.k_cache != BF16_NAN
    kc = np.full(w.k_cache.shape, E4M3_NAN, np.uint8)
    vc = np.full(w.v_cache.shape, E4M3_NAN, np.uint8)
    kc[hist] = random_e4m3_codes(g, (int(hist.sum()),))
    vc[hist] = random_e4m3_codes(g, (int(hist.sum()),))
    w2 = DecodeWorkload(name=w.name + "_e4m3", q=w.q, k_cache=kc, v_cache=vc,
                        block_tables=w.block_tables, context_lens=w.context_lens,
                        new_k=w.new_k, new_v=w.new_v, slot_mapping=w.slot_mapping,
                        scale=w.scale, meta=dict(w.meta, k_scale=k_scale, v_scale=v_scale))
    return w2


def kv_bytes_read(w: DecodeWorkload, elt: int = 2) -> int:
    """Algorithmic bytes of one decode-attention pass: every context token's
    K and V row for every KV head, the block-table entries those tokens use,
    context_lens, q in and the output out (bf16)."""
    toks = int(w.context_lens.astype(np.int64).sum())
    blocks = sum(blocks_needed(L, w.block_size) for L in w.context_lens)
    return (toks * w.num_kv_heads * w.head_size * elt * 2 + blocks * 4 + w.num_seqs * 4
            + 2 * w.num_seqs * w.num_q_heads * w.head_size * 2)


# ---------------------------------------------------------- cache write ---
@dataclass
class WriteWorkload:
    name: str
    key: np.ndarray            # [N, H, d] bf16 codes
    value: np.ndarray
    slot_mapping: np.ndarray   # [N] int64
    swa_slot_mapping: np.ndarray | None
    num_blocks: int            # of the target cache
    block_size: int
    k_scale: float | None
    v_scale: float | None
    cache_dtype: str           # "bf16" | "e4m3"
    meta: dict = field(default_factory=dict)


def make_prefill_write(name, seed, num_tokens, num_heads, head_size, block_size,
                       skip_frac=0.05, cache_dtype="bf16", scale=None, swa_window=None):
    """Prefill cache write: slot_mapping is a random permutation of the
    pool's num_tokens slots with a random `skip_frac` of the entries set to -1.

    With swa_window=W: the target cache is a W-slot SWA pool; the second-stage
    table has one entry per first-stage slot, all -1 except the slots of the
    last W tokens, which map to a random permutation of the W SWA slots."""
    g = _gen(seed)
    N, H, d, bs = num_tokens, num_heads, head_size, block_size
    key = randn_bf16(g, (N, H, d))
    value = randn_bf16(g, (N, H, d))
    slots = randperm(g, N)
    n_skip = int(round(skip_frac * N))
    skip_pos = randperm(g, N)[:n_skip]
    slots[skip_pos] = -1
    num_slots = N
    swa = None
    if swa_window:
        W = int(swa_window)
        swa = np.full(num_slots, -1, dtype=np.int64)
        swa_perm = randperm(g, W)
        for i, p in enumerate(range(N - W, N)):
            if slots[p] >= 0:
                swa[slots[p]] = swa_perm[i]
        num_slots = W
    num_blocks = blocks_needed(num_slots, bs)
    return WriteWorkload(name=name, key=key, value=value, slot_mapping=slots,
                         swa_slot_mapping=swa, num_blocks=num_blocks, block_size=bs,
                         k_scale=scale, v_scale=scale, cache_dtype=cache_dtype,
                         meta=dict(seed=seed, skip_frac=skip_frac, swa_window=swa_window))


def write_tokens_effective(w: WriteWorkload) -> int:
    """Tokens that land in the cache (first- and second-stage skips removed)."""
    s = w.slot_mapping
    ok = s >= 0
    if w.swa_slot_mapping is not None:
        t = np.where(ok, w.swa_slot_mapping[np.where(ok, s, 0)], -1)
        ok = t >= 0
    return int(ok.sum())


def write_bytes(w: WriteWorkload, src_elt: int = 2) -> int:
    """Algorithmic bytes of one cache-write pass: the slot index of every
    token (and its SWA entry), plus K and V of every written token read and
    written at the cache's element size."""
    n = w.key.shape[0]
    row = w.key.shape[1] * w.key.shape[2]
    out_elt = 1 if w.cache_dtype == "e4m3" else 2
    written = write_tokens_effective(w)
    idx = n * 8 + (0 if w.swa_slot_mapping is None else int((w.slot_mapping >= 0).sum()) * 8)
    return idx + written * row * 2 * (src_elt + out_elt)


# ------------------------------------------------------------------ MLA ---
@dataclass
class MLAWorkload:
    name: str
    k_nope: np.ndarray        # [N, H, nope] bf16 codes
    k_rope: np.ndarray        # [N, 1, rope]
    c_kv: np.ndarray          # [N, latent] (latent cache content)
    k_pe: np.ndarray          # [N, rope]   (rope part cached beside it)
    slot_mapping: np.ndarray  # [N] int64 into the latent cache
    num_blocks: int
    block_size: int
    meta: dict = field(default_factory=dict)


def make_mla(name, seed, num_tokens, num_heads=128, nope_dim=128, rope_dim=64, latent_dim=512,
             block_size=64):
    g = _gen(seed)
    N = num_tokens
    k_nope = randn_bf16(g, (N, num_heads, nope_dim))
    k_rope = randn_bf16(g, (N, 1, rope_dim))
    c_kv = randn_bf16(g, (N, latent_dim))
    k_pe = randn_bf16(g, (N, rope_dim))
    slots = randperm(g, N)
    return MLAWorkload(name=name, k_nope=k_nope, k_rope=k_rope, c_kv=c_kv, k_pe=k_pe,
                       slot_mapping=slots, num_blocks=blocks_needed(N, block_size),
                       block_size=block_size, meta=dict(seed=seed))


# ------------------------------------------------------ named workloads ---
# The five workloads the hot path is specified on.  Sizes are the spec's; the
# seeds are 0..4 in this order.
def tiny_decode(seed=0, **kw):
    """B=4, context in [1, 64], bs=16, pool of 64 blocks, H_Q=16, H_KV=8, d=128."""
    return make_decode("tiny_decode_b4_ctx1-64", seed, 4, 1, 64, 16, 8, 128, 16,
                       pool_blocks=64, **kw)


def qwen3_decode(seed=1, **kw):
    """Qwen3-0.6B-shaped: B=64, context in [512, 4096], bs=16, H_Q=16, H_KV=8, d=128."""
    return make_decode("qwen3_0.6b_decode_b64_ctx512-4096", seed, 64, 512, 4096, 16, 8, 128, 16,
                       **kw)


def prefill_write(seed=2, variant="e4m3", num_tokens=32768, **kw):
    """32768 tokens, H_KV=8, d=128, bs=16, 5% skipped.  Variants: 'e4m3'
    (scale 0.05), 'bf16' (unscaled), 'e4m3_swa' (scale 0.05, SWA window 4096)."""
    if variant == "e4m3":
        return make_prefill_write("prefill_write_32k_e4m3", seed, num_tokens, 8, 128, 16,
                                  cache_dtype="e4m3", scale=0.05, **kw)
    if variant == "bf16":
        return make_prefill_write("prefill_write_32k_bf16", seed, num_tokens, 8, 128, 16,
                                  cache_dtype="bf16", scale=None, **kw)
    if variant == "e4m3_swa":
        return make_prefill_write("prefill_write_32k_e4m3_swa4096", seed, num_tokens, 8, 128, 16,
                                  cache_dtype="e4m3", scale=0.05, swa_window=4096, **kw)
    raise ValueError(variant)


def mla_assembly(seed=3, num_tokens=16384, **kw):
    """N=16384: k_nope [N,128,128] + k_rope [N,1,64] -> k [N,128,192];
    latent [N,512] + rope [N,64] -> paged latent cache, bs=64."""
    return make_mla("mla_k_assembly_16k", seed, num_tokens, **kw)


def long_context_decode(seed=4, block_size=16, num_seqs=8, **kw):
    """B=8, context in [32768, 131072], H_Q=32, H_KV=8, d=128, bs 16 or 64
    (num_seqs < 8 keeps the first sequences' draws: a smaller profiling case)."""
    return make_decode(f"long_context_decode_b{num_seqs}_ctx32k-128k_bs{block_size}", seed,
                       num_seqs, 32768, 131072, 32, 8, 128, block_size, **kw)


# -------------------------------------------------------------- prefill ---
@dataclass
class PrefillWorkload:
    """Causal varlen prefill over the paged cache: sequence b has L_b =
    context_lens[b] cached tokens (all K/V already written), of which the
    last n_b are new; q holds the new tokens' queries back to back."""
    name: str
    q: np.ndarray             # [total_new, H_Q, d] bf16 codes
    k_cache: np.ndarray       # [num_blocks, bs, H_KV, d]
    v_cache: np.ndarray
    block_tables: np.ndarray  # [B, max_blocks_per_seq] int32
    context_lens: np.ndarray  # [B] int32
    cu_seqlens_q: np.ndarray  # [B + 1] int32
    scale: float

    @property
    def num_seqs(self): return self.context_lens.shape[0]
    @property
    def num_q_heads(self): return self.q.shape[1]
    @property
    def num_kv_heads(self): return self.k_cache.shape[2]
    @property
    def block_size(self): return self.k_cache.shape[1]
    @property
    def max_q_len(self): return int(np.diff(self.cu_seqlens_q).max()) if self.num_seqs else 0


def make_prefill(name, seed, context_lens, new_lens, num_q_heads, num_kv_heads, head_size,
                 block_size, q_std=1.0) -> PrefillWorkload:
    """Caches hold random history for all context_lens[b] positions (a
    decode-step layout of one more token whose extra row stays NaN and is
    never read); q: N(0, q_std^2) bf16 for the new tokens."""
    ctx = np.asarray(context_lens, np.int32)
    new = np.asarray(new_lens, np.int32)
    d = make_decode(name, seed, len(ctx), 0, 0, num_q_heads, num_kv_heads, head_size, block_size,
                    context_lens=ctx + 1)
    g = _gen(seed + 7919)
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    q = randn_bf16(g, (int(cu[-1]), num_q_heads, head_size), std=q_std)
    return PrefillWorkload(name=name, q=q, k_cache=d.k_cache, v_cache=d.v_cache,
                           block_tables=d.block_tables, context_lens=ctx, cu_seqlens_q=cu,
                           scale=1.0 / math.sqrt(head_size))


def prefill_flops(w: PrefillWorkload) -> int:
    """Useful FLOPs of causal prefill: new token j of sequence b attends to
    p + 1 keys (p = L - n + j); QK and PV cost 2 d FLOPs per key each."""
    d = w.q.shape[2]
    tot = 0
    for b in range(w.num_seqs):
        L, n = int(w.context_lens[b]), int(w.cu_seqlens_q[b + 1] - w.cu_seqlens_q[b])
        keys = sum(max(L - n + j + 1, 0) for j in range(n)) if n < 4096 else \
            n * (L - n) + n * (n + 1) // 2
        tot += keys * w.num_q_heads * 4 * d
    return tot


# ----------------------------------------------------------- MLA decode ---
@dataclass
class MLADecodeWorkload:
    """One MLA decode step over a paged latent cache.

    latent_cache [num_blocks, bs, 1, d_c + d_r]: per token [c_kv | k_pe].
    q_lat [B, H, d_c + d_r]: the absorbed query, drawn directly (attention
    tests); q_nope [B, H, d_h], q_pe [B, H, d_r], w_uk [d_c, H * d_h] and
    w_uv [d_c, H * d_v] are the inputs of the absorbed chain."""
    name: str
    q_lat: np.ndarray
    latent_cache: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    q_nope: np.ndarray
    q_pe: np.ndarray
    w_uk: np.ndarray
    w_uv: np.ndarray
    latent_dim: int
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self): return self.q_lat.shape[0]
    @property
    def num_heads(self): return self.q_lat.shape[1]
    @property
    def row_dim(self): return self.q_lat.shape[2]
    @property
    def rope_dim(self): return self.row_dim - self.latent_dim
    @property
    def num_blocks(self): return self.latent_cache.shape[0]
    @property
    def block_size(self): return self.latent_cache.shape[1]
    @property
    def max_blocks_per_seq(self): return self.block_tables.shape[1]
    @property
    def max_context_len(self): return int(self.context_lens.max()) if self.context_lens.size else 0


def make_mla_decode(name, seed, num_seqs, ctx_lo, ctx_hi, num_heads, block_size=64,
                    latent_dim=512, rope_dim=64, nope_dim=128, v_head_dim=128, q_std=1.0,
                    context_lens=None, pool_factor=1.1, with_weights=True) -> MLADecodeWorkload:
    """Seeded MLA decode step.  Latent rows and queries are N(0, 1) bf16
    (latent rows as in the latent-cache write workload); W_UK ~ N(0, 1/d_h)
    and W_UV ~ N(0, 1/d_c), so the absorbed query and the output stay O(1).
    Blocks come from one random permutation of a pool sized to the
    context +10%; rows past each context and unused blocks are bf16 NaN.
    Softmax scale 1/sqrt(d_h + d_r), the unabsorbed head's width."""
    g = _gen(seed)
    B, H, bs = num_seqs, num_heads, block_size
    dk = latent_dim + rope_dim
    if context_lens is None:
        context_lens = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g).numpy()
    context_lens = np.asarray(context_lens, dtype=np.int32)
    nblk = [blocks_needed(L, bs) for L in context_lens]
    need = int(sum(nblk))
    pool = max(1, math.ceil(pool_factor * need))
    mbps = max(1, max(nblk) if nblk else 1)
    perm = randperm(g, pool)
    block_tables = np.full((B, mbps), -1, dtype=np.int32)
    used = np.zeros(pool, dtype=bool)
    cur = 0
    for b in range(B):
        block_tables[b, :nblk[b]] = perm[cur:cur + nblk[b]]
        used[perm[cur:cur + nblk[b]]] = True
        cur += nblk[b]
    q_lat = randn_bf16(g, (B, H, dk), std=q_std)
    cache = np.full((pool, bs, 1, dk), BF16_NAN, dtype=np.uint16)
    used_ids = np.nonzero(used)[0]
    cache[used_ids] = randn_bf16(g, (used_ids.size, bs, 1, dk))
    for b in range(B):
        L = int(context_lens[b])
        if L > 0 and L % bs:
            cache[int(block_tables[b, nblk[b] - 1]), L % bs:] = BF16_NAN
    if with_weights:
        q_nope = randn_bf16(g, (B, H, nope_dim))
        q_pe = randn_bf16(g, (B, H, rope_dim))
        w_uk = randn_bf16(g, (latent_dim, H * nope_dim), std=1.0 / math.sqrt(nope_dim))
        w_uv = randn_bf16(g, (latent_dim, H * v_head_dim), std=1.0 / math.sqrt(latent_dim))
    else:
        q_nope = q_pe = w_uk = w_uv = None
    return MLADecodeWorkload(name=name, q_lat=q_lat, latent_cache=cache,
                             block_tables=block_tables, context_lens=context_lens,
                             q_nope=q_nope, q_pe=q_pe, w_uk=w_uk, w_uv=w_uv,
                             latent_dim=latent_dim,
                             scale=1.0 / math.sqrt(nope_dim + rope_dim),
                             meta=dict(seed=seed, ctx_lo=ctx_lo, ctx_hi=ctx_hi, pool_blocks=pool))


def mla_decode(seed=5, num_heads=128, **kw):
    """DeepSeek-V3-shaped MLA decode step: B=64, context in [512, 4096] (the
    decode batch's length mix), H=128 heads (all heads on one GPU), latent
    512 + rope 64 per token, bs=64 (the latent-cache write's block size)."""
    return make_mla_decode(f"mla_decode_b64_ctx512-4096_h{num_heads}", seed, 64, 512, 4096,
                           num_heads, **kw)


def mla_bytes_read(w: MLADecodeWorkload, elt: int = 2) -> int:
    """Algorithmic bytes of one MLA decode attention: every context token's
    latent row once, plus q_lat in and o_lat out (bf16)."""
    tokens = int(w.context_lens.astype(np.int64).sum())
    B, H, dk = w.q_lat.shape
    return tokens * dk * elt + B * H * (dk + w.latent_dim) * 2


def mla_flops(w: MLADecodeWorkload) -> int:
    """2 * (d_c + d_r) + 2 * d_c flops per (token, head): the score and the
    weighted sum."""
    tokens = int(w.context_lens.astype(np.int64).sum())
    return tokens * w.num_heads * 2 * (w.row_dim + w.latent_dim)
