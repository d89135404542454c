"""The seeded inputs follow the stated recipe (no GPU): N(0,1) values rounded
to bf16, block pools drawn by random permutation with each sequence's
blocks in logical order and never shared, NaN poison in every cache row
that holds no history (the new token's row, rows past the end, unused
blocks), 5 % skipped slots in the prefill writes, and the SWA table of the
last 4096 positions.  Full-size shapes are checked where generating them is
cheap; the generators' structure is checked at small sizes otherwise."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_309_gb300 import workloads as wl


def _vals(codes):
    return torch.from_numpy(np.ascontiguousarray(codes).view(np.int16)).view(
        torch.bfloat16).float().numpy()


def _check_decode_structure(w, pool_blocks=None):
    B, bs = w.num_seqs, w.block_size
    pool = w.k_cache.shape[0]
    need = sum(math.ceil(int(L) / bs) for L in w.context_lens)
    assert pool == (pool_blocks if pool_blocks is not None else max(1, math.ceil(1.1 * need)))
    used = []
    for b in range(B):
        L = int(w.context_lens[b])
        n = math.ceil(L / bs)
        row = w.block_tables[b]
        assert (row[:n] >= 0).all() and (row[:n] < pool).all() and (row[n:] == -1).all()
        used += [int(x) for x in row[:n]]
        for j in range(L):
            blk, off = int(row[j // bs]), j % bs
            k, v = w.k_cache[blk, off], w.v_cache[blk, off]
            if j < L - 1:   # history: finite N(0,1) values
                assert np.isfinite(_vals(k)).all() and np.isfinite(_vals(v)).all()
            else:           # the new token's row is poisoned until the step writes it
                assert (k == wl.BF16_NAN).all() and (v == wl.BF16_NAN).all()
                assert int(w.slot_mapping[b]) == blk * bs + off
        if L:               # rows past the end of the last block are poisoned
            last = int(row[n - 1])
            assert (w.k_cache[last, (L - 1) % bs:] == wl.BF16_NAN).all()
    assert len(set(used)) == len(used)                     # no block is shared
    unused = sorted(set(range(pool)) - set(used))
    assert (w.k_cache[unused] == wl.BF16_NAN).all() and (w.v_cache[unused] == wl.BF16_NAN).all()


def test_tiny_decode_full_size():
    w = wl.tiny_decode()
    assert w.name == "tiny_decode_b4_ctx1-64"
    assert w.q.shape == (4, 16, 128) and w.k_cache.shape == (64, 16, 8, 128)
    assert ((w.context_lens >= 1) & (w.context_lens <= 64)).all()
    assert w.scale == pytest.approx(1 / math.sqrt(128))
    _check_decode_structure(w, pool_blocks=64)


@pytest.mark.parametrize("bs", [16, 64])
def test_decode_generator_structure_small(bs):
    """The generator behind the Qwen3-shaped and long-context workloads, at a
    small size: contexts in range, pool = ceil(1.1 x blocks needed)."""
    w = wl.make_decode("small", 11, 6, 40, 300, 8, 2, 128, bs)
    assert ((w.context_lens >= 40) & (w.context_lens <= 300)).all()
    _check_decode_structure(w)


def test_seeded_and_deterministic():
    a, b, c = wl.tiny_decode(), wl.tiny_decode(), wl.tiny_decode(seed=7)
    assert (a.q == b.q).all() and (a.k_cache == b.k_cache).all()
    assert (a.block_tables == b.block_tables).all()
    assert not (a.q == c.q).all()


def test_values_are_standard_normal_bf16():
    x = _vals(wl.randn_bf16(torch.Generator().manual_seed(3), (1 << 20,)))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    # rounded to bf16: the low 16 bits of the fp32 pattern are zero
    assert (x.view(np.uint32) & 0xFFFF == 0).all()


@pytest.mark.parametrize("variant", ["e4m3", "bf16", "e4m3_swa"])
def test_prefill_write_full_size(variant):
    w = wl.prefill_write(variant=variant)
    N = 32768
    assert w.key.shape == (N, 8, 128) and w.value.shape == (N, 8, 128)
    assert w.block_size == 16
    s = w.slot_mapping
    assert (s == -1).sum() == round(0.05 * N)               # 5 % skipped
    kept = s[s >= 0]
    assert len(np.unique(kept)) == kept.size and kept.max() < N
    if variant == "bf16":
        assert w.cache_dtype == "bf16" and w.k_scale is None
    else:
        assert w.cache_dtype == "e4m3" and w.k_scale == w.v_scale == 0.05
    if variant == "e4m3_swa":
        W = 4096
        swa = w.swa_slot_mapping
        assert swa.size == N and w.num_blocks == W // 16
        last = s[N - W:]
        tgt = swa[last[last >= 0]]
        # the last W positions map onto distinct SWA slots; nothing else does
        assert (tgt >= 0).all() and len(np.unique(tgt)) == tgt.size and tgt.max() < W
        assert (swa >= 0).sum() == tgt.size
    else:
        assert w.swa_slot_mapping is None and w.num_blocks == N // 16


def test_mla_generator_structure_small():
    m = wl.make_mla("small", 3, 100)
    assert m.k_nope.shape == (100, 128, 128) and m.k_rope.shape == (100, 1, 64)
    assert m.c_kv.shape == (100, 512) and m.k_pe.shape == (100, 64)
    assert sorted(m.slot_mapping.tolist()) == list(range(100))  # a permutation, no skips
    assert m.block_size == 64 and m.num_blocks == 2
