"""GPU parity of the decode step (new-token cache write + paged decode
attention with split-K and LSE merge) against the oracle.

Tolerance (bf16 output, fp32 accumulation vs the float64 oracle):
    |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|           (the stated bar)
and, because N(0,1) workloads give small outputs, also a tight bound that
the bar would not catch:
    |gpu - oracle| <= 2^-8 * |oracle| + 2e-4 * max(1, max|oracle row|)
(bf16 rounding is <= 2^-9 relative; the rest covers fp32 accumulation).
Two GPU results compared with each other get twice the rounding term.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import bf16_codes_to_f64, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def gpu_decode_step(w, max_context_len=None, write=True, dev_cache=None):
    """Upload the workload, write the new tokens, decode.  Returns
    (out as float64 [B, H_Q, d], device error word, device caches)."""
    need_gpu()
    if dev_cache is None:
        kc, vc = to_dev(w.k_cache, "bf16"), to_dev(w.v_cache, "bf16")
    else:
        kc, vc = dev_cache
    if write:
        pa.pa_reshape_and_cache(to_dev(w.new_k, "bf16"), to_dev(w.new_v, "bf16"), kc, vc,
                                torch.from_numpy(w.slot_mapping).cuda())
    q = to_dev(w.q, "bf16")
    out = torch.full_like(q, float("nan"))
    mcl = w.max_context_len if max_context_len is None else max_context_len
    ws = pa.decode_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size, mcl)
    pa.pa_paged_decode_attention(out, q, kc, vc, torch.from_numpy(w.block_tables).cuda(),
                                 torch.from_numpy(w.context_lens).cuda(), w.scale, mcl, ws)
    torch.cuda.synchronize()
    return bf16_codes_to_f64(to_host(out, "bf16")), pa.read_device_error(ws), (kc, vc)


def oracle_write(w):
    """Apply the decode step's cache write to the host caches (in place)."""
    if w.num_seqs:
        oracle.reshape_and_cache(w.new_k, w.new_v, oracle.BF16, w.k_cache, w.v_cache, oracle.BF16,
                                 w.slot_mapping)


def oracle_rows(w, rows):
    out = {}
    for b, h in rows:
        r, lse, ps = oracle.paged_decode_row(w.q, w.k_cache, w.v_cache, w.block_tables,
                                             w.context_lens, b, h, w.scale)
        out[(b, h)] = r
    return out


def check(got_row, ref_row, what=""):
    err = np.abs(got_row - ref_row)
    assert np.isfinite(got_row).all(), what
    assert (err <= ATOL + RTOL * np.abs(ref_row)).all(), (what, err.max())
    tight = 2.0 ** -8 * np.abs(ref_row) + 2e-4 * max(1.0, np.abs(ref_row).max())
    assert (err <= tight).all(), (what, (err - tight).max(), err.max())


def check_gpu_pair(got_row, other_row, what=""):
    """Two GPU results, each rounded to bf16 once: they may differ by one
    bf16 ulp (2^-7 relative at the bottom of a binade) plus the fp32 term."""
    err = np.abs(got_row - other_row)
    assert np.isfinite(got_row).all() and np.isfinite(other_row).all(), what
    assert (err <= ATOL + RTOL * np.abs(other_row)).all(), (what, err.max())
    tight = 2.0 ** -7 * np.abs(other_row) + 2e-4 * max(1.0, np.abs(other_row).max())
    assert (err <= tight).all(), (what, (err - tight).max(), err.max())


def check_all(w, got):
    ref, _ = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                 w.scale)
    for b in range(w.num_seqs):
        for h in range(w.num_q_heads):
            check(got[b, h], ref[b, h].astype(np.float64), (b, h))
    return ref


# --------------------------------------------------------- the workloads ---
def test_tiny_decode_step():
    """B=4, context 1..64, bs=16, 64-block pool, H_Q=16, H_KV=8: every row."""
    w = wl.tiny_decode()
    got, err, _ = gpu_decode_step(w)
    assert err == 0
    oracle_write(w)
    check_all(w, got)


def test_qwen3_decode_step_full():
    """B=64, context 512..4096, bs=16, H_Q=16, H_KV=8 (G=2): every row."""
    w = wl.qwen3_decode()
    got, err, _ = gpu_decode_step(w)
    assert err == 0
    oracle_write(w)
    check_all(w, got)


@pytest.mark.slow
@pytest.mark.parametrize("bs", [16, 64])
def test_long_context_decode_sampled(bs):
    """B=8, context 32K..128K, H_Q=32, H_KV=8 (G=4), shuffled pool, split-K
    plan of the benchmark: sampled rows against the oracle, all rows finite,
    every sequence's longest and shortest head checked."""
    w = wl.long_context_decode(block_size=bs)
    got, err, _ = gpu_decode_step(w)
    assert err == 0
    splits, tps = pa.pa_paged_decode_plan(w.num_seqs, w.num_kv_heads, w.max_context_len)
    assert splits > 1  # the split + merge path is the one exercised
    assert np.isfinite(got).all()
    oracle_write(w)
    rng = np.random.default_rng(bs)
    rows = [(b, int(rng.integers(w.num_q_heads))) for b in range(w.num_seqs)]
    rows += [(int(np.argmax(w.context_lens)), 31), (int(np.argmin(w.context_lens)), 0)]
    ref = oracle_rows(w, rows)
    for key, r in ref.items():
        check(got[key], r, key)


# ----------------------------------------------------------- edge cases ----
def test_peaked_softmax_large_outputs():
    """q scaled by 6: sharp softmax, outputs of order one, so the tolerance
    bites; ragged lengths straddle tiles and splits."""
    w = wl.make_decode("peaked", 21, 6, 1, 700, 32, 8, 128, 16, q_std=6.0,
                       context_lens=[1, 63, 64, 65, 700, 129])
    got, err, _ = gpu_decode_step(w, max_context_len=700)
    assert err == 0
    oracle_write(w)
    ref = check_all(w, got)
    assert np.abs(ref).max() > 0.5


@pytest.mark.parametrize("HQ,HKV", [(8, 8), (16, 8), (32, 8), (64, 8), (32, 2), (16, 1)])
def test_group_sizes(HQ, HKV):
    w = wl.make_decode(f"g{HQ}_{HKV}", 30 + HQ, 3, 1, 300, HQ, HKV, 128, 16, q_std=3.0)
    got, err, _ = gpu_decode_step(w)
    assert err == 0
    oracle_write(w)
    check_all(w, got)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256])
def test_block_sizes(bs):
    w = wl.make_decode(f"bs{bs}", 40 + bs, 3, 1, 600, 32, 8, 128, bs, q_std=3.0,
                       context_lens=[600, 257, 1])
    got, err, _ = gpu_decode_step(w)
    assert err == 0
    oracle_write(w)
    check_all(w, got)


def test_single_token_context_is_exact():
    """L = 1: the softmax weight is 1, the output is that token's value."""
    w = wl.make_decode("one", 5, 5, 1, 1, 16, 8, 128, 16, context_lens=[1] * 5)
    got, err, _ = gpu_decode_step(w)
    assert err == 0
    G = 2
    for b in range(5):
        for h in range(16):
            assert (got[b, h] == bf16_codes_to_f64(w.new_v[b, h // G])).all()


def test_empty_context_rows_are_zero():
    w = wl.make_decode("empty", 6, 4, 1, 80, 16, 8, 128, 16, context_lens=[0, 80, 0, 3])
    for mcl in (80, 4096):  # one split and several splits
        got, err, _ = gpu_decode_step(w, max_context_len=mcl)
        assert err == 0
        assert (got[0] == 0).all() and (got[2] == 0).all()
    oracle_write(w)
    check_all(w, got)


def test_invariance_block_permutation_and_split_count():
    """Same logical KV: a second physical permutation gives identical bits
    (splits are in logical-token space); a different split count stays
    within tolerance; block size 16 vs 64 stays within tolerance."""
    w1 = wl.make_decode("inv", 50, 4, 900, 2000, 32, 8, 128, 16, q_std=3.0)
    got1, _, _ = gpu_decode_step(w1)
    # re-place the same logical rows under another permutation
    perm = np.random.default_rng(1).permutation(w1.num_blocks)
    w2 = wl.make_decode("inv", 50, 4, 900, 2000, 32, 8, 128, 16, q_std=3.0)
    inv_bt = np.where(w2.block_tables >= 0, perm[np.maximum(w2.block_tables, 0)], -1)
    k2 = np.empty_like(w2.k_cache)
    v2 = np.empty_like(w2.v_cache)
    k2[perm] = w2.k_cache
    v2[perm] = w2.v_cache
    w2.k_cache, w2.v_cache = k2, v2
    w2.block_tables = inv_bt.astype(np.int32)
    w2.slot_mapping = np.array([perm[s // 16] * 16 + s % 16 for s in w2.slot_mapping], np.int64)
    got2, _, _ = gpu_decode_step(w2)
    assert (got1 == got2).all()
    # more splits (the host cache gets the new tokens first)
    oracle_write(w1)
    got3, _, _ = gpu_decode_step(w1, max_context_len=131072, write=False)
    for b in range(w1.num_seqs):
        for h in range(w1.num_q_heads):
            check_gpu_pair(got3[b, h], got1[b, h], ("splits", b, h))
    # the same logical rows re-paged at block size 64
    w4 = repage(w1, 64, seed=3)
    got4, _, _ = gpu_decode_step(w4, write=False)
    for b in range(w1.num_seqs):
        for h in range(w1.num_q_heads):
            check_gpu_pair(got4[b, h], got1[b, h], ("bs64", b, h))


def repage(w, bs, seed):
    """Copy of workload w (history already written) with every sequence's
    logical rows moved into a fresh shuffled pool of block size bs."""
    import copy
    r = copy.copy(w)
    nblk = [wl.blocks_needed(L, bs) for L in w.context_lens]
    nb = sum(nblk) + 2
    perm = np.random.default_rng(seed).permutation(nb)
    HKV, d = w.num_kv_heads, w.head_size
    kc = np.full((nb, bs, HKV, d), wl.BF16_NAN, np.uint16)
    vc = np.full((nb, bs, HKV, d), wl.BF16_NAN, np.uint16)
    bt = np.full((w.num_seqs, max(nblk)), -1, np.int32)
    cur = 0
    old_bs = w.block_size
    for b, L in enumerate(w.context_lens):
        j = np.arange(L)
        rows_k = w.k_cache[w.block_tables[b, j // old_bs], j % old_bs]
        rows_v = w.v_cache[w.block_tables[b, j // old_bs], j % old_bs]
        for i in range(nblk[b]):
            blk = perm[cur]
            cur += 1
            bt[b, i] = blk
            kc[blk, :min(bs, L - i * bs)] = rows_k[i * bs:(i + 1) * bs]
            vc[blk, :min(bs, L - i * bs)] = rows_v[i * bs:(i + 1) * bs]
    r.k_cache, r.v_cache, r.block_tables = kc, vc, bt
    return r


def test_out_of_range_block_ids_drop_tokens():
    w = wl.make_decode("oob", 60, 3, 100, 300, 16, 8, 128, 16, q_std=3.0)
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 1] = w.num_blocks + 3
    w.block_tables[1, 0] = -7
    w.block_tables[2, 2] = 2**31 - 1
    # history rows only (no write: the newest row is still NaN-poisoned)
    w.context_lens = (w.context_lens - 1).astype(np.int32)
    got, err, _ = gpu_decode_step(w, write=False)
    assert err == 0
    check_all(w, got)


def test_context_longer_than_hint_is_clipped_and_flagged():
    w = wl.make_decode("clip", 70, 2, 200, 200, 16, 8, 128, 16, context_lens=[200, 150])
    got, err, _ = gpu_decode_step(w, max_context_len=64)
    assert err & pa.PA_DEVERR_CONTEXT_CLIPPED
    assert np.isfinite(got).all()


def test_graph_capture_replays():
    """The decode step (write + split + merge) captured in a CUDA graph
    replays to the same result."""
    need_gpu()
    w = wl.make_decode("graph", 80, 4, 500, 3000, 32, 8, 128, 16)
    kc, vc = to_dev(w.k_cache, "bf16"), to_dev(w.v_cache, "bf16")
    nk, nv = to_dev(w.new_k, "bf16"), to_dev(w.new_v, "bf16")
    sl = torch.from_numpy(w.slot_mapping).cuda()
    q = to_dev(w.q, "bf16")
    bt = torch.from_numpy(w.block_tables).cuda()
    cl = torch.from_numpy(w.context_lens).cuda()
    out = torch.zeros_like(q)
    ws = pa.decode_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, 128, w.max_context_len)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm up outside capture
        pa.pa_reshape_and_cache(nk, nv, kc, vc, sl)
        pa.pa_paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, w.max_context_len, ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        pa.pa_reshape_and_cache(nk, nv, kc, vc, sl)
        pa.pa_paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, w.max_context_len, ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
