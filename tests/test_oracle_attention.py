"""Pins for the oracle's paged GQA decode attention (no GPU).

What the pages fix: the cache is read back along the block table
(nano-vLLM walkthrough section 2.6), blocks are physically scattered and the
table keeps their logical order (PagedAttention-principle post, "paged
attention原理"), and attention never stores the score matrix (same post,
decode dataflow).  What mathematics fixes: softmax rows sum to one, closed
forms for designed inputs, invariance under block permutation and block size.
Each test below is chosen so that a plausible slip (dropped scale, wrong GQA
head, wrong block index, off-by-one length) fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import workloads as wl

RNG = np.random.default_rng(11)


def f32_paged(K_logical, V_logical, bs, HKV, perm_seed=0, extra_blocks=3):
    """Place per-sequence logical [L, HKV, d] float32 K/V into a shuffled
    paged pool.  Returns (k_cache, v_cache, block_tables)."""
    B = len(K_logical)
    d = K_logical[0].shape[-1]
    nblk = [wl.blocks_needed(k.shape[0], bs) for k in K_logical]
    nb = sum(nblk) + extra_blocks
    perm = np.random.default_rng(perm_seed).permutation(nb)
    kc = np.full((nb, bs, HKV, d), np.nan, np.float32)
    vc = np.full((nb, bs, HKV, d), np.nan, np.float32)
    bt = np.full((B, max(1, max(nblk))), -1, np.int32)
    cur = 0
    for b in range(B):
        for j in range(nblk[b]):
            blk = perm[cur]
            cur += 1
            bt[b, j] = blk
            rows = K_logical[b][j * bs:(j + 1) * bs]
            kc[blk, :rows.shape[0]] = rows
            vc[blk, :rows.shape[0]] = V_logical[b][j * bs:(j + 1) * bs]
    return kc, vc, bt


def run_paged(q, kc, vc, bt, lens, scale, b, h):
    return oracle.paged_decode_row(q, kc, vc, bt, lens, b, h, scale,
                                   q_dtype=oracle.FP32, cache_dtype=oracle.FP32)


# ---------------------------------------------------------- closed forms ---
def test_rational_weights_exact():
    """Scores ln(w_j) give softmax weights w_j / sum(w): with integer w and
    integer V the output is a rational number, computed exactly."""
    d, scale = 4, 0.125
    w = [1, 2, 3, 6, 4]
    L = len(w)
    q = np.array([1.0, 0.0, 0.0, 0.0])
    K = np.zeros((L, d))
    K[:, 0] = [math.log(x) / scale for x in w]
    V = RNG.integers(-5, 6, size=(L, d)).astype(np.float64)
    out, lse, ps = oracle.dense_attention_row(q, K, V, scale)
    tot = sum(w)
    exact = [float(sum(Fraction(w[j], tot) * int(V[j, i]) for j in range(L))) for i in range(d)]
    assert np.allclose(out, exact, rtol=0, atol=1e-13)
    assert abs(lse - math.log(tot)) < 1e-13
    assert abs(ps - 1.0) < 1e-13


def test_two_tokens_three_to_one():
    # scale * q.k = (ln 3, 0) -> weights 3/4, 1/4; lse = ln 4
    q = np.array([2.0, 0.0])
    scale = 0.5
    K = np.array([[math.log(3.0), 7.0], [0.0, -3.0]])
    V = np.array([[4.0, -8.0], [8.0, 4.0]])
    out, lse, _ = oracle.dense_attention_row(q, K, V, scale)
    assert np.allclose(out, [5.0, -5.0], atol=1e-14)
    assert abs(lse - math.log(4.0)) < 1e-14


def test_single_token_returns_its_value():
    q = RNG.standard_normal(16)
    K = RNG.standard_normal((1, 16))
    V = RNG.standard_normal((1, 16))
    out, lse, ps = oracle.dense_attention_row(q, K, V, 0.3)
    assert (out == V[0]).all() and ps == 1.0
    assert abs(lse - 0.3 * float(q @ K[0])) < 1e-12


def test_constant_keys_give_mean_of_values_and_log_len():
    L, d = 37, 8
    q = RNG.standard_normal(d)
    K = np.tile(RNG.standard_normal(d), (L, 1))
    V = RNG.standard_normal((L, d))
    out, lse, _ = oracle.dense_attention_row(q, K, V, 0.7)
    assert np.allclose(out, V.mean(axis=0), atol=1e-14)
    assert abs(lse - (0.7 * float(q @ K[0]) + math.log(L))) < 1e-12


def test_weights_sum_to_one_and_unit_values():
    L, d = 200, 32
    q = RNG.standard_normal(d) * 3
    K = RNG.standard_normal((L, d))
    out, _, ps = oracle.dense_attention_row(q, K, np.ones((L, d)), 1 / math.sqrt(d))
    assert abs(ps - 1.0) < 1e-12
    assert np.allclose(out, 1.0, atol=1e-12)


def test_empty_context():
    q = RNG.standard_normal(8)
    out, lse, ps = oracle.dense_attention_row(q, np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    assert (out == 0).all() and lse == -math.inf and ps == 0.0


# --------------------------------------------------------- paged structure --
@pytest.mark.parametrize("HQ,HKV", [(16, 8), (32, 8), (8, 8), (8, 1)])
def test_gqa_head_mapping_consecutive(HQ, HKV):
    """KV head g holds the constant value g+1: query head h must read
    KV head h // (HQ/HKV)."""
    d, bs, L = 8, 4, 11
    K = [RNG.standard_normal((L, HKV, d)).astype(np.float32)]
    V = [np.broadcast_to((np.arange(HKV, dtype=np.float32) + 1)[None, :, None],
                         (L, HKV, d)).copy()]
    kc, vc, bt = f32_paged(K, V, bs, HKV)
    q = RNG.standard_normal((1, HQ, d)).astype(np.float32)
    lens = np.array([L], np.int32)
    G = HQ // HKV
    for h in range(HQ):
        out, _, _ = run_paged(q, kc, vc, bt, lens, 0.3, 0, h)
        assert np.allclose(out, h // G + 1, atol=1e-12), h


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_logical_order_and_length(bs):
    """K constant, V_j = j: the output is the mean position (L-1)/2, so a
    wrong block order, a wrong row-in-block or a wrong length shows up."""
    d, HKV = 4, 2
    lens = np.array([1, 5, 16, 33, 50], np.int32)
    K = [np.ones((L, HKV, d), np.float32) for L in lens]
    V = [np.broadcast_to(np.arange(L, dtype=np.float32)[:, None, None], (L, HKV, d)).copy()
         for L in lens]
    kc, vc, bt = f32_paged(K, V, bs, HKV, perm_seed=bs)
    q = RNG.standard_normal((len(lens), 2, d)).astype(np.float32)
    for b, L in enumerate(lens):
        out, _, _ = run_paged(q, kc, vc, bt, lens, 1.0, b, 1)
        assert np.allclose(out, (L - 1) / 2, atol=1e-12)


def _gather_dense(kc, vc, bt, L, bs, g):
    idx = np.arange(L)
    rows = bt[idx // bs].astype(np.int64) * bs + idx % bs
    flat_k = kc.reshape(-1, kc.shape[2], kc.shape[3])
    flat_v = vc.reshape(-1, vc.shape[2], vc.shape[3])
    return flat_k[rows, g].astype(np.float64), flat_v[rows, g].astype(np.float64)


def test_paged_equals_dense_on_gathered_copy():
    """numpy fancy indexing gathers the context in logical order; the paged
    row must equal the dense definition on that copy bit for bit."""
    w = wl.tiny_decode(seed=5)
    # the new token's row is still NaN-poisoned (nothing was written): zero it
    w.k_cache[w.k_cache == wl.BF16_NAN] = 0
    w.v_cache[w.v_cache == wl.BF16_NAN] = 0
    kf = oracle.decode(oracle.BF16, w.k_cache).astype(np.float32)
    vf = oracle.decode(oracle.BF16, w.v_cache).astype(np.float32)
    qf = oracle.decode(oracle.BF16, w.q)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        for h in (0, 5, w.num_q_heads - 1):
            Kd, Vd = _gather_dense(kf, vf, w.block_tables[b], L, w.block_size, h // G)
            dense = oracle.dense_attention_row(qf[b, h], Kd, Vd, np.float32(w.scale))
            paged = oracle.paged_decode_row(w.q, kf, vf, w.block_tables, w.context_lens, b, h,
                                            w.scale, cache_dtype=oracle.FP32)
            assert (dense[0] == paged[0]).all() and dense[1] == paged[1]


def test_block_permutation_and_block_size_invariance():
    """Same logical KV under two physical permutations and two block sizes:
    identical bits."""
    d, HKV, HQ = 16, 2, 4
    lens = np.array([3, 40, 64, 17], np.int32)
    K = [RNG.standard_normal((L, HKV, d)).astype(np.float32) for L in lens]
    V = [RNG.standard_normal((L, HKV, d)).astype(np.float32) for L in lens]
    q = RNG.standard_normal((4, HQ, d)).astype(np.float32)
    results = []
    for bs, seed in [(16, 1), (16, 2), (8, 3), (64, 4)]:
        kc, vc, bt = f32_paged(K, V, bs, HKV, perm_seed=seed)
        rows = [run_paged(q, kc, vc, bt, lens, 0.25, b, h)[0] for b in range(4) for h in range(HQ)]
        results.append(np.stack(rows))
    for r in results[1:]:
        assert (r == results[0]).all()


def test_tokens_past_context_are_never_read():
    """Rows past context_lens[b] hold NaN (from the paging helper); the
    output stays finite, and changing context_lens changes the output."""
    d, HKV, bs = 8, 1, 8
    L = 13
    K = [RNG.standard_normal((L, HKV, d)).astype(np.float32)]
    V = [RNG.standard_normal((L, HKV, d)).astype(np.float32)]
    kc, vc, bt = f32_paged(K, V, bs, HKV)
    q = RNG.standard_normal((1, 1, d)).astype(np.float32)
    out13 = run_paged(q, kc, vc, bt, np.array([13], np.int32), 0.5, 0, 0)[0]
    out12 = run_paged(q, kc, vc, bt, np.array([12], np.int32), 0.5, 0, 0)[0]
    assert np.isfinite(out13).all() and np.isfinite(out12).all()
    assert not np.allclose(out13, out12)
    out0, lse0, _ = run_paged(q, kc, vc, bt, np.array([0], np.int32), 0.5, 0, 0)
    assert (out0 == 0).all() and lse0 == -math.inf


def test_out_of_range_block_ids_are_left_out():
    """A block-table entry outside the pool drops that block's tokens from
    the softmax: equal to dense attention over the remaining rows."""
    d, HKV, bs, L = 8, 1, 4, 14
    K = [RNG.standard_normal((L, HKV, d)).astype(np.float32)]
    V = [RNG.standard_normal((L, HKV, d)).astype(np.float32)]
    kc, vc, bt = f32_paged(K, V, bs, HKV)
    bt = bt.copy()
    bt[0, 1] = kc.shape[0] + 5  # logical tokens 4..7 unreachable
    q = RNG.standard_normal((1, 1, d)).astype(np.float32)
    out, lse, _ = run_paged(q, kc, vc, bt, np.array([L], np.int32), 0.5, 0, 0)
    keep = [j for j in range(L) if not 4 <= j < 8]
    ref = oracle.dense_attention_row(q[0, 0].astype(np.float64),
                                     K[0][keep, 0].astype(np.float64),
                                     V[0][keep, 0].astype(np.float64), np.float32(0.5))
    assert (out == ref[0]).all() and lse == ref[1]


def test_full_and_row_entry_points_agree():
    w = wl.tiny_decode(seed=0)
    w.k_cache[w.k_cache == wl.BF16_NAN] = 0
    w.v_cache[w.v_cache == wl.BF16_NAN] = 0
    lens = np.maximum(w.context_lens - 1, 0).astype(np.int32)
    out, lse = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale)
    for b in range(w.num_seqs):
        for h in range(w.num_q_heads):
            r, l, _ = oracle.paged_decode_row(w.q, w.k_cache, w.v_cache, w.block_tables, lens,
                                              b, h, w.scale)
            assert (out[b, h] == r.astype(np.float32)).all()
            assert lse[b, h] == l or (math.isinf(l) and math.isinf(lse[b, h]))


# ------------------------------------------------- quantised (fp8) caches --
def _fp8_case(seed=3, L=(37, 100, 5), HKV=2, HQ=8, d=16, bs=8):
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    K = [rng.choice(finite, size=(n, HKV, d)) for n in L]
    V = [rng.choice(finite, size=(n, HKV, d)) for n in L]
    nblk = [wl.blocks_needed(n, bs) for n in L]
    nb = sum(nblk) + 2
    perm = rng.permutation(nb)
    kc = np.full((nb, bs, HKV, d), 0x7F, np.uint8)
    vc = np.full((nb, bs, HKV, d), 0x7F, np.uint8)
    bt = np.full((len(L), max(nblk)), -1, np.int32)
    cur = 0
    for b, n in enumerate(L):
        for j in range(nblk[b]):
            blk = perm[cur]
            cur += 1
            bt[b, j] = blk
            kc[blk, :min(bs, n - j * bs)] = K[b][j * bs:(j + 1) * bs]
            vc[blk, :min(bs, n - j * bs)] = V[b][j * bs:(j + 1) * bs]
    q = rng.standard_normal((len(L), HQ, d)).astype(np.float32)
    return q, kc, vc, bt, np.array(L, np.int32)


def test_fp8_cache_equals_decoded_fp32_cache():
    """An e4m3 cache with unit scales gives exactly the result of an fp32
    cache holding the decoded values (torch's e4m3 decode as the library)."""
    q, kc, vc, bt, lens = _fp8_case()
    k32 = torch.from_numpy(kc).view(torch.float8_e4m3fn).float().numpy()
    v32 = torch.from_numpy(vc).view(torch.float8_e4m3fn).float().numpy()
    for b in range(len(lens)):
        for h in (0, 3, 7):
            a = oracle.paged_decode_row(q, kc, vc, bt, lens, b, h, 0.01, q_dtype=oracle.FP32,
                                        cache_dtype=oracle.E4M3)
            r = oracle.paged_decode_row(q, k32, v32, bt, lens, b, h, 0.01, q_dtype=oracle.FP32,
                                        cache_dtype=oracle.FP32)
            assert (a[0] == r[0]).all() and a[1] == r[1]


def test_fp8_scales_act_on_scores_and_values():
    """k_scale multiplies every score (same as scaling the softmax scale);
    v_scale multiplies the output.  Powers of two keep both exact."""
    q, kc, vc, bt, lens = _fp8_case(seed=4)
    for b in range(len(lens)):
        for h in (1, 6):
            base = oracle.paged_decode_row(q, kc, vc, bt, lens, b, h, 0.04, q_dtype=oracle.FP32,
                                           cache_dtype=oracle.E4M3)
            ks = oracle.paged_decode_row(q, kc, vc, bt, lens, b, h, 0.01, q_dtype=oracle.FP32,
                                         cache_dtype=oracle.E4M3, k_scale=4.0)
            vs = oracle.paged_decode_row(q, kc, vc, bt, lens, b, h, 0.04, q_dtype=oracle.FP32,
                                         cache_dtype=oracle.E4M3, v_scale=0.125)
            assert np.allclose(ks[0], base[0], rtol=1e-14, atol=1e-14) and abs(ks[1] - base[1]) < 1e-12
            assert (vs[0] == base[0] * 0.125).all()


def test_fp8_constant_values_closed_form():
    """V codes all 0x38 (= 1.0) with v_scale 0.5: the output is 0.5."""
    q, kc, vc, bt, lens = _fp8_case(seed=5)
    vc[:] = 0x38
    out, _, _ = oracle.paged_decode_row(q, kc, vc, bt, lens, 1, 2, 0.05, q_dtype=oracle.FP32,
                                        cache_dtype=oracle.E4M3, k_scale=0.05, v_scale=0.5)
    assert np.allclose(out, 0.5, atol=1e-15)


# --------------------------------------------------- causal prefill rows ---
def _prefill_case(seed=8, ctx=(40, 90, 17), new=(40, 7, 17), HKV=2, HQ=4, d=16, bs=8):
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((L, HKV, d)).astype(np.float32) for L in ctx]
    V = [rng.standard_normal((L, HKV, d)).astype(np.float32) for L in ctx]
    kc, vc, bt = f32_paged(K, V, bs, HKV, perm_seed=seed)
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    q = rng.standard_normal((int(cu[-1]), HQ, d)).astype(np.float32)
    return q, kc, vc, bt, cu, np.array(ctx, np.int32), K, V


def test_prefill_last_row_is_decode():
    """The last new token sits at position L-1: its row equals decode
    attention over the whole context."""
    q, kc, vc, bt, cu, lens, _, _ = _prefill_case()
    for b in range(len(lens)):
        j = int(cu[b + 1] - cu[b]) - 1
        qd = np.zeros((len(lens), q.shape[1], q.shape[2]), np.float32)
        qd[b] = q[cu[b] + j]
        for h in range(q.shape[1]):
            a = oracle.paged_prefill_row(q, kc, vc, bt, cu, lens, b, j, h, 0.3, q_dtype=oracle.FP32,
                                         cache_dtype=oracle.FP32)
            r = run_paged(qd, kc, vc, bt, lens, 0.3, b, h)
            assert (a[0] == r[0]).all()


def test_prefill_first_token_of_fresh_sequence_sees_only_itself():
    """A fresh prefill (n = L): token 0 attends to key 0 alone -> v_0."""
    q, kc, vc, bt, cu, lens, K, V = _prefill_case()
    b = 0  # n == L == 40
    for h in range(q.shape[1]):
        out, _, ps = oracle.paged_prefill_row(q, kc, vc, bt, cu, lens, b, 0, h, 0.3,
                                              q_dtype=oracle.FP32, cache_dtype=oracle.FP32)
        assert (out == V[b][0, h // 2]).all() and ps == 1.0


def test_prefill_is_causal():
    """Changing K/V after position p leaves row p unchanged; changing a key
    at or before p changes it."""
    q, kc, vc, bt, cu, lens, K, V = _prefill_case()
    b, j = 1, 3                       # n = 7, L = 90 -> p = 86
    p = int(lens[b]) - 7 + j
    base = oracle.paged_prefill_row(q, kc, vc, bt, cu, lens, b, j, 1, 0.3, q_dtype=oracle.FP32,
                                    cache_dtype=oracle.FP32)[0]
    kc2, vc2 = kc.copy(), vc.copy()
    for t in range(p + 1, int(lens[b])):
        kc2[bt[b, t // 8], t % 8] = 5.0
        vc2[bt[b, t // 8], t % 8] = -7.0
    after = oracle.paged_prefill_row(q, kc2, vc2, bt, cu, lens, b, j, 1, 0.3,
                                     q_dtype=oracle.FP32, cache_dtype=oracle.FP32)[0]
    assert (after == base).all()
    vc2[bt[b, p // 8], p % 8] = -7.0
    changed = oracle.paged_prefill_row(q, kc2, vc2, bt, cu, lens, b, j, 1, 0.3,
                                       q_dtype=oracle.FP32, cache_dtype=oracle.FP32)[0]
    assert not np.allclose(changed, base)
