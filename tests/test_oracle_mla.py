"""Pins of the oracle's MLA decode (absorbed form) to things other than
itself.

PagedAttention-principle post, MLA section: only the latent c_kv is cached;
head h's K is c_kv W_UK_h (plus the rope part k_pe, shared by the heads) and
its V is c_kv W_UV_h.  The oracle computes the absorbed form instead
(q_lat = [W_UK_h q_nope | q_pe], one MQA over the latent rows, then W_UV_h).
The pins:
  * the absorbed chain equals explicit K/V reconstruction followed by plain
    per-head softmax attention (numpy, float64) -- a wrong W_UK/W_UV index,
    a dropped rope term or a wrong scale fails it;
  * the latent attention equals the already-pinned GQA oracle run with one
    KV head of width d_c + d_r (its first d_c outputs);
  * a one-token context returns that token's latent exactly;
  * invariance under a permutation of the physical blocks and under the
    block size;
  * brute force with math.exp on a tiny case;
  * abs_out bounds |out| and equals it for non-negative values.
"""
import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_309_gb300 import workloads as wl


def bf16_to_f64(codes):
    """bf16 codes -> float64 by bit placement (independent of the oracle)."""
    return (np.asarray(codes).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gather_rows(w, b):
    """Latent rows of sequence b in logical order (float64)."""
    L = int(w.context_lens[b])
    bs = w.block_size
    rows = [w.latent_cache[w.block_tables[b, j // bs], j % bs, 0] for j in range(L)]
    return bf16_to_f64(np.array(rows).reshape(L, w.row_dim))


def small(seed=11, B=2, H=3, dh=8, dr=4, dc=16, bs=4, lens=(7, 13)):
    return wl.make_mla_decode("pin", seed, B, 1, 1, H, block_size=bs, latent_dim=dc,
                              rope_dim=dr, nope_dim=dh, v_head_dim=dh, context_lens=list(lens))


def test_absorbed_chain_equals_explicit_reconstruction():
    w = small()
    dc, dr = w.latent_dim, w.rope_dim
    H, dh = w.num_heads, w.q_nope.shape[2]
    dv = w.w_uv.shape[1] // H
    q_lat = oracle.mla_absorb_q(w.q_nope, w.q_pe, w.w_uk)
    o_lat = np.empty((w.num_seqs, H, dc))
    for b in range(w.num_seqs):
        for h in range(H):
            o_lat[b, h] = oracle.mla_decode_row(q_lat, w.latent_cache, w.block_tables,
                                                w.context_lens, b, h, w.scale, dc,
                                                q_dtype=oracle.FP64)[0]
    out = oracle.mla_project_out(o_lat, w.w_uv, in_dtype=oracle.FP64)

    WUK, WUV = bf16_to_f64(w.w_uk), bf16_to_f64(w.w_uv)
    qn, qp = bf16_to_f64(w.q_nope), bf16_to_f64(w.q_pe)
    for b in range(w.num_seqs):
        R = gather_rows(w, b)
        C, KPE = R[:, :dc], R[:, dc:]
        for h in range(H):
            k = np.concatenate([C @ WUK[:, h * dh:(h + 1) * dh], KPE], axis=1)  # [L, dh + dr]
            v = C @ WUV[:, h * dv:(h + 1) * dv]                                 # [L, dv]
            q = np.concatenate([qn[b, h], qp[b, h]])
            s = float(np.float32(w.scale)) * (k @ q)  # the scale travels as float32
            p = np.exp(s - s.max())
            p /= p.sum()
            ref = p @ v
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-11, atol=1e-12)


def test_latent_attention_is_gqa_with_one_wide_kv_head():
    w = small(seed=12, B=3, H=4, dc=32, dr=8, bs=8, lens=(1, 17, 40))
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            got, lse, _ = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables,
                                                w.context_lens, b, h, w.scale, w.latent_dim)
            ref, lse_ref, _ = oracle.paged_decode_row(w.q_lat, w.latent_cache, w.latent_cache,
                                                      w.block_tables, w.context_lens, b, h,
                                                      w.scale)
            np.testing.assert_allclose(got, ref[:w.latent_dim], rtol=1e-14, atol=1e-15)
            assert abs(lse - lse_ref) <= 1e-12 * max(1.0, abs(lse_ref))


def test_one_token_returns_its_latent():
    w = small(seed=13, lens=(1, 1))
    for b in range(w.num_seqs):
        row = gather_rows(w, b)[0]
        for h in range(w.num_heads):
            got, lse, ab = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables,
                                                 w.context_lens, b, h, w.scale, w.latent_dim)
            assert (got == row[:w.latent_dim]).all()
            assert (ab == np.abs(row[:w.latent_dim])).all()
            q = bf16_to_f64(w.q_lat[b, h])
            ref = float(np.float32(w.scale)) * float(q @ row)
            assert math.isclose(lse, ref, rel_tol=1e-13, abs_tol=1e-13)


def test_empty_context():
    w = small(seed=14, lens=(0, 5))
    got, lse, ab = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables,
                                         w.context_lens, 0, 1, w.scale, w.latent_dim)
    assert (got == 0).all() and (ab == 0).all() and lse == -math.inf


def relayout(w, new_bs, seed):
    """Same logical rows, new block size and a fresh permutation of blocks."""
    rng = np.random.default_rng(seed)
    B = w.num_seqs
    nblk = [wl.blocks_needed(int(L), new_bs) for L in w.context_lens]
    pool = sum(nblk) + 3
    perm = rng.permutation(pool)
    bt = np.full((B, max(nblk)), -1, dtype=np.int32)
    cache = np.full((pool, new_bs, 1, w.row_dim), wl.BF16_NAN, dtype=np.uint16)
    cur = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[cur:cur + nblk[b]]
        cur += nblk[b]
        L = int(w.context_lens[b])
        for j in range(L):
            src = w.latent_cache[w.block_tables[b, j // w.block_size], j % w.block_size]
            cache[bt[b, j // new_bs], j % new_bs] = src
    return cache, bt


@pytest.mark.parametrize("new_bs", [1, 4, 16])
def test_block_permutation_and_size_invariance(new_bs):
    w = small(seed=15, B=2, H=2, bs=4, lens=(9, 14))
    cache, bt = relayout(w, new_bs, seed=new_bs)
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            a = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables, w.context_lens,
                                      b, h, w.scale, w.latent_dim)[0]
            c = oracle.mla_decode_row(w.q_lat, cache, bt, w.context_lens, b, h, w.scale,
                                      w.latent_dim)[0]
            assert (a == c).all()


def test_brute_force_tiny():
    """Pure-Python loops with math.exp (d_c = 4, d_r = 2, three tokens)."""
    w = small(seed=16, B=1, H=2, dh=2, dr=2, dc=4, bs=2, lens=(3,))
    rows = gather_rows(w, 0).tolist()
    for h in range(2):
        q = bf16_to_f64(w.q_lat[0, h]).tolist()
        sc = float(np.float32(w.scale))
        s = [sc * sum(qi * ri for qi, ri in zip(q, r)) for r in rows]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        ref = [sum(e[j] / tot * rows[j][i] for j in range(3)) for i in range(4)]
        got = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables, w.context_lens,
                                    0, h, w.scale, 4)[0]
        np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_abs_out_bounds_out():
    w = small(seed=17, lens=(11, 6))
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            got, _, ab = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables,
                                               w.context_lens, b, h, w.scale, w.latent_dim)
            assert (np.abs(got) <= ab * (1 + 1e-14)).all()
    # non-negative latents: the two coincide
    w.latent_cache = np.where(w.latent_cache == wl.BF16_NAN, w.latent_cache,
                              w.latent_cache & np.uint16(0x7FFF))
    got, _, ab = oracle.mla_decode_row(w.q_lat, w.latent_cache, w.block_tables, w.context_lens,
                                       1, 0, w.scale, w.latent_dim)
    np.testing.assert_allclose(got, ab, rtol=1e-14)


def test_absorb_and_project_one_hot_weights_per_head():
    """One-hot weights that differ per head: W_UK[h d_h + i, h d_h + i] = 1
    puts head h's q_nope in latent slots h d_h .. h d_h + d_h - 1 (zeros
    elsewhere); W_UV[h d_v + i, h d_v + i] = 1 makes out[b, h, i] =
    o_lat[b, h, h d_v + i]."""
    B, H, dh, dr, dc = 2, 3, 2, 2, 8
    rng = np.random.default_rng(5)
    qn = rng.standard_normal((B, H, dh))
    qp = rng.standard_normal((B, H, dr))
    w = np.zeros((dc, H * dh))
    for h in range(H):
        for i in range(dh):
            w[h * dh + i, h * dh + i] = 1.0
    q_lat = oracle.mla_absorb_q(qn, qp, w, in_dtype=oracle.FP64, w_dtype=oracle.FP64)
    for h in range(H):
        expect = np.zeros((B, dc))
        expect[:, h * dh:(h + 1) * dh] = qn[:, h]
        assert (q_lat[:, h, :dc] == expect).all() and (q_lat[:, h, dc:] == qp[:, h]).all()
    o_lat = rng.standard_normal((B, H, dc))
    out = oracle.mla_project_out(o_lat, w, in_dtype=oracle.FP64, w_dtype=oracle.FP64)
    for h in range(H):
        assert (out[:, h] == o_lat[:, h, h * dh:(h + 1) * dh]).all()


def test_absorb_and_project_identity_weights():
    """W_UK_h = [I_dh ; 0] puts q_nope in the first d_h latent slots; W_UV_h
    = [I_dv ; 0] reads the first d_v latent slots back."""
    B, H, dh, dr, dc = 2, 3, 4, 2, 8
    rng = np.random.default_rng(3)
    qn = rng.standard_normal((B, H, dh))
    qp = rng.standard_normal((B, H, dr))
    eye = np.zeros((dc, H * dh))
    for h in range(H):
        eye[:dh, h * dh:(h + 1) * dh] = np.eye(dh)
    q_lat = oracle.mla_absorb_q(qn, qp, eye, in_dtype=oracle.FP64, w_dtype=oracle.FP64)
    assert (q_lat[:, :, :dh] == qn).all() and (q_lat[:, :, dh:dc] == 0).all()
    assert (q_lat[:, :, dc:] == qp).all()
    o_lat = rng.standard_normal((B, H, dc))
    out = oracle.mla_project_out(o_lat, eye, in_dtype=oracle.FP64, w_dtype=oracle.FP64)
    assert (out == o_lat[:, :, :dh]).all()


# ---- the pages' explicit form (K and V rebuilt from the latent per head) --
def _explicit(w, b, h):
    return oracle.mla_decode_explicit_row(w.q_nope, w.q_pe, w.latent_cache, w.w_uk, w.w_uv,
                                          w.block_tables, w.context_lens, b, h, w.scale,
                                          w.latent_dim)


def _numpy_explicit(w, b, h):
    """K = [C W_UK_h | k_pe], V = C W_UV_h, softmax attention (numpy)."""
    dc, H, dh = w.latent_dim, w.num_heads, w.q_nope.shape[2]
    dv = w.w_uv.shape[1] // H
    WUK, WUV = bf16_to_f64(w.w_uk), bf16_to_f64(w.w_uv)
    R = gather_rows(w, b)
    C, KPE = R[:, :dc], R[:, dc:]
    k = np.concatenate([C @ WUK[:, h * dh:(h + 1) * dh], KPE], axis=1)
    v = C @ WUV[:, h * dv:(h + 1) * dv]
    q = np.concatenate([bf16_to_f64(w.q_nope)[b, h], bf16_to_f64(w.q_pe)[b, h]])
    s = float(np.float32(w.scale)) * (k @ q)
    p = np.exp(s - s.max())
    return (p / p.sum()) @ v, s.max() + math.log(np.exp(s - s.max()).sum())


def test_explicit_form_equals_numpy_reconstruction():
    w = small(seed=21, B=2, H=3, lens=(9, 22))
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            got, lse = _explicit(w, b, h)
            ref, rlse = _numpy_explicit(w, b, h)
            np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
            assert abs(lse - rlse) <= 1e-11 * max(1.0, abs(rlse))


def test_explicit_form_equals_absorbed_chain():
    w = small(seed=22, B=3, H=4, dh=16, dr=8, dc=32, bs=8, lens=(1, 19, 45))
    q_lat = oracle.mla_absorb_q(w.q_nope, w.q_pe, w.w_uk)
    o_lat = np.empty((w.num_seqs, w.num_heads, w.latent_dim))
    lses = np.empty((w.num_seqs, w.num_heads))
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            o_lat[b, h], lses[b, h], _ = oracle.mla_decode_row(
                q_lat, w.latent_cache, w.block_tables, w.context_lens, b, h, w.scale,
                w.latent_dim, q_dtype=oracle.FP64)
    chain = oracle.mla_project_out(o_lat, w.w_uv, in_dtype=oracle.FP64)
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            got, lse = _explicit(w, b, h)
            np.testing.assert_allclose(got, chain[b, h], rtol=1e-10, atol=1e-12)
            assert abs(lse - lses[b, h]) <= 1e-10 * max(1.0, abs(lse))


def test_explicit_one_token_is_its_projected_latent():
    # one token: softmax weight 1, so out = c_kv_0 W_UV_h (a plain product)
    w = small(seed=23, B=2, H=3, lens=(1, 1))
    dc, H = w.latent_dim, w.num_heads
    dv = w.w_uv.shape[1] // H
    WUV = bf16_to_f64(w.w_uv)
    for b in range(w.num_seqs):
        c0 = gather_rows(w, b)[0, :dc]
        for h in range(H):
            got, _ = _explicit(w, b, h)
            np.testing.assert_allclose(got, c0 @ WUV[:, h * dv:(h + 1) * dv], rtol=1e-12,
                                       atol=1e-13)


def test_explicit_empty_context_is_zero():
    w = small(seed=24, B=2, H=2, lens=(0, 5))
    got, lse = _explicit(w, 0, 1)
    assert (got == 0).all() and lse == -math.inf
