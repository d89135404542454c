"""Pins for the oracle's cache write and MLA K assembly (no GPU).

Sources: sglang cache_ops.py (reshape_and_cache_flash: "slot mapping",
"optional scale", "target layout" blocks; concat_and_cast_mha_k_kernel and
its wrapper), nano-vLLM walkthrough section 2.6 (store_kvcache_kernel and
its worked offset example), PagedAttention-principle post section
"paged attention原理" (block counts).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import workloads as wl
from tests.golden.load import load

RNG = np.random.default_rng(7)


def bf16(shape):
    return wl.randn_bf16(torch.Generator().manual_seed(int(RNG.integers(1 << 30))), shape)


def poison_cache(nb, bs, H, d, dtype=np.uint16, fill=0x7FC0):
    return np.full((nb, bs, H, d), fill, dtype=dtype)


# ------------------------------------------------------------ worked cases --
def test_walkthrough_worked_offset_example():
    """Token 5, head 3 of a [N, 8, 128] input sits at flat offsets
    5504..5631; after the write those values must appear in that token's
    slot, head 3, in order."""
    g = load("store_kvcache_worked_example.txt")
    H, d = g["num_kv_heads"], g["head_dim"]
    assert g["token"] * H * d == g["token_term"] and g["head"] * d == g["head_term"]
    N = 6
    # each input element holds its own flat offset (exact in fp32)
    key = np.arange(N * H * d, dtype=np.float32).reshape(N, H, d)
    kc = np.full((4, 4, H, d), np.nan, dtype=np.float32)
    slots = np.array([9, 3, 12, 0, 7, 13], dtype=np.int64)  # token 5 -> slot 13
    n = oracle.reshape_and_cache(key, None, oracle.FP32, kc, None, oracle.FP32, slots)
    assert n == N
    got = kc[13 // 4, 13 % 4, g["head"], :]
    assert got[0] == g["first"] and got[-1] == g["last"]
    assert (got == np.arange(g["first"], g["last"] + 1)).all()


def test_block_count_example():
    g = load("block_count_example.txt")
    assert wl.blocks_needed(g["tokens"], g["block_size"]) == g["blocks"]
    w = wl.make_decode("t", 0, 1, 68, 68, 2, 2, 8, 32, pool_blocks=5)
    assert (w.block_tables[0] >= 0).sum() == 3
    # one layer's K block is [block_size, HKV, DH]
    assert w.k_cache[0].size == 32 * 2 * 8


# ------------------------------------------------------------ index formula --
@pytest.mark.parametrize("bs", [1, 16, 64])
def test_target_index_is_block_and_offset(bs):
    """slot s lands at [s // bs, s % bs]: the same place as row s of the
    cache viewed as [num_blocks * bs, H, d] (numpy reshape)."""
    N, H, d, nb = 40, 3, 8, 64 // bs + 3
    key = bf16((N, H, d))
    val = bf16((N, H, d))
    slots = RNG.permutation(nb * bs)[:N].astype(np.int64)
    kc, vc = poison_cache(nb, bs, H, d), poison_cache(nb, bs, H, d)
    oracle.reshape_and_cache(key, val, oracle.BF16, kc, vc, oracle.BF16, slots)
    flat_k = kc.reshape(nb * bs, H, d)
    flat_v = vc.reshape(nb * bs, H, d)
    assert (flat_k[slots] == key).all() and (flat_v[slots] == val).all()
    untouched = np.setdiff1d(np.arange(nb * bs), slots)
    assert (flat_k[untouched] == 0x7FC0).all() and (flat_v[untouched] == 0x7FC0).all()


def test_padded_block_and_token_strides():
    """block_stride larger than bs*H*d, and key/value token strides larger
    than H*d, address the same logical elements (numpy strided views)."""
    N, H, d, bs, nb = 30, 2, 16, 4, 10
    big_k = bf16((N, H * d + 24))
    big_v = bf16((N, H * d + 40))
    key = big_k[:, : H * d]
    val = big_v[:, : H * d]
    slots = RNG.permutation(nb * bs)[:N].astype(np.int64)
    pad = 3 * 8
    store_k = np.full(nb * (bs * H * d + pad), 0x7FC0, np.uint16)
    store_v = np.full(nb * (bs * H * d + pad), 0x7FC0, np.uint16)
    kc = np.lib.stride_tricks.as_strided(store_k, (nb, bs, H, d),
                                         ((bs * H * d + pad) * 2, H * d * 2, d * 2, 2))
    vc = np.lib.stride_tricks.as_strided(store_v, (nb, bs, H, d),
                                         ((bs * H * d + pad) * 2, H * d * 2, d * 2, 2))
    oracle.reshape_and_cache(key, val, oracle.BF16, kc, vc, oracle.BF16, slots,
                             key_stride=H * d + 24, value_stride=H * d + 40,
                             block_stride=bs * H * d + pad, num_heads=H, head_size=d)
    for t in range(N):
        s = slots[t]
        assert (kc[s // bs, s % bs].reshape(-1) == key[t]).all()
        assert (vc[s // bs, s % bs].reshape(-1) == val[t]).all()
    # the padding between blocks is never written
    gaps = np.concatenate([store_k[(b + 1) * (bs * H * d + pad) - pad:(b + 1) * (bs * H * d + pad)]
                           for b in range(nb)])
    assert (gaps == 0x7FC0).all()


# ------------------------------------------------------------------- skips --
def test_negative_and_out_of_pool_slots_skip():
    N, H, d, bs, nb = 12, 2, 8, 4, 4
    key, val = bf16((N, H, d)), bf16((N, H, d))
    slots = np.array([0, -1, 5, -7, 15, 16, 99, 3, -1, 8, 1, 2], dtype=np.int64)
    kc, vc = poison_cache(nb, bs, H, d), poison_cache(nb, bs, H, d)
    n = oracle.reshape_and_cache(key, val, oracle.BF16, kc, vc, oracle.BF16, slots)
    ok = (slots >= 0) & (slots < nb * bs)
    assert n == ok.sum()
    flat = kc.reshape(-1, H, d)
    assert (flat[slots[ok]] == key[ok]).all()
    assert (np.delete(flat, slots[ok], axis=0) == 0x7FC0).all()


def test_swa_second_stage():
    """slot_mapping -> swa table -> target; -1 at either stage or an index
    past the table skips (the table is consulted only for s >= 0)."""
    N, H, d, bs = 10, 2, 8, 2
    key, val = bf16((N, H, d)), bf16((N, H, d))
    slots = np.array([0, 1, -1, 3, 4, 5, 6, 7, 8, 20], dtype=np.int64)
    swa = np.array([5, -1, 0, 1, 7, 2, 3, -1, 4], dtype=np.int64)  # 9 entries
    nb = 4
    kc, vc = poison_cache(nb, bs, H, d), poison_cache(nb, bs, H, d)
    n = oracle.reshape_and_cache(key, val, oracle.BF16, kc, vc, oracle.BF16, slots,
                                 swa_slot_mapping=swa)
    expect = {}
    for t, s in enumerate(slots):
        if s < 0 or s >= swa.size or swa[s] < 0 or swa[s] >= nb * bs:
            continue
        expect[swa[s]] = t
    assert n == len(expect) == 6
    flat = kc.reshape(-1, H, d)
    for tgt, t in expect.items():
        assert (flat[tgt] == key[t]).all()
    for tgt in set(range(nb * bs)) - set(expect):
        assert (flat[tgt] == 0x7FC0).all()


def test_swa_hand_worked_example():
    """Five tokens, a 5-entry SWA table and a 4-slot SWA pool (2 blocks of 2),
    resolved by hand: token 0 -> s=2 -> swa[2]=1; token 1 -> -1 (skip);
    token 2 -> s=4 -> swa[4]=2; token 3 -> s=0 -> swa[0]=-1 (skip);
    token 4 -> s=3 -> swa[3]=0.  Slot 3 is never written."""
    H, d = 1, 8
    key = bf16((5, H, d))
    slots = np.array([2, -1, 4, 0, 3], dtype=np.int64)
    swa = np.array([-1, -1, 1, 0, 2], dtype=np.int64)
    kc = poison_cache(2, 2, H, d)
    n = oracle.reshape_and_cache(key, None, oracle.BF16, kc, None, oracle.BF16, slots,
                                 swa_slot_mapping=swa)
    assert n == 3
    flat = kc.reshape(4, H, d)
    assert (flat[0] == key[4]).all() and (flat[1] == key[0]).all() and (flat[2] == key[2]).all()
    assert (flat[3] == 0x7FC0).all()


def test_duplicate_slot_refused():
    key = bf16((3, 1, 8))
    kc = poison_cache(2, 2, 1, 8)
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(key, None, oracle.BF16, kc, None, oracle.BF16,
                                 np.array([1, 2, 1], np.int64))


# ------------------------------------------------------------ scale + cast --
def test_roundtrip_unscaled_bf16_is_a_copy():
    w = wl.prefill_write(variant="bf16", num_tokens=2048)
    H, d = w.key.shape[1:]
    kc = poison_cache(w.num_blocks, w.block_size, H, d)
    vc = poison_cache(w.num_blocks, w.block_size, H, d)
    oracle.reshape_and_cache(w.key, w.value, oracle.BF16, kc, vc, oracle.BF16, w.slot_mapping)
    ok = w.slot_mapping >= 0
    assert (kc.reshape(-1, H, d)[w.slot_mapping[ok]] == w.key[ok]).all()
    assert (vc.reshape(-1, H, d)[w.slot_mapping[ok]] == w.value[ok]).all()


@pytest.mark.parametrize("scale", [0.05, 1.0, 1 / 3])
def test_scaled_e4m3_vs_library_division_and_cast(scale):
    """cache = e4m3(float32(x) / float32(scale)); division by numpy float32,
    rounding by torch's e4m3 cast (all values here stay inside +-448)."""
    N, H, d, bs = 256, 4, 32, 16
    key, val = bf16((N, H, d)), bf16((N, H, d))
    slots = RNG.permutation(N).astype(np.int64)
    kc = poison_cache(N // bs, bs, H, d, np.uint8, 0x7F)
    vc = poison_cache(N // bs, bs, H, d, np.uint8, 0x7F)
    oracle.reshape_and_cache(key, val, oracle.BF16, kc, vc, oracle.E4M3, slots,
                             k_scale=scale, v_scale=2 * scale)
    kf = torch.from_numpy(key.view(np.int16)).view(torch.bfloat16).float().numpy()
    vf = torch.from_numpy(val.view(np.int16)).view(torch.bfloat16).float().numpy()
    yk = kf / np.float32(scale)
    yv = vf / np.float32(2 * scale)
    assert np.abs(yk).max() <= 448
    ek = torch.from_numpy(yk).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ev = torch.from_numpy(yv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (kc.reshape(-1, H, d)[slots] == ek).all()
    assert (vc.reshape(-1, H, d)[slots] == ev).all()


def test_scaled_e4m3_saturates():
    key = np.array([[[1000.0, -1000.0, np.inf, 447.0, 449.0, 0.0, -0.0, 1.0]]], np.float32)
    kc = np.zeros((1, 1, 1, 8), np.uint8)
    oracle.reshape_and_cache(key, None, oracle.FP32, kc, None, oracle.E4M3,
                             np.array([0], np.int64), k_scale=1.0, v_scale=1.0)
    assert list(kc.reshape(-1)) == [0x7E, 0xFE, 0x7E, 0x7E, 0x7E, 0x00, 0x80, 0x38]


def test_scaled_bf16_vs_library():
    N, H, d = 64, 2, 16
    key = bf16((N, H, d))
    slots = np.arange(N, dtype=np.int64)
    kc = poison_cache(4, 16, H, d)
    oracle.reshape_and_cache(key, None, oracle.BF16, kc, None, oracle.BF16, slots,
                             k_scale=0.3, v_scale=0.3)
    kf = torch.from_numpy(key.view(np.int16)).view(torch.bfloat16).float().numpy()
    ref = torch.from_numpy(kf / np.float32(0.3)).to(torch.bfloat16).view(torch.int16).numpy()
    assert (kc.reshape(-1, H, d) == ref.view(np.uint16)).all()


def test_scaled_same_format_power_of_two_scales_closed_form():
    """Dividing by 2 or by 1/2 is exact, so a scaled bf16 -> bf16 write only
    moves the exponent field of a normal value (well inside the range) by one:
    code - 0x80 for K with k_scale = 2, code + 0x80 for V with v_scale = 0.5."""
    N, H, d = 48, 2, 16
    key, val = bf16((N, H, d)), bf16((N, H, d))
    for a in (key, val):  # keep exponent fields in [2, 253]
        e = (a >> 7) & 0xFF
        a[(e < 2) | (e > 253)] = 0x3F80  # 1.0
    slots = RNG.permutation(N).astype(np.int64)
    kc, vc = poison_cache(3, 16, H, d), poison_cache(3, 16, H, d)
    oracle.reshape_and_cache(key, val, oracle.BF16, kc, vc, oracle.BF16, slots, k_scale=2.0,
                             v_scale=0.5)
    assert (kc.reshape(-1, H, d)[slots] == key - 0x80).all()
    assert (vc.reshape(-1, H, d)[slots] == val + 0x80).all()


def test_fp16_and_fp32_sources():
    N, H, d = 32, 2, 8
    x = RNG.standard_normal((N, H, d)).astype(np.float32)
    slots = RNG.permutation(N).astype(np.int64)
    c32 = np.zeros((2, 16, H, d), np.float32)
    oracle.reshape_and_cache(x, None, oracle.FP32, c32, None, oracle.FP32, slots)
    assert (c32.reshape(-1, H, d)[slots] == x).all()
    c16 = np.zeros((2, 16, H, d), np.uint16)
    oracle.reshape_and_cache(x.astype(np.float16).view(np.uint16), None, oracle.FP16, c16, None,
                             oracle.FP16, slots)
    assert (c16.reshape(-1, H, d)[slots] == x.astype(np.float16).view(np.uint16)).all()
    cb = np.zeros((2, 16, H, d), np.uint16)
    oracle.reshape_and_cache(x, None, oracle.FP32, cb, None, oracle.BF16, slots)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (cb.reshape(-1, H, d)[slots] == ref).all()


# --------------------------------------------------------------- MLA concat --
def test_concat_mla_k_vs_numpy():
    N, H, nope, rope = 9, 5, 16, 8
    kn, kr = bf16((N, H, nope)), bf16((N, 1, rope))
    k = np.zeros((N, H, nope + rope), np.uint16)
    oracle.concat_mla_k(k, oracle.BF16, kn, kr, oracle.BF16)
    ref = np.concatenate([kn, np.broadcast_to(kr, (N, H, rope))], axis=-1)
    assert (k == ref).all()
    # the rope slice is identical for every head
    assert (k[:, :, nope:] == k[:, :1, nope:]).all()


def test_concat_mla_k_strided_and_cast():
    N, H, nope, rope = 7, 3, 8, 8
    big = bf16((N, H + 2, nope + 8))
    kn = big[:, 1:H + 1, :nope]             # strided view
    krb = bf16((N, 2, rope))
    kr = krb[:, :1, :]
    kbig = np.zeros((N, H + 1, nope + rope + 8), np.float32)
    k = kbig[:, :H, : nope + rope]
    oracle.concat_mla_k(k, oracle.FP32, kn, kr, oracle.BF16)
    to32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).float().numpy()
    ref = np.concatenate([to32(kn), np.broadcast_to(to32(kr), (N, H, rope))], axis=-1)
    assert (k == ref).all()
    assert (kbig[:, H:, :] == 0).all() and (kbig[:, :, nope + rope:] == 0).all()
