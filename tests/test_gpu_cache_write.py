"""GPU parity of pa_reshape_and_cache against the oracle: bit-exact.

Every case poison-fills both caches, runs the CUDA write and the oracle
write on the same seeded inputs, and compares every byte of the caches
(NaN codes compare equal to each other).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import codes_equal, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

_ORC = {"bf16": oracle.BF16, "fp16": oracle.FP16, "fp32": oracle.FP32, "e4m3": oracle.E4M3}
_NP = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "e4m3": np.uint8}
_POISON = {"bf16": 0x7FC0, "fp16": 0x7E00, "fp32": np.nan, "e4m3": 0x7F}


def run_both(key, value, src, slots, nb, bs, cdt, swa=None, scale=None, key_stride_pad=0,
             block_pad=0):
    """Run CUDA and oracle writes; return (gpu_k, gpu_v, ora_k, ora_v) cache codes."""
    need_gpu()
    N, H, d = key.shape
    row = H * d
    # source with optional token-stride padding
    def padded(x):
        if key_stride_pad == 0:
            return x
        big = np.zeros((N, row + key_stride_pad), dtype=x.dtype)
        big[:, :row] = x.reshape(N, row)
        return big
    kbig = padded(key)
    vbig = None if value is None else padded(value)
    # caches: [nb, bs*row + block_pad] storage viewed as [nb, bs, H, d]
    bstride = bs * row + block_pad
    ck = np.full(nb * bstride, _POISON[cdt], dtype=_NP[cdt])
    cv = np.full(nb * bstride, _POISON[cdt], dtype=_NP[cdt])
    # GPU
    kd = to_dev(kbig, src)
    vd = None if vbig is None else to_dev(vbig, src)
    kview = kd.as_strided((N, H, d), (kbig.shape[1] if key_stride_pad else row, d, 1))
    vview = None if vd is None else vd.as_strided((N, H, d), (kview.stride(0), d, 1))
    gk = to_dev(ck, cdt)
    gv = None if value is None else to_dev(cv, cdt)
    gkc = gk.as_strided((nb, bs, H, d), (bstride, row, d, 1))
    gvc = None if gv is None else gv.as_strided((nb, bs, H, d), (bstride, row, d, 1))
    sl = torch.from_numpy(slots).cuda()
    sw = None if swa is None else torch.from_numpy(swa).cuda()
    ksc = vsc = None
    if scale is not None:
        ksc = torch.tensor([scale[0]], dtype=torch.float32, device="cuda")
        vsc = torch.tensor([scale[1]], dtype=torch.float32, device="cuda")
    pa.pa_reshape_and_cache(kview, vview, gkc, gvc, sl, sw, ksc, vsc)
    torch.cuda.synchronize()
    out_k = to_host(gk, cdt)
    out_v = None if gv is None else to_host(gv, cdt)
    # oracle
    ok_ = ck.copy()
    ov_ = None if value is None else cv.copy()
    okc = np.lib.stride_tricks.as_strided(ok_, (nb, bs, H, d),
                                          tuple(x * ok_.itemsize for x in (bstride, row, d, 1)))
    ovc = None if ov_ is None else np.lib.stride_tricks.as_strided(
        ov_, (nb, bs, H, d), tuple(x * ov_.itemsize for x in (bstride, row, d, 1)))
    oracle.reshape_and_cache(kbig, vbig, _ORC[src], okc, ovc, _ORC[cdt], slots,
                             swa_slot_mapping=swa, k_scale=None if scale is None else scale[0],
                             v_scale=None if scale is None else scale[1],
                             key_stride=kbig.shape[1] if key_stride_pad else row,
                             value_stride=kbig.shape[1] if key_stride_pad else row,
                             block_stride=bstride, num_heads=H, head_size=d)
    return out_k, out_v, ok_, ov_


def assert_same(a, b, kind):
    eq = codes_equal(a, b, kind)
    if not eq.all():
        bad = np.nonzero(~eq)[0]
        raise AssertionError(f"{bad.size} mismatches, first at {bad[:5]}: gpu {a[bad[:5]]} "
                             f"oracle {b[bad[:5]]}")


# ---------------------------------------------------- the prefill workload --
@pytest.mark.parametrize("variant", ["e4m3", "bf16", "e4m3_swa"])
def test_prefill_write_32k_full(variant):
    """32768 tokens, H=8, d=128, bs=16, 5% skipped; fp8 (scale 0.05),
    bf16 (unscaled) and fp8 + SWA window 4096."""
    w = wl.prefill_write(variant=variant)
    sc = None if w.k_scale is None else (w.k_scale, w.v_scale)
    gk, gv, ok_, ov_ = run_both(w.key, w.value, "bf16", w.slot_mapping, w.num_blocks,
                                w.block_size, w.cache_dtype, swa=w.swa_slot_mapping, scale=sc)
    assert_same(gk, ok_, w.cache_dtype)
    assert_same(gv, ov_, w.cache_dtype)


# ------------------------------------------------- exhaustive rounding ----
@pytest.mark.parametrize("cdt", ["e4m3", "bf16", "fp16"])
@pytest.mark.parametrize("scale", [1.0, 0.05, 2.0 ** -4, 1.0 / 3.0])
def test_every_bf16_pattern(cdt, scale):
    """All 65536 bf16 bit patterns through the scaled cast (inf, NaN,
    subnormals, values past 448 included)."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    key = codes.reshape(512, 1, 128)
    value = codes[::-1].copy().reshape(512, 1, 128)
    slots = np.random.default_rng(3).permutation(512).astype(np.int64)
    gk, gv, ok_, ov_ = run_both(key, value, "bf16", slots, 32, 16, cdt, scale=(scale, 2 * scale))
    assert_same(gk, ok_, cdt)
    assert_same(gv, ov_, cdt)


@pytest.mark.parametrize("src,cdt", [("fp32", "e4m3"), ("fp32", "bf16"), ("fp32", "fp16"),
                                     ("fp16", "e4m3"), ("fp16", "bf16"), ("fp32", "fp32"),
                                     ("fp16", "fp16"), ("bf16", "fp32")])
def test_dtype_pairs(src, cdt):
    rng = np.random.default_rng(5)
    N, H, d = 300, 4, 64
    x = (rng.standard_normal((2, N, H, d)) * rng.choice([1e-3, 1, 50, 1e4], (2, N, H, 1)))
    x = x.astype(np.float32)
    x.reshape(-1)[:50] = [np.inf, -np.inf, np.nan, 0.0, -0.0] * 10
    if src == "fp32":
        key, value = x[0], x[1]
    elif src == "fp16":
        with np.errstate(over="ignore"):
            key, value = x[0].astype(np.float16).view(np.uint16), x[1].astype(np.float16).view(np.uint16)
    else:
        key = torch.from_numpy(x[0]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        value = torch.from_numpy(x[1]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(512)[:N].astype(np.int64)
    for sc in (None, (0.7, 3.0)):
        gk, gv, ok_, ov_ = run_both(key, value, src, slots, 32, 16, cdt, scale=sc)
        assert_same(gk, ok_, cdt)
        assert_same(gv, ov_, cdt)


# ---------------------------------------------------- layouts and skips ----
@pytest.mark.parametrize("H,d,bs", [(8, 128, 16), (1, 576, 64), (3, 64, 8), (128, 192, 4),
                                    (2, 8, 1), (1, 8, 16), (16, 1024, 2),
                                    (8, 128, 12), (2, 64, 3)])  # block sizes not powers of two
def test_shapes(H, d, bs):
    rng = np.random.default_rng(H * 1000 + d)
    N = 37
    key = wl.randn_bf16(torch.Generator().manual_seed(H + d), (N, H, d))
    value = wl.randn_bf16(torch.Generator().manual_seed(H + d + 1), (N, H, d))
    nb = (N + 11) // bs + 2
    slots = rng.permutation(nb * bs)[:N].astype(np.int64)
    slots[::7] = -1
    gk, gv, ok_, ov_ = run_both(key, value, "bf16", slots, nb, bs, "bf16")
    assert_same(gk, ok_, "bf16")
    assert_same(gv, ov_, "bf16")
    gk, gv, ok_, ov_ = run_both(key, value, "bf16", slots, nb, bs, "e4m3", scale=(0.1, 0.2))
    assert_same(gk, ok_, "e4m3")
    assert_same(gv, ov_, "e4m3")


def test_strided_source_and_padded_blocks():
    rng = np.random.default_rng(9)
    N, H, d, bs, nb = 200, 8, 128, 16, 20
    key = wl.randn_bf16(torch.Generator().manual_seed(1), (N, H, d))
    value = wl.randn_bf16(torch.Generator().manual_seed(2), (N, H, d))
    slots = rng.permutation(nb * bs)[:N].astype(np.int64)
    gk, gv, ok_, ov_ = run_both(key, value, "bf16", slots, nb, bs, "e4m3", scale=(0.05, 0.05),
                                key_stride_pad=3 * 1024 + 8, block_pad=64)
    assert_same(gk, ok_, "e4m3")
    assert_same(gv, ov_, "e4m3")


def test_key_only_cache():
    rng = np.random.default_rng(4)
    N, H, d, bs, nb = 100, 1, 576, 64, 3
    key = wl.randn_bf16(torch.Generator().manual_seed(3), (N, H, d))
    slots = rng.permutation(nb * bs)[:N].astype(np.int64)
    gk, gv, ok_, ov_ = run_both(key, None, "bf16", slots, nb, bs, "bf16")
    assert gv is None and ov_ is None
    assert_same(gk, ok_, "bf16")


def test_skips_and_out_of_range():
    N, H, d, bs, nb = 64, 2, 64, 4, 8
    key = wl.randn_bf16(torch.Generator().manual_seed(7), (N, H, d))
    value = wl.randn_bf16(torch.Generator().manual_seed(8), (N, H, d))
    slots = np.full(N, -1, np.int64)
    slots[:10] = [0, 5, 31, 32, 1000, -5, 7, 2**40, 12, 3]   # 32, 1000 and 2^40 are past the pool
    gk, gv, ok_, ov_ = run_both(key, value, "bf16", slots, nb, bs, "bf16")
    assert_same(gk, ok_, "bf16")
    assert_same(gv, ov_, "bf16")
    # SWA: indices past the table and -1 entries skip
    swa = np.array([3, -1, 9, 40, 0, 1, 2, 4], np.int64)
    slots2 = np.array([0, 1, 2, 3, 8, 100, -1, 4, 5, 6, 7] + [-1] * (N - 11), np.int64)
    gk, gv, ok_, ov_ = run_both(key, value, "bf16", slots2, nb, bs, "e4m3", swa=swa,
                                scale=(0.5, 0.25))
    assert_same(gk, ok_, "e4m3")
    assert_same(gv, ov_, "e4m3")


def test_all_skipped_and_empty():
    N, H, d, bs, nb = 16, 8, 128, 16, 2
    key = wl.randn_bf16(torch.Generator().manual_seed(11), (N, H, d))
    slots = np.full(N, -1, np.int64)
    gk, gv, ok_, ov_ = run_both(key, key, "bf16", slots, nb, bs, "bf16")
    assert (gk == 0x7FC0).all() and (gv == 0x7FC0).all()
    need_gpu()
    e = torch.empty((0, H, d), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((nb, bs, H, d), dtype=torch.bfloat16, device="cuda")
    pa.pa_reshape_and_cache(e, e, c, c.clone(), torch.empty(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert (c == 0).all()


def test_decode_step_write_then_read_back():
    """The decode step writes each sequence's newest token at its slot;
    reading the slot back through the block table returns the token."""
    need_gpu()
    w = wl.qwen3_decode()
    kc = to_dev(w.k_cache, "bf16")
    vc = to_dev(w.v_cache, "bf16")
    pa.pa_reshape_and_cache(to_dev(w.new_k, "bf16"), to_dev(w.new_v, "bf16"), kc, vc,
                            torch.from_numpy(w.slot_mapping).cuda())
    torch.cuda.synchronize()
    gk = to_host(kc, "bf16")
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        blk = w.block_tables[b, (L - 1) // w.block_size]
        assert (gk[blk, (L - 1) % w.block_size] == w.new_k[b]).all()


def test_scaled_division_is_ieee_over_fp32_domain():
    """fp32 -> fp32 writes isolate the scale division: random fp32 bit
    patterns (every exponent, subnormals, inf, NaN) divided by scales from
    2^-40 to 2^40, bit-exact against the oracle's IEEE single division."""
    need_gpu()
    rng = np.random.default_rng(77)
    N, H, d = 256, 2, 512  # 262144 values per scale
    bits = rng.integers(0, 2**32, size=(N, H, d), dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x.reshape(-1)[:8] = [0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -3e-39, 3.4e38]
    scales = [0.05, 1.0 / 3.0, 0.7, 3.0, 2.0 ** -4, 1.0, 1e-9, 7.5e8, 2.0 ** -40, 2.0 ** 40,
              1.17549435e-38, 3.0e-30, 6.0e29]
    scales += list(np.exp2(rng.uniform(-40, 40, size=11)).astype(np.float32))
    slots = np.arange(N, dtype=np.int64)
    for s in scales:
        gk, gv, ok_, ov_ = run_both(x, x, "fp32", slots, N // 16, 16, "fp32",
                                    scale=(float(np.float32(s)), float(np.float32(s) * 3)))
        assert_same(gk, ok_, "fp32")
        assert_same(gv, ov_, "fp32")
