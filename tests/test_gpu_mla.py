"""GPU parity of pa_concat_mla_k (and the MLA latent-cache write built on it)
against the oracle: bit-exact."""
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


def concat_both(kn, kr, src, kdt, pad_heads=0, pad_tok=0):
    need_gpu()
    N, H, nope = kn.shape
    rope = kr.shape[2]
    width = nope + rope
    k_store = np.zeros((N, H + pad_heads, width + pad_tok), dtype=_NP[kdt])
    gk = to_dev(k_store, kdt)
    gk_view = gk[:, :H, :width]
    pa.pa_concat_mla_k(gk_view, to_dev(kn, src), to_dev(kr, src))
    torch.cuda.synchronize()
    got = to_host(gk, kdt)
    ref = k_store.copy()
    oracle.concat_mla_k(ref[:, :H, :width], _ORC[kdt], kn, kr, _ORC[src])
    return got, ref


def test_mla_k_assembly_16k_full():
    """k_nope [16384,128,128] + k_rope [16384,1,64] -> k [16384,128,192] (bf16)."""
    w = wl.mla_assembly()
    got, ref = concat_both(w.k_nope, w.k_rope, "bf16", "bf16")
    assert (got == ref).all()
    # the rope slice is the same for every head
    assert (got[:, :, 128:] == got[:, :1, 128:]).all()


@pytest.mark.parametrize("kdt", ["fp32", "fp16", "e4m3"])
def test_cast_targets(kdt):
    w = wl.mla_assembly(num_tokens=64)
    got, ref = concat_both(w.k_nope, w.k_rope, "bf16", kdt)
    assert codes_equal(got, ref, kdt).all()


@pytest.mark.parametrize("N,H,nope,rope", [(1, 1, 8, 8), (5, 3, 64, 16), (33, 16, 512, 64),
                                           (7, 128, 128, 64), (2, 1, 512, 64)])
def test_shapes_and_strided_output(N, H, nope, rope):
    g = torch.Generator().manual_seed(N * 7 + H)
    kn = wl.randn_bf16(g, (N, H, nope))
    kr = wl.randn_bf16(g, (N, 1, rope))
    got, ref = concat_both(kn, kr, "bf16", "bf16", pad_heads=2, pad_tok=24)
    assert (got == ref).all()


def test_fp32_source():
    rng = np.random.default_rng(2)
    kn = rng.standard_normal((9, 4, 32)).astype(np.float32)
    kr = rng.standard_normal((9, 1, 16)).astype(np.float32)
    for kdt in ("bf16", "fp32", "e4m3"):
        got, ref = concat_both(kn, kr, "fp32", kdt)
        assert codes_equal(got, ref, kdt).all()


def test_mla_latent_cache_write_16k():
    """Latent cache write: [c_kv (512) | k_pe (64)] per token, assembled with
    pa_concat_mla_k (one head), scattered K-only into [256, 64, 1, 576]."""
    need_gpu()
    w = wl.mla_assembly()
    N = w.c_kv.shape[0]
    lat = torch.empty((N, 1, 576), dtype=torch.bfloat16, device="cuda")
    pa.pa_concat_mla_k(lat, to_dev(w.c_kv.reshape(N, 1, 512), "bf16"),
                       to_dev(w.k_pe.reshape(N, 1, 64), "bf16"))
    cache = torch.full((w.num_blocks, w.block_size, 1, 576), float("nan"), dtype=torch.bfloat16,
                       device="cuda")
    pa.pa_reshape_and_cache(lat, None, cache, None, torch.from_numpy(w.slot_mapping).cuda())
    torch.cuda.synchronize()
    got = to_host(cache, "bf16")
    # oracle: the same two steps
    lat_ref = np.zeros((N, 1, 576), np.uint16)
    oracle.concat_mla_k(lat_ref, oracle.BF16, w.c_kv.reshape(N, 1, 512), w.k_pe.reshape(N, 1, 64),
                        oracle.BF16)
    ref = np.full((w.num_blocks, w.block_size, 1, 576), 0x7FC0, np.uint16)
    oracle.reshape_and_cache(lat_ref, None, oracle.BF16, ref, None, oracle.BF16, w.slot_mapping)
    assert codes_equal(got, ref, "bf16").all()
    # c_kv comes first, then the rope part
    s = int(w.slot_mapping[0])
    assert (got[s // 64, s % 64, 0, :512] == w.c_kv[0]).all()
    assert (got[s // 64, s % 64, 0, 512:] == w.k_pe[0]).all()


# ------------------------------------------- one-pass latent-cache write --
def fused_latent_write(ckv, kpe, slots, num_blocks, bs, src, cdt, scale=None, pad=0):
    """pa_concat_and_cache_mla on the GPU (sources optionally inside wider
    rows, `pad` extra elements per token) and the oracle's two steps
    (concat with one head, then the K-only cache write); cache codes of both."""
    need_gpu()
    N, dc = ckv.shape
    dr = kpe.shape[1]
    big_c = np.zeros((N, dc + pad), dtype=ckv.dtype)
    big_c[:, :dc] = ckv
    big_p = np.zeros((N, dr + pad), dtype=kpe.dtype)
    big_p[:, :dr] = kpe
    poison = {"bf16": 0x7FC0, "fp16": 0x7E00, "fp32": np.float32("nan"), "e4m3": 0x7F}[cdt]
    init = np.full((num_blocks, bs, 1, dc + dr), poison, dtype=_NP[cdt])
    cache = to_dev(init, cdt)
    sd = None if scale is None else torch.tensor([scale], dtype=torch.float32, device="cuda")
    pa.pa_concat_and_cache_mla(to_dev(big_c, src)[:, :dc], to_dev(big_p, src)[:, :dr], cache,
                               torch.from_numpy(np.asarray(slots, np.int64)).cuda(), sd)
    torch.cuda.synchronize()
    got = to_host(cache, cdt)
    lat = np.zeros((N, 1, dc + dr), dtype=_NP[src])
    oracle.concat_mla_k(lat, _ORC[src], ckv.reshape(N, 1, dc), kpe.reshape(N, 1, dr), _ORC[src])
    ref = init.copy()
    oracle.reshape_and_cache(lat, None, _ORC[src], ref, None, _ORC[cdt],
                             np.asarray(slots, np.int64), k_scale=scale, v_scale=scale)
    return got, ref


def test_concat_and_cache_mla_16k_full():
    """The latent write of the MLA workload in one pass: bit-exact against
    the oracle's concat + cache write, every byte of the cache."""
    w = wl.mla_assembly()
    got, ref = fused_latent_write(w.c_kv, w.k_pe, w.slot_mapping, w.num_blocks, w.block_size,
                                  "bf16", "bf16")
    assert codes_equal(got, ref, "bf16").all()
    s = int(w.slot_mapping[5])
    assert (got[s // 64, s % 64, 0, :512] == w.c_kv[5]).all()
    assert (got[s // 64, s % 64, 0, 512:] == w.k_pe[5]).all()


@pytest.mark.parametrize("cdt,scale", [("e4m3", 0.05), ("bf16", 0.3), ("e4m3", None),
                                       ("fp32", None)])
def test_concat_and_cache_mla_scaled_casts_and_skips(cdt, scale):
    w = wl.mla_assembly(num_tokens=300)
    slots = w.slot_mapping.copy()
    slots[::7] = -1                                   # padding tokens
    slots[3] = w.num_blocks * w.block_size + 5        # outside the pool
    got, ref = fused_latent_write(w.c_kv, w.k_pe, slots, w.num_blocks, w.block_size, "bf16", cdt,
                                  scale=scale, pad=24)
    assert codes_equal(got, ref, cdt).all()


@pytest.mark.parametrize("N,dc,dr,bs", [(1, 8, 8, 8), (37, 512, 64, 16), (64, 256, 32, 128),
                                         (9, 576, 64, 16), (20, 1024, 64, 32)])
def test_concat_and_cache_mla_shapes(N, dc, dr, bs):
    g = torch.Generator().manual_seed(N + dc)
    ckv = wl.randn_bf16(g, (N, dc))
    kpe = wl.randn_bf16(g, (N, dr))
    nb = (N + bs - 1) // bs + 1
    slots = wl.randperm(g, nb * bs)[:N].astype(np.int64)
    got, ref = fused_latent_write(ckv, kpe, slots, nb, bs, "bf16", "bf16")
    assert codes_equal(got, ref, "bf16").all()
    rng = np.random.default_rng(N)
    got, ref = fused_latent_write(rng.standard_normal((N, dc)).astype(np.float32),
                                  rng.standard_normal((N, dr)).astype(np.float32), slots, nb, bs,
                                  "fp32", "e4m3", scale=0.25)
    assert codes_equal(got, ref, "e4m3").all()
