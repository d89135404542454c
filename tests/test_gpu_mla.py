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
