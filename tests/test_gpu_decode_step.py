"""GPU parity of pa_paged_decode_step (new-token write + attention in one
launch) against the two-call path and the oracle.

The fused step converts the new row with the same code as the cache write
and feeds the attention the same values, so its output and caches must be
bit-identical to pa_reshape_and_cache followed by pa_paged_decode_attention;
the oracle checks use the decode tests' tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import bf16_codes_to_f64, need_gpu, to_dev, to_host
from tests.test_gpu_decode import check, oracle_write

pytestmark = pytest.mark.gpu


def run(w, fused, kind="bf16", scales=None, max_context_len=None):
    need_gpu()
    kc, vc = to_dev(w.k_cache, kind), to_dev(w.v_cache, kind)
    nk, nv = to_dev(w.new_k, "bf16"), to_dev(w.new_v, "bf16")
    sl = torch.from_numpy(w.slot_mapping).cuda()
    q = to_dev(w.q, "bf16")
    bt = torch.from_numpy(w.block_tables).cuda()
    cl = torch.from_numpy(w.context_lens).cuda()
    out = torch.full_like(q, float("nan"))
    mcl = w.max_context_len if max_context_len is None else max_context_len
    ws = pa.decode_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size, mcl)
    ks = vs = None
    if scales is not None:
        ks = torch.tensor([scales[0]], dtype=torch.float32, device="cuda")
        vs = torch.tensor([scales[1]], dtype=torch.float32, device="cuda")
    if fused:
        pa.pa_paged_decode_step(out, q, nk, nv, sl, kc, vc, bt, cl, w.scale, mcl, ws,
                                k_scale=ks, v_scale=vs)
    else:
        pa.pa_reshape_and_cache(nk, nv, kc, vc, sl, None, ks, vs)
        pa.pa_paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, mcl, ws, k_scale=ks,
                                     v_scale=vs)
    torch.cuda.synchronize()
    return (to_host(out, "bf16"), to_host(kc, kind), to_host(vc, kind),
            pa.read_device_error(ws))


def same_as_two_calls(w, kind="bf16", scales=None, max_context_len=None):
    a = run(w, True, kind, scales, max_context_len)
    b = run(w, False, kind, scales, max_context_len)
    assert (a[0] == b[0]).all(), "output differs from the two-call path"
    assert (a[1] == b[1]).all() and (a[2] == b[2]).all(), "caches differ"
    return a


@pytest.mark.parametrize("maker", ["tiny", "qwen3"])
def test_step_bf16_matches_two_calls_and_oracle(maker):
    w = wl.tiny_decode() if maker == "tiny" else wl.qwen3_decode()
    out, kc, vc, err = same_as_two_calls(w)
    assert err == 0
    oracle_write(w)
    assert (kc == w.k_cache).all() and (vc == w.v_cache).all()
    ref, _ = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                 w.scale)
    got = bf16_codes_to_f64(out)
    for b in range(w.num_seqs):
        for h in range(w.num_q_heads):
            check(got[b, h], ref[b, h].astype(np.float64), (b, h))


@pytest.mark.parametrize("bs,mcl", [(8, None), (16, 4096), (64, None), (256, 4096)])
def test_step_block_sizes_and_splits(bs, mcl):
    w = wl.make_decode(f"st{bs}", 90 + bs, 5, 1, 700, 32, 8, 128, bs, q_std=3.0,
                       context_lens=[700, 1, 64, 65, 300])
    out, _, _, err = same_as_two_calls(w, max_context_len=mcl)
    assert err == 0


@pytest.mark.parametrize("HQ,HKV", [(8, 8), (16, 8), (64, 8), (32, 2)])
def test_step_group_sizes(HQ, HKV):
    w = wl.make_decode(f"sg{HQ}", 95 + HQ, 3, 10, 500, HQ, HKV, 128, 16, q_std=2.0)
    _, _, _, err = same_as_two_calls(w)
    assert err == 0


def test_step_fp8_with_scales():
    w = wl.as_fp8_history(wl.qwen3_decode(), seed=111)
    out, kc, vc, err = same_as_two_calls(w, kind="e4m3", scales=(0.05, 0.07))
    assert err == 0
    oracle.reshape_and_cache(w.new_k, w.new_v, oracle.BF16, w.k_cache, w.v_cache, oracle.E4M3,
                             w.slot_mapping, k_scale=0.05, v_scale=0.07)
    assert (kc == w.k_cache).all() and (vc == w.v_cache).all()
    got = bf16_codes_to_f64(out)
    for b in range(0, w.num_seqs, 7):
        for h in (0, 9, 15):
            r = oracle.paged_decode_row(w.q, w.k_cache, w.v_cache, w.block_tables,
                                        w.context_lens, b, h, w.scale, cache_dtype=oracle.E4M3,
                                        k_scale=0.05, v_scale=0.07)[0]
            check(got[b, h], r, (b, h))


def test_step_skipped_and_mismatched_slots():
    """slot -1 skips the write (the row keeps its old, here NaN-free,
    content); a slot elsewhere in the pool is written but flagged."""
    w = wl.make_decode("sm", 120, 4, 100, 400, 16, 8, 128, 16)
    # give the newest rows real history values so that a skipped write is finite
    rng = np.random.default_rng(0)
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        blk = w.block_tables[b, (L - 1) // 16]
        w.k_cache[blk, (L - 1) % 16] = w.new_k[b] ^ np.uint16(1)
        w.v_cache[blk, (L - 1) % 16] = w.new_v[b] ^ np.uint16(1)
    free = np.setdiff1d(np.arange(w.num_blocks), w.block_tables[w.block_tables >= 0])
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[1] = -1
    w.slot_mapping[2] = int(free[0]) * 16 + 3        # an unused block: written, flagged
    out, kc, vc, err = same_as_two_calls(w)
    assert err & pa.PA_DEVERR_SLOT_MISMATCH
    assert (kc[free[0], 3] == w.new_k[2]).all()
    assert np.isfinite(bf16_codes_to_f64(out)).all()
