"""GPU parity of decode attention over an FP8 E4M3 cache against the oracle.

The decode step writes the bf16 new tokens into the e4m3 cache with
k_scale / v_scale (pa_reshape_and_cache, bit-exact against the oracle's
write), then pa_paged_decode_attention_fp8 attends with K = code * k_scale,
V = code * v_scale.  The oracle does the same write and the same attention
in double.  Tolerance as in test_gpu_decode.py (the stated 1e-2 bar and the
tight bf16-output bound); the f16 weights add 2^-12 relative at most.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import bf16_codes_to_f64, need_gpu, to_dev, to_host
from tests.test_gpu_decode import check

pytestmark = pytest.mark.gpu


def fp8_decode_step(w, ks, vs, max_context_len=None, via_scaled_entry=True):
    need_gpu()
    kc = to_dev(w.k_cache, "e4m3")
    vc = to_dev(w.v_cache, "e4m3")
    ksd = torch.tensor([ks], dtype=torch.float32, device="cuda")
    vsd = torch.tensor([vs], dtype=torch.float32, device="cuda")
    pa.pa_reshape_and_cache(to_dev(w.new_k, "bf16"), to_dev(w.new_v, "bf16"), kc, vc,
                            torch.from_numpy(w.slot_mapping).cuda(), None, ksd, vsd)
    q = to_dev(w.q, "bf16")
    out = torch.full_like(q, float("nan"))
    mcl = w.max_context_len if max_context_len is None else max_context_len
    ws = pa.decode_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size, mcl)
    bt = torch.from_numpy(w.block_tables).cuda()
    cl = torch.from_numpy(w.context_lens).cuda()
    if via_scaled_entry:
        pa.pa_paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, mcl, ws, k_scale=ksd,
                                     v_scale=vsd)
    else:
        pa.pa_paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, mcl, ws)
    torch.cuda.synchronize()
    return (bf16_codes_to_f64(to_host(out, "bf16")), pa.read_device_error(ws),
            to_host(kc, "e4m3"), to_host(vc, "e4m3"))


def oracle_fp8(w, ks, vs, rows=None):
    """Oracle write of the new tokens (in place), then attention rows."""
    oracle.reshape_and_cache(w.new_k, w.new_v, oracle.BF16, w.k_cache, w.v_cache, oracle.E4M3,
                             w.slot_mapping, k_scale=ks, v_scale=vs)
    if rows is None:
        rows = [(b, h) for b in range(w.num_seqs) for h in range(w.num_q_heads)]
    return {r: oracle.paged_decode_row(w.q, w.k_cache, w.v_cache, w.block_tables,
                                       w.context_lens, r[0], r[1], w.scale,
                                       cache_dtype=oracle.E4M3, k_scale=ks, v_scale=vs)[0]
            for r in rows}


def test_fp8_qwen3_decode_step_full():
    """B=64, context 512..4096, G=2, e4m3 cache with scales 0.05: every row,
    and the decode step's cache write bit-exact."""
    w = wl.as_fp8_history(wl.qwen3_decode(), seed=101)
    got, err, gk, gv = fp8_decode_step(w, 0.05, 0.05)
    assert err == 0
    ref = oracle_fp8(w, 0.05, 0.05)
    assert (gk == w.k_cache).all() and (gv == w.v_cache).all()
    for key, r in ref.items():
        check(got[key], r, key)


@pytest.mark.slow
@pytest.mark.parametrize("bs", [16, 64])
def test_fp8_long_context_sampled(bs):
    """B=8, context 32K..128K, G=4, e4m3 cache, split-K: sampled rows."""
    w = wl.as_fp8_history(wl.long_context_decode(block_size=bs), seed=102)
    got, err, _, _ = fp8_decode_step(w, 0.05, 0.07)
    assert err == 0 and np.isfinite(got).all()
    rng = np.random.default_rng(bs)
    rows = [(b, int(rng.integers(w.num_q_heads))) for b in range(w.num_seqs)]
    for key, r in oracle_fp8(w, 0.05, 0.07, rows).items():
        check(got[key], r, key)


@pytest.mark.parametrize("HQ,HKV", [(8, 8), (16, 8), (32, 8), (64, 8), (32, 2)])
def test_fp8_group_sizes(HQ, HKV):
    w = wl.as_fp8_history(wl.make_decode(f"f{HQ}", 60 + HQ, 3, 1, 400, HQ, HKV, 128, 16,
                                         q_std=3.0), seed=103)
    got, err, _, _ = fp8_decode_step(w, 0.1, 0.03)
    assert err == 0
    for key, r in oracle_fp8(w, 0.1, 0.03).items():
        check(got[key], r, key)


@pytest.mark.parametrize("bs", [8, 32, 128, 256])
def test_fp8_block_sizes_ragged(bs):
    w = wl.as_fp8_history(wl.make_decode(f"fb{bs}", 70 + bs, 4, 1, 600, 32, 8, 128, bs,
                                         q_std=2.0, context_lens=[600, 65, 1, 0]), seed=104)
    got, err, _, _ = fp8_decode_step(w, 0.05, 0.05, max_context_len=4096)
    assert err == 0
    assert (got[3] == 0).all()
    for key, r in oracle_fp8(w, 0.05, 0.05).items():
        check(got[key], r, key)


def test_fp8_unit_scales_through_the_plain_entry():
    """pa_paged_decode_attention accepts an e4m3 cache with unit scales."""
    w = wl.as_fp8_history(wl.make_decode("fu", 80, 3, 50, 700, 16, 8, 128, 16, q_std=0.3),
                          seed=105)
    got, err, _, _ = fp8_decode_step(w, 1.0, 1.0, via_scaled_entry=False)
    assert err == 0
    for key, r in oracle_fp8(w, 1.0, 1.0).items():
        check(got[key], r, key)


def test_fp8_large_q_needs_the_prescale():
    """q of order 1e4 (beyond what f16 holds after the products' scaling)
    still matches: q is carried with a power-of-two prescale."""
    w = wl.as_fp8_history(wl.make_decode("fq", 81, 2, 100, 300, 16, 8, 128, 16, q_std=2e4),
                          seed=106)
    got, err, _, _ = fp8_decode_step(w, 1e-5, 0.05)
    assert err == 0
    for key, r in oracle_fp8(w, 1e-5, 0.05).items():
        check(got[key], r, key)
