"""GPU parity of pa_paged_prefill_attention (causal varlen prefill over the
paged cache) against the oracle's causal rows.

Tolerance: the stated bar |gpu - ref| <= 1e-2 + 1e-2 |ref| on every element,
and, per row, RMS(gpu - ref) <= 2^-8 RMS(ref) + 1e-3: bf16 output rounding is
<= 2^-9 relative and the weights enter P.V rounded to bf16 (2^-9 relative
each, with independent signs across keys), fp32 accumulation adds little.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import bf16_codes_to_f64, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu


def gpu_prefill(w, max_q_len=None):
    need_gpu()
    q = to_dev(w.q, "bf16")
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_paged_prefill_attention(out, q, to_dev(w.k_cache, "bf16"), to_dev(w.v_cache, "bf16"),
                                  torch.from_numpy(w.block_tables).cuda(),
                                  torch.from_numpy(w.cu_seqlens_q).cuda(),
                                  torch.from_numpy(w.context_lens).cuda(), w.scale,
                                  w.max_q_len if max_q_len is None else max_q_len, err)
    torch.cuda.synchronize()
    return bf16_codes_to_f64(to_host(out, "bf16")), int(err.item())


def check_rows(w, got, rows):
    for (b, j, h) in rows:
        ref = oracle.paged_prefill_row(w.q, w.k_cache, w.v_cache, w.block_tables, w.cu_seqlens_q,
                                       w.context_lens, b, j, h, w.scale)[0]
        g = got[w.cu_seqlens_q[b] + j, h]
        e = np.abs(g - ref)
        assert np.isfinite(g).all(), (b, j, h)
        assert (e <= 1e-2 + 1e-2 * np.abs(ref)).all(), ((b, j, h), e.max())
        rms_e = np.sqrt((e ** 2).mean())
        assert rms_e <= 2.0 ** -8 * np.sqrt((ref ** 2).mean()) + 1e-3, ((b, j, h), rms_e)


def all_rows(w):
    return [(b, j, h) for b in range(w.num_seqs)
            for j in range(int(w.cu_seqlens_q[b + 1] - w.cu_seqlens_q[b]))
            for h in range(w.num_q_heads)]


def test_fresh_and_chunked_prefill_every_row():
    """Fresh prefills (n = L, ragged lengths) and chunked ones (a cached
    prefix, L > n), G = 4, bs = 16: every row."""
    w = wl.make_prefill("pf", 1, [200, 77, 1, 300, 64], [200, 77, 1, 37, 1], 16, 4, 128, 16,
                        q_std=2.0)
    got, err = gpu_prefill(w)
    assert err == 0
    check_rows(w, got, all_rows(w))


@pytest.mark.parametrize("HQ,HKV", [(8, 8), (16, 8), (32, 8), (64, 8), (32, 2)])
def test_group_sizes(HQ, HKV):
    w = wl.make_prefill(f"pg{HQ}", 2 + HQ, [130, 70], [130, 33], HQ, HKV, 128, 16, q_std=2.0)
    got, err = gpu_prefill(w)
    assert err == 0
    rng = np.random.default_rng(HQ)
    rows = all_rows(w)
    check_rows(w, got, [rows[i] for i in rng.choice(len(rows), 400, replace=False)])


@pytest.mark.parametrize("bs", [8, 64, 256])
def test_block_sizes(bs):
    w = wl.make_prefill(f"pb{bs}", 3 + bs, [300, 129], [300, 65], 32, 8, 128, bs, q_std=2.0)
    got, err = gpu_prefill(w)
    assert err == 0
    rng = np.random.default_rng(bs)
    rows = all_rows(w)
    check_rows(w, got, [rows[i] for i in rng.choice(len(rows), 400, replace=False)])


def test_long_prefill_sampled_and_last_row_is_decode():
    """4096-token prefill, H_Q=32, H_KV=8: sampled rows against the oracle;
    the last row of each sequence matches decode attention of the same
    context (GPU vs GPU, two bf16 roundings)."""
    w = wl.make_prefill("pl", 9, [4096, 2500], [4096, 1000], 32, 8, 128, 16)
    got, err = gpu_prefill(w)
    assert err == 0
    rng = np.random.default_rng(9)
    rows = [(0, int(j), int(h)) for j, h in zip(rng.integers(0, 4096, 40), rng.integers(0, 32, 40))]
    rows += [(1, int(j), int(h)) for j, h in zip(rng.integers(0, 1000, 40), rng.integers(0, 32, 40))]
    rows += [(0, 4095, 31), (1, 999, 0), (0, 0, 5)]
    check_rows(w, got, rows)
    # decode over the same context with the last new token's query
    qd = np.stack([w.q[w.cu_seqlens_q[b + 1] - 1] for b in range(2)])
    out = torch.empty((2, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = pa.decode_workspace(2, 32, 8, 128, 4096)
    pa.pa_paged_decode_attention(out, to_dev(qd, "bf16"), to_dev(w.k_cache, "bf16"),
                                 to_dev(w.v_cache, "bf16"), torch.from_numpy(w.block_tables).cuda(),
                                 torch.from_numpy(w.context_lens).cuda(), w.scale, 4096, ws)
    dec = bf16_codes_to_f64(to_host(out, "bf16"))
    for b in range(2):
        last = got[w.cu_seqlens_q[b + 1] - 1]
        e = np.abs(last - dec[b])
        assert (e <= 1e-2 + 1e-2 * np.abs(dec[b])).all()


def test_positions_below_zero_and_empty_sequences():
    """n > L: the first n - L new tokens have no keys (zero rows); n = 0
    sequences are skipped."""
    w = wl.make_prefill("pz", 11, [5, 50, 40], [8, 0, 40], 16, 8, 128, 16)
    got, err = gpu_prefill(w)
    assert err == 0
    assert (got[0:3] == 0).all()       # positions -3..-1
    check_rows(w, got, [(0, j, h) for j in range(3, 8) for h in (0, 7, 15)] +
               [(2, j, h) for j in (0, 17, 39) for h in (1, 14)])
