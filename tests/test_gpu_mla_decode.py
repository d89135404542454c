"""GPU parity of MLA decode over the paged latent cache against the oracle.

Three calls: pa_mla_absorb_q (q_lat = [W_UK_h q_nope | q_pe]),
pa_mla_decode_attention (one MQA over the 576-element latent rows, values =
their first 512 elements) and pa_mla_project_out (o_lat W_UV_h).  Each is
checked on its own inputs against the oracle in double.

Tolerance.  The stated bar, |gpu - oracle| <= 1e-2 + 1e-2 |oracle|, and a
bound derived from the arithmetic:
  attention: the softmax weights enter P.V rounded to bf16 (relative error
    <= 2^-8 each), which moves out[i] by at most 2^-8 sum_j p_j |v_j[i]| (the
    oracle's abs_out); the output is rounded to bf16 once (<= 2^-8 |out|);
    fp32 scores and sums add ~1e-6 relative.  So
      |gpu - oracle| <= 2^-8 |oracle| + 1.01 * 2^-8 abs_out + 1e-5.
  projections: fp32 sums of <= 512 products (<= 512 * 2^-24 relative to
    sum |x w|) and one bf16 rounding:
      |gpu - oracle| <= 2^-8 |oracle| + 1e-4 sum_k |x_k w_k| + 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import bf16_codes_to_f64, need_gpu, to_dev, to_host

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def check_attn(got, ref, abs_out, what=""):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert (err <= ATOL + RTOL * np.abs(ref)).all(), (what, err.max())
    tight = 2.0 ** -8 * np.abs(ref) + 1.01 * 2.0 ** -8 * abs_out + 1e-5
    assert (err <= tight).all(), (what, (err - tight).max(), err.max())


def gpu_mla(w, max_context_len=None, ws=None, q_lat=None, cache=None):
    """Run pa_mla_decode_attention; returns (o_lat float64 [B, H, 512],
    device error word)."""
    need_gpu()
    q = to_dev(w.q_lat if q_lat is None else q_lat, "bf16")
    c = to_dev(w.latent_cache, "bf16") if cache is None else cache
    out = torch.full((w.num_seqs, w.num_heads, w.latent_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    mcl = w.max_context_len if max_context_len is None else max_context_len
    if ws is None:
        ws = pa.mla_decode_workspace(w.num_seqs, w.num_heads, mcl)
    pa.pa_mla_decode_attention(out, q, c, torch.from_numpy(w.block_tables).cuda(),
                               torch.from_numpy(w.context_lens).cuda(), w.scale, mcl, ws)
    torch.cuda.synchronize()
    return bf16_codes_to_f64(to_host(out, "bf16")), pa.read_device_error(ws)


def oracle_rows(w, rows, q_lat=None):
    q = w.q_lat if q_lat is None else q_lat
    out = {}
    for b, h in rows:
        r, _, ab = oracle.mla_decode_row(q, w.latent_cache, w.block_tables, w.context_lens, b, h,
                                         w.scale, w.latent_dim)
        out[(b, h)] = (r, ab)
    return out


def all_rows(w):
    return [(b, h) for b in range(w.num_seqs) for h in range(w.num_heads)]


@pytest.mark.parametrize("H", [16, 32, 48, 64, 128, 256])
def test_mla_head_counts_every_row(H):
    """Head tiles of 16 (H = 16, 32, 48: tcgen05, tokens on M), 64 (H = 64:
    mma.sync) and 128 (H = 128, 256: tcgen05, heads on M); ragged contexts
    including 1 and a partial last tile."""
    w = wl.make_mla_decode(f"h{H}", 200 + H, 3, 1, 1, H, block_size=64,
                           context_lens=[1, 97, 300], with_weights=False)
    got, err = gpu_mla(w)
    assert err == 0
    for key, (r, ab) in oracle_rows(w, all_rows(w)).items():
        check_attn(got[key], r, ab, key)


@pytest.mark.parametrize("H", [16, 128])
def test_mla_two_and_three_piece_merges(H):
    """Thirty sequences of 600..700 tokens: each spans two or three chunks
    of the cost-balanced schedule, so every sequence ends in a merge of two
    or three pieces (the register-load merge of the tcgen05 kernel); rows of
    every sequence against the oracle."""
    rng = np.random.default_rng(77 + H)
    lens = [int(x) for x in rng.integers(600, 701, size=30)]
    w = wl.make_mla_decode(f"m23_{H}", 330 + H, 30, 1, 1, H, block_size=64, context_lens=lens,
                           with_weights=False)
    got, err = gpu_mla(w)
    assert err == 0
    rows = [(b, h) for b in range(30) for h in (0, H // 2 + 3, H - 1)]
    for key, (r, ab) in oracle_rows(w, rows).items():
        check_attn(got[key], r, ab, key)


@pytest.mark.parametrize("H", [16, 128])
def test_mla_many_short_sequences(H):
    """Two hundred sequences of 1..300 tokens (more than the 128 whose tile
    counts the tcgen05 kernel's schedule keeps in registers, and more
    sequences than clusters): sampled rows of every tenth sequence and the
    last one against the oracle."""
    rng = np.random.default_rng(91 + H)
    B = 200
    lens = [int(x) for x in rng.integers(1, 301, size=B)]
    w = wl.make_mla_decode(f"many_{H}", 350 + H, B, 1, 1, H, block_size=16, context_lens=lens,
                           with_weights=False)
    got, err = gpu_mla(w)
    assert err == 0
    rows = [(b, h) for b in list(range(0, B, 10)) + [B - 1] for h in (0, H - 1)]
    for key, (r, ab) in oracle_rows(w, rows).items():
        check_attn(got[key], r, ab, key)


@pytest.mark.parametrize("H", [16, 48, 64, 128])
@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128, 256])
def test_mla_block_sizes_ragged(bs, H):
    """Every block size on each kernel: many boxes per tile (bs < 64), one
    box at a row offset inside the block (bs > 64), an empty sequence, one
    token, a tile edge and a partial last tile."""
    w = wl.make_mla_decode(f"bs{bs}", 210 + bs, 5, 1, 1, H, block_size=bs,
                           context_lens=[0, 1, 64, 65, 531], with_weights=False)
    got, err = gpu_mla(w, max_context_len=600)
    assert err == 0
    assert (got[0] == 0).all()
    rows = [(b, h) for b in range(1, 5) for h in sorted({0, min(17, H - 1), H - 1})]
    for key, (r, ab) in oracle_rows(w, rows).items():
        check_attn(got[key], r, ab, key)


def test_mla_decode_workload_sampled():
    """The DeepSeek-V3-shaped step: B=64, context 512..4096, H=128, bs=64,
    split-K with the in-kernel merge; three heads of every sequence."""
    w = wl.mla_decode(with_weights=False)
    got, err = gpu_mla(w)
    assert err == 0 and np.isfinite(got).all()
    rng = np.random.default_rng(5)
    rows = [(b, int(h)) for b in range(w.num_seqs) for h in rng.choice(128, 3, replace=False)]
    for key, (r, ab) in oracle_rows(w, rows).items():
        check_attn(got[key], r, ab, key)


@pytest.mark.parametrize("H", [16, 64, 128])
def test_mla_long_context_many_splits(H):
    w = wl.make_mla_decode(f"long{H}", 230 + H, 2, 1, 1, H, block_size=64,
                           context_lens=[20000, 7777], with_weights=False)
    got, err = gpu_mla(w)
    assert err == 0
    rows = [(b, h) for b in range(2) for h in (0, H // 2 + 1, H - 1)]
    for key, (r, ab) in oracle_rows(w, rows).items():
        check_attn(got[key], r, ab, key)


def test_mla_invalid_block_ids_are_dropped():
    w = wl.make_mla_decode("holes", 240, 2, 1, 1, 16, block_size=16, context_lens=[200, 90],
                           with_weights=False)
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 3] = -1
    w.block_tables[1, 1] = w.num_blocks + 5
    got, err = gpu_mla(w)
    assert err == 0
    for key, (r, ab) in oracle_rows(w, all_rows(w)).items():
        check_attn(got[key], r, ab, key)


def test_mla_repeat_reuses_workspace_and_is_deterministic():
    """The split counters return to zero: a second call on the same
    workspace gives bit-identical output."""
    w = wl.make_mla_decode("rep", 250, 4, 1000, 3000, 128, with_weights=False)
    ws = pa.mla_decode_workspace(w.num_seqs, w.num_heads, w.max_context_len) if \
        torch.cuda.is_available() else None
    a, e1 = gpu_mla(w, ws=ws)
    b, e2 = gpu_mla(w, ws=ws)
    assert e1 == 0 and e2 == 0
    assert (a == b).all()
    assert (ws[256:].view(torch.int32)[:w.num_seqs * 2] == 0).all()


@pytest.mark.parametrize("H", [16, 128])
def test_mla_context_hint_and_clipping(H):
    """A max_context_len hint below the real lengths changes nothing (each
    CTA takes an equal share of the real tiles); a length beyond the block
    table is clipped to it and flagged."""
    # sequence 0 fills its last block: clipping to the table adds no
    # NaN-poisoned row past its context
    w = wl.make_mla_decode("clip", 260, 2, 1, 1, H, block_size=16, context_lens=[512, 300],
                           with_weights=False)
    got, err = gpu_mla(w, max_context_len=256)
    assert err == 0
    for key, (r, ab) in oracle_rows(w, [(0, 0), (0, H - 1), (1, 3)]).items():
        check_attn(got[key], r, ab, key)
    w.context_lens = w.context_lens.copy()
    w.context_lens[0] = w.max_blocks_per_seq * 16 + 40   # past the table
    got, err = gpu_mla(w)
    assert err & pa.PA_DEVERR_CONTEXT_CLIPPED
    assert np.isfinite(got).all()
    w.context_lens[0] = w.max_blocks_per_seq * 16        # what the clipped row attends to
    for key, (r, ab) in oracle_rows(w, [(0, 0), (0, H - 1)]).items():
        check_attn(got[key], r, ab, key)


def test_mla_large_scores():
    """q of order 30: scores in the hundreds, a sharp softmax."""
    w = wl.make_mla_decode("sharp", 270, 3, 50, 400, 64, q_std=30.0, with_weights=False)
    got, err = gpu_mla(w)
    assert err == 0
    for key, (r, ab) in oracle_rows(w, all_rows(w)[::5]).items():
        check_attn(got[key], r, ab, key)


# ------------------------------------------------------------ projections --
def check_proj(got, ref, absum, what=""):
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    tight = 2.0 ** -8 * np.abs(ref) + 1e-4 * absum + 1e-6
    assert (err <= tight).all(), (what, (err - tight).max(), err.max())


@pytest.mark.parametrize("B", [1, 64, 70])
def test_mla_absorb_q(B):
    w = wl.make_mla_decode("abs", 280 + B, B, 10, 20, 128, with_weights=True)
    need_gpu()
    q_lat = torch.empty((B, 128, 576), dtype=torch.bfloat16, device="cuda")
    pa.pa_mla_absorb_q(q_lat, to_dev(w.q_nope, "bf16"), to_dev(w.q_pe, "bf16"),
                       to_dev(w.w_uk, "bf16"))
    torch.cuda.synchronize()
    got = bf16_codes_to_f64(to_host(q_lat, "bf16"))
    ref = oracle.mla_absorb_q(w.q_nope, w.q_pe, w.w_uk)
    qn = bf16_codes_to_f64(w.q_nope)
    W = bf16_codes_to_f64(w.w_uk).reshape(512, 128, 128)       # [c, h, i]
    absum = np.einsum("bhi,chi->bhc", np.abs(qn), np.abs(W))
    check_proj(got[:, :, :512], ref[:, :, :512], absum, "nope part")
    assert (to_host(q_lat, "bf16")[:, :, 512:] == w.q_pe).all()  # rope part copied exactly


@pytest.mark.parametrize("B", [1, 64, 70])
def test_mla_project_out(B):
    w = wl.make_mla_decode("proj", 290 + B, B, 10, 20, 128, with_weights=True)
    need_gpu()
    o_lat = wl.randn_bf16(torch.Generator().manual_seed(B), (B, 128, 512), std=0.05)
    out = torch.empty((B, 128, 128), dtype=torch.bfloat16, device="cuda")
    pa.pa_mla_project_out(out, to_dev(o_lat, "bf16"), to_dev(w.w_uv, "bf16"))
    torch.cuda.synchronize()
    got = bf16_codes_to_f64(to_host(out, "bf16"))
    ref = oracle.mla_project_out(o_lat, w.w_uv)
    ol = bf16_codes_to_f64(o_lat)
    W = bf16_codes_to_f64(w.w_uv).reshape(512, 128, 128)       # [c, h, i]
    absum = np.einsum("bhc,chi->bhi", np.abs(ol), np.abs(W))
    check_proj(got, ref, absum)


@pytest.mark.parametrize("nope,dc,dv,H,B", [
    (64, 512, 64, 16, 5),      # absorb K = 64: both on the cp.async ring kernel
    (256, 256, 128, 32, 64),   # absorb K = 256: both on the ring kernel
    (128, 1024, 128, 16, 9),   # absorb on the TMA kernel with N = 1024; project K = 1024
    (128, 512, 128, 16, 130),  # three 64-row tiles, the last one ragged
])
def test_mla_projection_shapes(nope, dc, dv, H, B):
    """Both projections over shapes that select each kernel path (the TMA
    kernel for absorb at d_h = 128, the ring kernel otherwise), against the
    oracle."""
    w = wl.make_mla_decode("pshape", 310 + B, B, 10, 20, H, with_weights=True, nope_dim=nope,
                           latent_dim=dc, v_head_dim=dv)
    need_gpu()
    q_lat = torch.empty((B, H, dc + 64), dtype=torch.bfloat16, device="cuda")
    pa.pa_mla_absorb_q(q_lat, to_dev(w.q_nope, "bf16"), to_dev(w.q_pe, "bf16"),
                       to_dev(w.w_uk, "bf16"))
    o_lat = wl.randn_bf16(torch.Generator().manual_seed(B), (B, H, dc), std=0.05)
    out = torch.empty((B, H, dv), dtype=torch.bfloat16, device="cuda")
    pa.pa_mla_project_out(out, to_dev(o_lat, "bf16"), to_dev(w.w_uv, "bf16"))
    torch.cuda.synchronize()
    got = bf16_codes_to_f64(to_host(q_lat, "bf16"))
    ref = oracle.mla_absorb_q(w.q_nope, w.q_pe, w.w_uk)
    absum = np.einsum("bhi,chi->bhc", np.abs(bf16_codes_to_f64(w.q_nope)),
                      np.abs(bf16_codes_to_f64(w.w_uk).reshape(dc, H, nope)))
    check_proj(got[:, :, :dc], ref[:, :, :dc], absum, "absorb")
    assert (to_host(q_lat, "bf16")[:, :, dc:] == w.q_pe).all()
    got = bf16_codes_to_f64(to_host(out, "bf16"))
    ref = oracle.mla_project_out(o_lat, w.w_uv)
    absum = np.einsum("bhc,chi->bhi", np.abs(bf16_codes_to_f64(o_lat)),
                      np.abs(bf16_codes_to_f64(w.w_uv).reshape(dc, H, dv)))
    check_proj(got, ref, absum, "project")


def test_mla_chain_matches_explicit_attention():
    """absorb -> attention -> project on the GPU against the pages' own form
    of MLA decode (the oracle rebuilds each head's K = [c_kv W_UK_h | k_pe]
    and V = c_kv W_UV_h from the cached latent rows, then runs plain softmax
    attention) on sampled heads of every sequence, and against the oracle's
    absorbed chain on every row, both within the stated bar."""
    w = wl.make_mla_decode("chain", 300, 4, 100, 900, 128, with_weights=True)
    need_gpu()
    B, H = w.num_seqs, w.num_heads
    q_lat = torch.empty((B, H, 576), dtype=torch.bfloat16, device="cuda")
    pa.pa_mla_absorb_q(q_lat, to_dev(w.q_nope, "bf16"), to_dev(w.q_pe, "bf16"),
                       to_dev(w.w_uk, "bf16"))
    q_codes = to_host(q_lat, "bf16")
    o_lat_f, err = gpu_mla(w, q_lat=q_codes)
    assert err == 0
    o_lat = torch.from_numpy(
        (o_lat_f.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16).view(np.int16)
    ).cuda().view(torch.bfloat16)
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
    pa.pa_mla_project_out(out, o_lat, to_dev(w.w_uv, "bf16"))
    torch.cuda.synchronize()
    got = bf16_codes_to_f64(to_host(out, "bf16"))
    # the oracle's absorbed chain in double from the original inputs
    ql = oracle.mla_absorb_q(w.q_nope, w.q_pe, w.w_uk)
    ol = np.empty((B, H, 512))
    for b in range(B):
        for h in range(H):
            ol[b, h] = oracle.mla_decode_row(ql, w.latent_cache, w.block_tables, w.context_lens,
                                             b, h, w.scale, 512, q_dtype=oracle.FP64)[0]
    ref = oracle.mla_project_out(ol, w.w_uv, in_dtype=oracle.FP64)
    err_ = np.abs(got - ref)
    assert (err_ <= ATOL + RTOL * np.abs(ref)).all(), err_.max()
    # the pages' form: K and V rebuilt per head, no absorption
    for b in range(B):
        for h in (0, 1, 63, 64, 127):
            exp_row, _ = oracle.mla_decode_explicit_row(w.q_nope, w.q_pe, w.latent_cache, w.w_uk,
                                                        w.w_uv, w.block_tables, w.context_lens,
                                                        b, h, w.scale, 512)
            e = np.abs(got[b, h] - exp_row)
            assert (e <= ATOL + RTOL * np.abs(exp_row)).all(), (b, h, e.max())
