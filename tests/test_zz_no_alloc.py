"""The allocation-free decode entry point, pa_paged_decode_attention_static.

It exists for callers that cannot call cudaMalloc -- for example a plugin
whose host runtime owns all device memory and passes in only the tensors it
works on, or a loop that must not risk the device synchronisation an
allocation can trigger.  Instead of a caller-provided workspace it uses a
16 MiB scratch array compiled into the library.

Checked here through the C ABI: two calls in a row (different inputs, then
the first again) give the same result as pa_paged_decode_attention, within
the decode tests' tolerance, and take no device memory (neither from
torch's allocator nor from the device's free memory); a ragged batch with
an empty context, split over many CTAs, matches the CPU oracle directly; an
oversized problem is refused before any launch; the optional error word
receives the device-side error bits.
This file is collected last so that a failing run has already run the rest.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_309_gb300 import pa
from paged_kv_cache_309_gb300 import workloads as wl
from tests.gpu_util import need_gpu, to_dev

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def _inputs(seed):
    w = wl.make_decode(f"noalloc{seed}", seed, 8, 3000, 8000, 32, 8, 128, 16, q_std=3.0)
    d = dict(q=to_dev(w.q, "bf16"), k=to_dev(w.k_cache, "bf16"), v=to_dev(w.v_cache, "bf16"),
             bt=torch.from_numpy(w.block_tables).cuda(), cl=torch.from_numpy(w.context_lens).cuda())
    # the history only: the newest row is still NaN-poisoned, keep it out
    d["cl"] = (d["cl"] - 1).to(torch.int32)
    return w, d


def _with_workspace(w, d):
    out = torch.empty_like(d["q"])
    ws = pa.decode_workspace(w.num_seqs, w.num_q_heads, w.num_kv_heads, 128, w.max_context_len)
    pa.pa_paged_decode_attention(out, d["q"], d["k"], d["v"], d["bt"], d["cl"], w.scale,
                                 w.max_context_len, ws)
    return out


def _static(w, d, err):
    out = torch.full_like(d["q"], float("nan"))
    pa.pa_paged_decode_attention_static(out, d["q"], d["k"], d["v"], d["bt"], d["cl"], w.scale,
                                        w.max_context_len, err)
    return out


def _close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    err = np.abs(g - r)
    assert (err <= ATOL + RTOL * np.abs(r)).all(), err.max()
    assert (err <= 2.0 ** -8 * np.abs(r) + 2e-4 * max(1.0, np.abs(r).max())).all(), err.max()


def test_static_scratch_matches_workspace_call_twice():
    need_gpu()
    w1, d1 = _inputs(91)
    w2, d2 = _inputs(92)
    splits, _ = pa.pa_paged_decode_plan(w1.num_seqs, w1.num_kv_heads, w1.max_context_len)
    assert splits > 1  # the scratch really holds split partials
    ref1 = _with_workspace(w1, d1)
    ref2 = _with_workspace(w2, d2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _static(w1, d1, err)
    b = _static(w2, d2, err)   # second call in a row, other inputs
    c = _static(w1, d1, err)   # and the first problem again over the leftovers
    torch.cuda.synchronize()
    _close(a, ref1)
    _close(b, ref2)
    _close(c, ref1)
    assert int(err.item()) == 0


def test_static_calls_take_no_device_memory():
    need_gpu()
    w, d = _inputs(94)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _with_workspace(w, d)
    outs = [torch.empty_like(d["q"]) for _ in range(2)]
    pa.pa_paged_decode_attention_static(outs[0], d["q"], d["k"], d["v"], d["bt"], d["cl"],
                                        w.scale, w.max_context_len, err)  # warm-up: set-up done
    torch.cuda.synchronize()
    need = pa.pa_paged_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, 128,
                                             w.max_context_len)
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for o in outs:
        pa.pa_paged_decode_attention_static(o, d["q"], d["k"], d["v"], d["bt"], d["cl"],
                                            w.scale, w.max_context_len, err)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    # a hidden workspace allocation would take at least `need` bytes
    assert free_before - free_after < need, (free_before, free_after, need)
    for o in outs:
        _close(o, ref)
    assert int(err.item()) == 0


def test_static_ragged_batch_with_empty_context_matches_oracle():
    need_gpu()
    # history lengths 0 .. 7800: the empty sequence's CTAs all exit early,
    # the others spread over many splits that share the scratch counters
    lens = [1, 5001, 138, 7801, 2601, 2, 6401, 3101]
    w = wl.make_decode("noalloc_ragged", 95, 8, 0, 0, 32, 8, 128, 16, q_std=3.0,
                       context_lens=lens)
    hist = (w.context_lens - 1).astype(np.int32)
    splits, _ = pa.pa_paged_decode_plan(8, 8, int(hist.max()))
    assert splits > 8
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((8, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):  # the second call runs over the first one's leftovers
        pa.pa_paged_decode_attention_static(
            out, to_dev(w.q, "bf16"), to_dev(w.k_cache, "bf16"), to_dev(w.v_cache, "bf16"),
            torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(hist).cuda(), w.scale,
            int(hist.max()), err)
        torch.cuda.synchronize()
        ref, _ = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, hist, w.scale)
        got = out.float().cpu().numpy().astype(np.float64)
        e = np.abs(got - ref)
        assert (e <= ATOL + RTOL * np.abs(ref)).all(), e.max()
        assert (got[0] == 0).all()  # the empty context gives a zero row
    assert int(err.item()) == 0


def test_static_error_word_and_null_error_word():
    need_gpu()
    w, d = _inputs(93)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(d["q"])
    # a context-length hint below the real lengths is clipped and flagged
    pa.pa_paged_decode_attention_static(out, d["q"], d["k"], d["v"], d["bt"], d["cl"], w.scale,
                                        64, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_DEVERR_CONTEXT_CLIPPED
    # the binding refuses a word the kernel's 4-byte atomic would overrun
    for bad in (torch.zeros(1, dtype=torch.uint8, device="cuda"),
                torch.zeros(0, dtype=torch.int32, device="cuda")):
        with pytest.raises(ValueError, match="error_word"):
            pa.pa_paged_decode_attention_static(out, d["q"], d["k"], d["v"], d["bt"], d["cl"],
                                                w.scale, w.max_context_len, bad)
    # without an error word the call still runs
    ref = _with_workspace(w, d)
    got = _static(w, d, None)
    torch.cuda.synchronize()
    _close(got, ref)


def test_static_refuses_problems_larger_than_its_scratch():
    need_gpu()
    B, HQ, HKV = 64, 64, 8
    need = pa.pa_paged_decode_workspace_size(B, HQ, HKV, 128, 131072)
    assert need > 16 << 20
    q = torch.zeros((B, HQ, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 16, HKV, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    cl = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(pa.PAError) as e:
        pa.pa_paged_decode_attention_static(out, q, kc, kc, bt, cl, 0.1, 131072)
    assert e.value.status == pa.PA_ERR_WORKSPACE
