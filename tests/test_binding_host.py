"""The Python binding refuses, on the host and before any launch, tensors the
kernels cannot address: a CPU tensor passed where the C ABI expects a device
pointer would be dereferenced by the GPU as a device address.  Runs without a
GPU: every call below must raise ValueError before the library is touched."""
import pytest
import torch

from paged_kv_cache_309_gb300 import pa


def _t(shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)  # CPU tensors


def _decode_args():
    q = _t((2, 8, 128))
    kc = _t((4, 16, 4, 128))
    return dict(out=q.clone(), q=q, k_cache=kc, v_cache=kc.clone(),
                block_tables=_t((2, 1), torch.int32), context_lens=_t((2,), torch.int32))


@pytest.fixture(autouse=True)
def _no_library(monkeypatch):
    # any call that got past the checks would load libpa.so: make that an error
    def fail():
        raise AssertionError("the binding reached the library with a host tensor")
    monkeypatch.setattr(pa, "_load", fail)


def test_reshape_and_cache_refuses_host_tensors():
    x = _t((4, 8, 128))
    c = _t((4, 16, 8, 128))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_reshape_and_cache(x, x.clone(), c, c.clone(), _t((4,), torch.int64))


def test_reshape_and_cache_refuses_one_scale():
    x = _t((4, 8, 128))
    with pytest.raises(ValueError):
        pa.pa_reshape_and_cache(x, x, x, x, x, k_scale=_t((1,), torch.float32))


def test_concat_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_concat_mla_k(_t((2, 4, 192)), _t((2, 4, 128)), _t((2, 1, 64)))


def test_decode_wrappers_refuse_host_tensors():
    a = _decode_args()
    with pytest.raises(ValueError, match="out must be a CUDA tensor"):
        pa.pa_paged_decode_attention(a["out"], a["q"], a["k_cache"], a["v_cache"],
                                     a["block_tables"], a["context_lens"], 0.1, 16,
                                     _t((256,), torch.uint8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_paged_decode_attention_static(a["out"], a["q"], a["k_cache"], a["v_cache"],
                                            a["block_tables"], a["context_lens"], 0.1, 16)


def test_decode_step_and_prefill_refuse_host_tensors():
    a = _decode_args()
    nk = _t((2, 4, 128))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_paged_decode_step(a["out"], a["q"], nk, nk.clone(), _t((2,), torch.int64),
                                a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"],
                                0.1, 16, _t((256,), torch.uint8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_paged_prefill_attention(a["out"], a["q"], a["k_cache"], a["v_cache"],
                                      a["block_tables"], _t((3,), torch.int32),
                                      a["context_lens"], 0.1, 1, _t((1,), torch.int32))


def test_error_word_is_required_and_checked():
    with pytest.raises(ValueError, match="error_word"):
        pa.pa_selftest_bounded_wait(None)
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_selftest_bounded_wait(_t((1,), torch.int32))
    a = _decode_args()
    with pytest.raises(ValueError, match="error_word"):
        pa.pa_paged_prefill_attention(a["out"], a["q"], a["k_cache"], a["v_cache"],
                                      a["block_tables"], _t((3,), torch.int32),
                                      a["context_lens"], 0.1, 1, None)


def test_mla_wrappers_refuse_host_tensors():
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_mla_absorb_q(_t((2, 128, 576)), _t((2, 128, 128)), _t((2, 128, 64)),
                           _t((512, 128 * 128)))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_mla_decode_attention(_t((2, 16, 512)), _t((2, 16, 576)), _t((4, 64, 1, 576)),
                                   _t((2, 1), torch.int32), _t((2,), torch.int32), 0.1, 64,
                                   _t((256,), torch.uint8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        pa.pa_mla_project_out(_t((2, 16, 128)), _t((2, 16, 512)), _t((512, 16 * 128)))
