"""The C-ABI library on a host without a GPU: it loads, exports every
function include/pa.h declares, plans splits correctly and rejects bad
arguments before launching anything (every call below returns during the
host-side checks; none reaches a kernel launch)."""
import ctypes
import math

import pytest

from paged_kv_cache_309_gb300 import build as pabuild
from paged_kv_cache_309_gb300 import pa


@pytest.fixture(scope="module")
def lib():
    pabuild.build()
    return pa.library()


def test_exports_every_declared_function(lib):
    names = pa.declared_functions()
    assert {"pa_reshape_and_cache", "pa_concat_mla_k", "pa_paged_decode_attention",
            "pa_paged_decode_workspace_size", "pa_paged_decode_plan",
            "pa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(6):
        s = lib.pa_status_string(code).decode()
        assert s.startswith("PA_")
    assert b"unknown" in lib.pa_status_string(99)


@pytest.mark.parametrize("B,HKV,ctx,sms", [(8, 8, 131072, 152), (64, 8, 4096, 152),
                                           (4, 8, 64, 152), (1, 1, 1, 152), (1, 8, 1000, 152),
                                           (256, 8, 32768, 152), (8, 8, 131072, 148),
                                           (3, 2, 777, 10)])
def test_plan_covers_context(B, HKV, ctx, sms):
    splits, tps = pa.pa_paged_decode_plan(B, HKV, ctx, sms)
    assert splits >= 1 and tps >= 64 and tps % 64 == 0
    assert splits * tps >= ctx                      # every token has a split
    assert (splits - 1) * tps < ctx                 # no split starts past the context
    if splits > 1:
        # enough CTAs to fill the machine many times over
        assert B * HKV * splits >= min(32 * sms, B * HKV * math.ceil(ctx / 64)) * 0.5


def test_plan_long_context_example():
    # B=8, H_KV=8, up to 128K tokens on 152 SMs: ~4864 CTAs planned
    splits, tps = pa.pa_paged_decode_plan(8, 8, 131072, 152)
    assert (splits, tps) == (76, 1728)


def test_plan_zero_context():
    assert pa.pa_paged_decode_plan(4, 8, 0, 152) == (1, 64)


def test_workspace_size_formula(lib):
    # one split (short context): only the 256-byte header
    assert lib.pa_paged_decode_workspace_size(4, 16, 8, 128, 64) == 256
    # several splits: header + split counters + lse partials (each 256-aligned)
    # + fp32 output partials
    splits, _ = pa.pa_paged_decode_plan(8, 8, 131072, 0)
    rows = 8 * 32 * splits
    al = lambda x: (x + 255) // 256 * 256
    want = 256 + al(8 * 8 * 4) + al(rows * 4) + rows * 128 * 4
    if splits > 1:
        assert lib.pa_paged_decode_workspace_size(8, 32, 8, 128, 131072) == want


P = ctypes.c_void_p
FAKE = P(0x100000)          # 16-byte aligned, never dereferenced
FAKE_MIS = P(0x100008)      # misaligned


def _rc(lib, **kw):
    a = dict(key=FAKE, value=FAKE, src=pa.PA_BF16, n=4, h=8, d=128, ks=1024, vs=1024,
             kc=FAKE, vc=FAKE, cd=pa.PA_BF16, nb=4, bs=16, bstride=16 * 1024, slot=FAKE,
             swa=None, swa_len=0, ksc=None, vsc=None)
    a.update(kw)
    return lib.pa_reshape_and_cache(a["key"], a["value"], a["src"], a["n"], a["h"], a["d"],
                                    a["ks"], a["vs"], a["kc"], a["vc"], a["cd"], a["nb"],
                                    a["bs"], a["bstride"], a["slot"], a["swa"], a["swa_len"],
                                    a["ksc"], a["vsc"], None)


def test_reshape_and_cache_rejects(lib):
    assert _rc(lib, key=None) == pa.PA_ERR_INVALID
    assert _rc(lib, slot=None) == pa.PA_ERR_INVALID
    assert _rc(lib, value=None) == pa.PA_ERR_INVALID          # value_cache given
    assert _rc(lib, ksc=FAKE) == pa.PA_ERR_INVALID            # only one scale
    assert _rc(lib, n=-1) == pa.PA_ERR_INVALID
    assert _rc(lib, h=0) == pa.PA_ERR_INVALID
    assert _rc(lib, src=pa.PA_FP8_E4M3) == pa.PA_ERR_UNSUPPORTED
    assert _rc(lib, cd=7) == pa.PA_ERR_UNSUPPORTED
    assert _rc(lib, h=1, d=12) == pa.PA_ERR_ALIGN             # row not a multiple of 8
    assert _rc(lib, ks=1028) == pa.PA_ERR_ALIGN
    assert _rc(lib, bstride=16 * 1024 + 4) == pa.PA_ERR_ALIGN
    assert _rc(lib, key=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert _rc(lib, ks=512) == pa.PA_ERR_INVALID              # token rows overlap
    assert _rc(lib, bstride=1024) == pa.PA_ERR_INVALID        # blocks overlap
    assert _rc(lib, n=0) == pa.PA_OK                          # nothing to do, no launch


def _dec(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, cd=pa.PA_BF16, bt=FAKE, cl=FAKE, B=4, HQ=32,
             HKV=8, d=128, bs=16, mbps=8, nb=64, scale=0.088, maxctx=128, ws=None, wsb=0)
    a.update(kw)
    return lib.pa_paged_decode_attention(a["out"], a["q"], a["kc"], a["vc"], a["cd"], a["bt"],
                                         a["cl"], a["B"], a["HQ"], a["HKV"], a["d"], a["bs"],
                                         a["mbps"], a["nb"], a["scale"], a["maxctx"], a["ws"],
                                         a["wsb"], None)


def test_decode_rejects(lib):
    assert _dec(lib, q=None, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_INVALID
    assert _dec(lib, HQ=12, HKV=8, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_INVALID
    assert _dec(lib, scale=float("nan"), ws=FAKE, wsb=1 << 20) == pa.PA_ERR_INVALID
    assert _dec(lib, cd=pa.PA_FP16, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_UNSUPPORTED
    assert _dec(lib, d=64, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_UNSUPPORTED
    assert _dec(lib, HQ=24, HKV=8, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_UNSUPPORTED  # G=3
    assert _dec(lib, bs=12, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_UNSUPPORTED
    assert _dec(lib, bs=4, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_UNSUPPORTED
    assert _dec(lib, nb=1 << 28, bs=16, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_UNSUPPORTED
    assert _dec(lib, out=FAKE_MIS, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_ALIGN
    assert _dec(lib) == pa.PA_ERR_WORKSPACE
    assert _dec(lib, ws=FAKE, wsb=16) == pa.PA_ERR_WORKSPACE
    assert _dec(lib, ws=P(0x100010), wsb=1 << 20) == pa.PA_ERR_ALIGN
    assert _dec(lib, nb=0, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_INVALID
    assert _dec(lib, maxctx=-1, ws=FAKE, wsb=1 << 20) == pa.PA_ERR_INVALID


def test_concat_rejects(lib):
    def c(**kw):
        a = dict(k=FAKE, kd=pa.PA_BF16, kn=FAKE, kr=FAKE, sd=pa.PA_BF16, n=4, h=128, nope=128,
                 rope=64, k0=128 * 192, k1=192, n0=128 * 128, n1=128, r0=64)
        a.update(kw)
        return lib.pa_concat_mla_k(a["k"], a["kd"], a["kn"], a["kr"], a["sd"], a["n"], a["h"],
                                   a["nope"], a["rope"], a["k0"], a["k1"], a["n0"], a["n1"],
                                   a["r0"], None)
    assert c(k=None) == pa.PA_ERR_INVALID
    assert c(h=0) == pa.PA_ERR_INVALID
    assert c(sd=pa.PA_FP8_E4M3) == pa.PA_ERR_UNSUPPORTED
    assert c(nope=100) == pa.PA_ERR_ALIGN
    assert c(k1=190) == pa.PA_ERR_ALIGN
    assert c(k1=184) == pa.PA_ERR_INVALID          # heads overlap in k
    assert c(kr=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert c(n=0) == pa.PA_OK


def test_concat_and_cache_mla_rejects(lib):
    def c(**kw):
        a = dict(kvc=FAKE, kpe=FAKE, sd=pa.PA_BF16, n=4, dc=512, dr=64, cs=512, ps=64,
                 cache=FAKE, cd=pa.PA_BF16, nb=4, bs=64, bstride=64 * 576, slot=FAKE, sc=None)
        a.update(kw)
        return lib.pa_concat_and_cache_mla(a["kvc"], a["kpe"], a["sd"], a["n"], a["dc"], a["dr"],
                                           a["cs"], a["ps"], a["cache"], a["cd"], a["nb"],
                                           a["bs"], a["bstride"], a["slot"], a["sc"], None)
    assert c(kvc=None) == pa.PA_ERR_INVALID
    assert c(kpe=None) == pa.PA_ERR_INVALID
    assert c(slot=None) == pa.PA_ERR_INVALID
    assert c(dr=0) == pa.PA_ERR_INVALID
    assert c(sd=pa.PA_FP8_E4M3) == pa.PA_ERR_UNSUPPORTED
    assert c(dc=500) == pa.PA_ERR_ALIGN
    assert c(ps=68) == pa.PA_ERR_ALIGN
    assert c(cs=256) == pa.PA_ERR_INVALID           # token rows of kv_c overlap
    assert c(bstride=64 * 512) == pa.PA_ERR_INVALID  # blocks overlap
    assert c(cache=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert c(n=0) == pa.PA_OK


def _mla(lib, **kw):
    a = dict(out=FAKE, q=FAKE, cache=FAKE, bt=FAKE, cl=FAKE, B=4, H=128, dc=512, dr=64, bs=64,
             mbps=8, nb=64, scale=0.072, maxctx=512, ws=FAKE, wsb=1 << 28)
    a.update(kw)
    return lib.pa_mla_decode_attention(a["out"], a["q"], a["cache"], a["bt"], a["cl"], a["B"],
                                       a["H"], a["dc"], a["dr"], a["bs"], a["mbps"], a["nb"],
                                       a["scale"], a["maxctx"], a["ws"], a["wsb"], None)


def test_mla_decode_rejects(lib):
    assert _mla(lib, q=None) == pa.PA_ERR_INVALID
    assert _mla(lib, B=-1) == pa.PA_ERR_INVALID
    assert _mla(lib, scale=float("inf")) == pa.PA_ERR_INVALID
    assert _mla(lib, maxctx=-1) == pa.PA_ERR_INVALID
    assert _mla(lib, dc=256) == pa.PA_ERR_UNSUPPORTED
    assert _mla(lib, dr=32) == pa.PA_ERR_UNSUPPORTED
    assert _mla(lib, H=24) == pa.PA_ERR_UNSUPPORTED            # not a multiple of 16
    assert _mla(lib, bs=4) == pa.PA_ERR_UNSUPPORTED
    assert _mla(lib, bs=48) == pa.PA_ERR_UNSUPPORTED
    assert _mla(lib, out=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert _mla(lib, ws=None) == pa.PA_ERR_WORKSPACE
    assert _mla(lib, wsb=16) == pa.PA_ERR_WORKSPACE
    assert _mla(lib, ws=P(0x100010)) == pa.PA_ERR_ALIGN


def test_mla_workspace_size(lib):
    assert lib.pa_mla_decode_workspace_size(4, 24, 512) == 0      # heads not a multiple of 16
    assert lib.pa_mla_decode_workspace_size(4, 128, -1) == 0
    assert lib.pa_mla_decode_workspace_size(0, 128, 512) >= 256
    # both kernels: counters + two partial slots per chunk of the balanced
    # schedule, independent of the context length
    for B, H in ((64, 128), (64, 16), (4096, 64), (3, 48)):
        a = lib.pa_mla_decode_workspace_size(B, H, 512)
        assert a > 256 and a == lib.pa_mla_decode_workspace_size(B, H, 131072)
    # the partial slots do not depend on the batch: only the counters grow with B
    al = lambda x: (x + 255) // 256 * 256
    for H, per_b in ((16, 4), (64, 4), (128, 8)):
        d = lib.pa_mla_decode_workspace_size(4096, H, 512) - lib.pa_mla_decode_workspace_size(
            64, H, 512)
        assert d == al(4096 * per_b) - al(64 * per_b)


def test_mla_projections_reject(lib):
    ab = lambda **kw: lib.pa_mla_absorb_q(*[dict(dict(y=FAKE, qn=FAKE, qp=FAKE, w=FAKE, B=4,
                                                      H=128, dh=128, dr=64, dc=512), **kw)[k]
                                            for k in ("y", "qn", "qp", "w", "B", "H", "dh", "dr",
                                                      "dc")], None)
    assert ab(qn=None) == pa.PA_ERR_INVALID
    assert ab(H=0) == pa.PA_ERR_INVALID
    assert ab(dh=96) == pa.PA_ERR_UNSUPPORTED
    assert ab(dr=4) == pa.PA_ERR_UNSUPPORTED
    assert ab(w=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert ab(B=0) == pa.PA_OK
    pr = lambda **kw: lib.pa_mla_project_out(*[dict(dict(y=FAKE, x=FAKE, w=FAKE, B=4, H=128,
                                                         dc=512, dv=128), **kw)[k]
                                               for k in ("y", "x", "w", "B", "H", "dc", "dv")],
                                             None)
    assert pr(w=None) == pa.PA_ERR_INVALID
    assert pr(dv=100) == pa.PA_ERR_UNSUPPORTED
    assert pr(x=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert pr(B=0) == pa.PA_OK


_DEC_KEYS = ("out", "q", "kc", "vc", "cd", "bt", "cl", "B", "HQ", "HKV", "d", "bs", "mbps",
             "nb", "scale", "maxctx")


def _dec_args(**kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, cd=pa.PA_BF16, bt=FAKE, cl=FAKE, B=4, HQ=32,
             HKV=8, d=128, bs=16, mbps=8, nb=64, scale=0.088, maxctx=128)
    a.update(kw)
    return a


def test_decode_fp8_rejects(lib):
    def fp8(ksc=FAKE, vsc=FAKE, ws=FAKE, wsb=1 << 20, **kw):
        a = _dec_args(**kw)
        return lib.pa_paged_decode_attention_fp8(
            a["out"], a["q"], a["kc"], a["vc"], ksc, vsc, a["bt"], a["cl"], a["B"], a["HQ"],
            a["HKV"], a["d"], a["bs"], a["mbps"], a["nb"], a["scale"], a["maxctx"], ws, wsb,
            None)
    assert fp8(vsc=None) == pa.PA_ERR_INVALID                 # one scale without the other
    assert fp8(ksc=None) == pa.PA_ERR_INVALID
    assert fp8(q=None) == pa.PA_ERR_INVALID                   # the shared decode checks
    assert fp8(HQ=12) == pa.PA_ERR_INVALID
    assert fp8(d=64) == pa.PA_ERR_UNSUPPORTED
    assert fp8(bs=12) == pa.PA_ERR_UNSUPPORTED
    assert fp8(kc=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert fp8(ws=None) == pa.PA_ERR_WORKSPACE
    assert fp8(wsb=16) == pa.PA_ERR_WORKSPACE
    assert fp8(ws=P(0x100010)) == pa.PA_ERR_ALIGN             # workspace below 256 B alignment


def test_decode_step_rejects(lib):
    def step(nk=FAKE, nv=FAKE, sl=FAKE, ksc=None, vsc=None, ws=FAKE, wsb=1 << 20, **kw):
        a = _dec_args(**kw)
        return lib.pa_paged_decode_step(
            a["out"], a["q"], nk, nv, sl, a["kc"], a["vc"], a["cd"], ksc, vsc, a["bt"], a["cl"],
            a["B"], a["HQ"], a["HKV"], a["d"], a["bs"], a["mbps"], a["nb"], a["scale"],
            a["maxctx"], ws, wsb, None)
    assert step(ksc=FAKE) == pa.PA_ERR_INVALID                # one scale
    assert step(ksc=FAKE, vsc=FAKE) == pa.PA_ERR_INVALID      # scales with a bf16 cache
    assert step(nk=None) == pa.PA_ERR_INVALID                 # new tokens missing
    assert step(sl=None) == pa.PA_ERR_INVALID
    assert step(nv=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert step(cd=pa.PA_FP16) == pa.PA_ERR_UNSUPPORTED
    assert step(scale=float("inf")) == pa.PA_ERR_INVALID
    assert step(ws=None) == pa.PA_ERR_WORKSPACE
    assert step(ws=P(0x100010)) == pa.PA_ERR_ALIGN


def test_prefill_rejects(lib):
    def pf(cu=FAKE, mql=64, err=FAKE, **kw):
        a = _dec_args(**kw)
        return lib.pa_paged_prefill_attention(
            a["out"], a["q"], a["kc"], a["vc"], a["cd"], a["bt"], cu, a["cl"], a["B"], a["HQ"],
            a["HKV"], a["d"], a["bs"], a["mbps"], a["nb"], a["scale"], mql, err, None)
    assert pf(B=0) == pa.PA_OK                                # nothing to attend, no launch
    assert pf(mql=0) == pa.PA_OK
    assert pf(mql=-1) == pa.PA_ERR_INVALID
    assert pf(HQ=0) == pa.PA_ERR_INVALID
    assert pf(nb=0) == pa.PA_ERR_INVALID
    assert pf(cu=None) == pa.PA_ERR_INVALID
    assert pf(err=None) == pa.PA_ERR_INVALID                  # the error word is required
    assert pf(HQ=12) == pa.PA_ERR_INVALID
    assert pf(scale=float("nan")) == pa.PA_ERR_INVALID
    assert pf(cd=pa.PA_FP8_E4M3) == pa.PA_ERR_UNSUPPORTED
    assert pf(d=64) == pa.PA_ERR_UNSUPPORTED
    assert pf(HQ=24) == pa.PA_ERR_UNSUPPORTED                 # G = 3
    assert pf(bs=4) == pa.PA_ERR_UNSUPPORTED
    assert pf(nb=1 << 28) == pa.PA_ERR_UNSUPPORTED            # slots past int32
    assert pf(out=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert pf(err=P(0x100002)) == pa.PA_ERR_ALIGN


def test_static_decode_rejects(lib):
    def st(err=None, **kw):
        a = _dec_args(**kw)
        return lib.pa_paged_decode_attention_static(*[a[k] for k in _DEC_KEYS], err, None)
    assert st(q=None) == pa.PA_ERR_INVALID
    assert st(HQ=12) == pa.PA_ERR_INVALID
    assert st(d=64) == pa.PA_ERR_UNSUPPORTED
    assert st(vc=FAKE_MIS) == pa.PA_ERR_ALIGN
    assert st(err=P(0x100002)) == pa.PA_ERR_ALIGN             # error word not 4-byte aligned
    assert st(B=0) == pa.PA_OK                                # no sequences: returns before
                                                              # touching the device scratch


def test_selftest_rejects(lib):
    assert lib.pa_selftest_bounded_wait(None, None) == pa.PA_ERR_INVALID
    assert lib.pa_selftest_bounded_wait(P(0x100002), None) == pa.PA_ERR_INVALID


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the built CUDA library every call raises."""
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "LIB_PATH", str(tmp_path / "libpa.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pa.library()
    with pytest.raises(RuntimeError, match="missing"):
        pa.pa_paged_decode_plan(8, 8, 1000)
    with pytest.raises(RuntimeError, match="missing"):
        pa.pa_paged_decode_workspace_size(8, 32, 8, 128, 1000)
