"""Pins for the oracle's number formats (no GPU).

The oracle builds bf16, fp16 and fp8 e4m3 from their bit-field definitions
and rounds to the nearest value with ties to even.  These tests hold it to
things other than itself: closed-form values of the formats, and the
rounding casts of numpy (fp16) and torch (bf16, e4m3 inside its finite
range) used as library routines.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _bits_f32(n):
    return RNG.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)


# ----------------------------------------------------------- closed forms --
def test_format_sizes_and_maxima():
    # e4m3: exponent fields 0..15, mantissa 0..7, only S.1111.111 is NaN: 127 finite >= 0
    n, mx = oracle.format_info(oracle.E4M3)
    assert n == 127 and mx == 448.0
    # bf16: exponent fields 0..254 finite, 128 mantissas each
    n, mx = oracle.format_info(oracle.BF16)
    assert n == 255 * 128 and mx == (2 - 2**-7) * 2.0**127
    n, mx = oracle.format_info(oracle.FP16)
    assert n == 31 * 1024 and mx == 65504.0


@pytest.mark.parametrize("y,code", [
    (448.0, 0x7E), (464.0, 0x7E), (480.0, 0x7E), (1e6, 0x7E), (np.inf, 0x7E),
    (-np.inf, 0xFE), (-500.0, 0xFE),
    (2.0**-9, 0x01), (2.0**-10, 0x00), (3 * 2.0**-10, 0x02), (5 * 2.0**-10, 0x02),
    (7 * 2.0**-10, 0x04), (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (1.0625, 0x38),
    (1.1875, 0x3A), (-2.0, 0xC0), (2.0**-6, 0x08), (7 * 2.0**-9, 0x07), (240.0, 0x77),
    (256.0, 0x78), (0.05, 0x15)])
def test_e4m3_spot_values(y, code):
    # closed forms: 1.0 = exponent 7 (bias 7) -> 0x38; 1.0625 is the midpoint
    # of 1.0 (mantissa 0, even) and 1.125 -> 0x38; 1.1875 the midpoint of
    # 1.125 (odd) and 1.25 -> 0x3A; 2^-9 is the smallest subnormal; 2^-10 a tie
    # between 0 and 2^-9 -> 0; 3*2^-10 between 2^-9 (odd) and 2^-8 -> 2^-8;
    # 0.05 = 1.6 * 2^-5 -> nearest 1.625*2^-5 = exponent field 2, mantissa 5 = 0x15.
    assert int(oracle.encode(oracle.E4M3, np.array([y], np.float32))[0]) == code


def test_e4m3_nan():
    c = oracle.encode(oracle.E4M3, np.array([np.nan], np.float32))[0]
    assert c & 0x7F == 0x7F
    assert np.isnan(oracle.decode(oracle.E4M3, np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_every_code_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(oracle.E4M3, codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()
    assert nan.sum() == 2


def test_e4m3_encode_vs_torch_in_range():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest-even; inside +-448
    # it is a library stand-in for the definition.
    finite = oracle.decode(oracle.E4M3, np.arange(0, 127, dtype=np.uint8))
    mids = (finite[:-1] + finite[1:]) / 2
    y = np.concatenate([finite, mids, -mids, RNG.uniform(-448, 448, 200000),
                        RNG.standard_normal(100000) * 20, RNG.standard_normal(100000) * 1e-2])
    y = y.astype(np.float32)
    y = y[np.abs(y) <= 448]
    ours = oracle.encode(oracle.E4M3, y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (ours == ref).all()


def test_e4m3_roundtrip_and_monotone():
    codes = np.arange(0, 127, dtype=np.uint8)
    vals = oracle.decode(oracle.E4M3, codes)
    assert (np.diff(vals) > 0).all()
    assert (oracle.encode(oracle.E4M3, vals.astype(np.float32)) == codes).all()


def test_bf16_decode_every_code_vs_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(oracle.BF16, codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()


def test_bf16_encode_vs_torch():
    # random bit patterns (all exponents, subnormals, inf, NaN) and exact ties
    finite = oracle.decode(oracle.BF16, np.arange(0, 0x7F80, 97, dtype=np.uint16))
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    top = np.float32((2 - 2**-7) * 2.0**127)
    edge = np.array([top, np.nextafter(np.float32(3.4028235e38), np.float32(0)),
                     np.float32(3.4028235e38), np.float32(-3.4028235e38)], np.float32)
    y = np.concatenate([_bits_f32(1_000_000), mids, -mids, edge]).astype(np.float32)
    ours = oracle.encode(oracle.BF16, y)
    ref = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(y)
    assert (ours[~nan] == ref[~nan]).all()
    assert ((ours[nan] & 0x7F80) == 0x7F80).all() and ((ours[nan] & 0x7F) != 0).all()


def test_bf16_overflow_rounds_to_inf():
    # midpoint between the largest bf16 and 2^128 is (2 - 2^-8) * 2^127: its
    # tie goes to the even neighbour, 2^128, i.e. inf; just below stays finite
    mid = np.float32((2 - 2**-8) * 2.0**127)
    below = np.nextafter(mid, np.float32(0))
    c = oracle.encode(oracle.BF16, np.array([mid, below, np.inf, -mid], np.float32))
    assert list(c) == [0x7F80, 0x7F7F, 0x7F80, 0xFF80]


def test_fp16_encode_decode_vs_numpy():
    y = np.concatenate([_bits_f32(1_000_000),
                        RNG.standard_normal(100000).astype(np.float32) * 1e-5,
                        np.array([65504, 65519.99, 65520, 1e9, -1e9, 2**-24, 2**-25,
                                  3 * 2**-25, 0.0, -0.0], np.float32)]).astype(np.float32)
    ours = oracle.encode(oracle.FP16, y)
    with np.errstate(over="ignore"):
        ref = y.astype(np.float16).view(np.uint16)
    nan = np.isnan(y)
    assert (ours[~nan] == ref[~nan]).all()
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = oracle.decode(oracle.FP16, codes)
    r = codes.view(np.float16).astype(np.float64)
    rn = np.isnan(r)
    assert (np.isnan(dec) == rn).all() and (dec[~rn] == r[~rn]).all()


def test_fp32_passthrough():
    y = _bits_f32(1000)
    out = oracle.encode(oracle.FP32, y)
    same = (out.view(np.uint32) == y.view(np.uint32)) | (np.isnan(out) & np.isnan(y))
    assert same.all()
