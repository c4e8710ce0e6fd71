"""Pins of the oracle's element decoders and output rounding (CPU only).

Each decoder is checked against an implementation that shares nothing with the
oracle: numpy's float16, torch's bfloat16 / float8_e4m3fn / float8_e8m0fnu
casts, and for E2M1 (which neither library can convert) a generic minifloat
decoder that is itself first checked against torch on E4M3 and E5M2.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or a == b


def test_f16_decode_all_codes_vs_numpy():
    ref = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    got = oracle.f16_bits_to_f64_array(np.arange(65536, dtype=np.uint16))
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_decode_all_codes_vs_torch():
    ref = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_bits_to_f64_array(np.arange(65536, dtype=np.uint16).astype(np.int16).view(np.uint16))
    # torch's int16 view starts at 0x0000 too, codes in the same order
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def _f16_rounding_cases():
    rng = np.random.default_rng(5)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 5, 3000))
    # exact midpoints between neighbouring fp16 values (ties), normal and subnormal
    h = np.arange(0, 0x7bff, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    h2 = (np.arange(0, 0x7bff, 37, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    xs += list((h + h2) / 2) + list(-(h + h2) / 2)
    xs += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
           3 * 2.0 ** -26, 2.0 ** -26, 6.0e-8, 2.0 ** -14 - 2.0 ** -25, float("inf"), -float("inf")]
    return xs


def test_f64_to_f16_rne_vs_numpy():
    for x in _f16_rounding_cases():
        want = int(np.array([x], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.f64_to_f16(x) == want, x
    assert math.isnan(oracle.f16_to_f64(oracle.f64_to_f16(float("nan"))))


def test_f64_to_bf16_rne_vs_torch():
    rng = np.random.default_rng(6)
    xs = list((rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)).astype(np.float32))
    # exact ties between neighbouring bf16 values (representable in fp32)
    codes = torch.arange(0, 0x7f7f, 97, dtype=torch.int32).to(torch.int16)
    lo = codes.view(torch.bfloat16).double()
    hi = (codes + 1).view(torch.bfloat16).double()
    xs += list(((lo + hi) / 2).float().numpy()) + list((-(lo + hi) / 2).float().numpy())
    xs += [np.float32(3.3895314e38), np.float32(3.4e38), np.float32(1e-40), np.float32(0.0)]
    for x in xs:
        want = int(torch.tensor([float(x)], dtype=torch.float32).to(torch.bfloat16)
                   .view(torch.int16).item()) & 0xFFFF
        assert oracle.f64_to_bf16(float(x)) == want, x


def test_e4m3_all_codes_vs_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        assert _same(oracle.e4m3_to_f64(c), float(ref[c])), hex(c)
    assert oracle.e4m3_to_f64(0x7E) == 448.0


def test_e5m2_all_codes_vs_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    for c in range(256):
        assert _same(oracle.e5m2_to_f64(c), float(ref[c])), hex(c)
    assert oracle.e5m2_to_f64(0x7B) == 57344.0 and oracle.e5m2_to_f64(0x7C) == float("inf")
    assert oracle.e5m2_to_f64(0x01) == 2.0 ** -16  # smallest subnormal


def test_e8m0_all_codes_vs_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for c in range(256):
        assert _same(oracle.e8m0_to_f64(c), float(ref[c])), hex(c)
    assert oracle.e8m0_to_f64(127) == 1.0


def _minifloat(code, ebits, mbits, bias, nan_codes=(), inf=False):
    """Generic sign/exponent/mantissa decoder, used only to cross-check E2M1."""
    s = code >> (ebits + mbits)
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if code & ((1 << (ebits + mbits)) - 1) in nan_codes:
        return float("nan")
    if inf and e == (1 << ebits) - 1:
        return float("nan") if m else (-1) ** s * float("inf")
    if e == 0:
        v = m / (1 << mbits) * 2.0 ** (1 - bias)
    else:
        v = (1 + m / (1 << mbits)) * 2.0 ** (e - bias)
    return -v if s else v


def test_generic_minifloat_matches_torch_fp8():
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    e5 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    for c in range(256):
        assert _same(_minifloat(c, 4, 3, 7, nan_codes=(0x7F,)), float(e4[c]))
        assert _same(_minifloat(c, 5, 2, 15, inf=True), float(e5[c]))


def test_e2m1_all_codes_vs_generic_minifloat():
    for c in range(16):
        assert oracle.e2m1_to_f64(c) == _minifloat(c, 2, 1, 1), c
    mags = sorted({abs(oracle.e2m1_to_f64(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert oracle.e2m1_to_f64(0xF) == -6.0
