"""Pins for the oracle's storage-format decoders and its E4M3 encoder.

The decoders are checked exhaustively against torch's own conversions (an
independent implementation) and against values fixed by the format
definitions; the encoder against torch's float8_e4m3fn rounding, hand-made
ties and the saturation rule.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc


def test_f16_decoder_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16).to(torch.float64).numpy()
    got = np.array([orc.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_decoder_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_decoder_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_decoder_format_facts():
    # OCP FP8 E4M3: max finite 448 = 1.75 * 2^8, min normal 2^-6, min subnormal 2^-9,
    # only S.1111.111 is NaN, no infinities.
    assert orc.e4m3_to_double(0x7E) == 448.0
    assert orc.e4m3_to_double(0xFE) == -448.0
    assert orc.e4m3_to_double(0x08) == 2.0 ** -6
    assert orc.e4m3_to_double(0x01) == 2.0 ** -9
    assert orc.e4m3_to_double(0x38) == 1.0
    assert math.isnan(orc.e4m3_to_double(0x7F)) and math.isnan(orc.e4m3_to_double(0xFF))
    finite = [orc.e4m3_to_double(c) for c in range(256) if c not in (0x7F, 0xFF)]
    assert all(math.isfinite(v) for v in finite)
    pos = [orc.e4m3_to_double(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))  # codes are monotone in value


def test_e4m3_encoder_roundtrip_all_codes():
    for c in range(256):
        v = orc.e4m3_to_double(c)
        if math.isnan(v):
            continue
        assert orc.e4m3_from_float(v) == c


def test_e4m3_encoder_ties_to_even():
    # Midpoint between 1.0 (0x38, mantissa 0) and 1.125 (0x39, mantissa 1) -> 1.0;
    # midpoint between 1.125 and 1.25 (0x3A, mantissa 2) -> 1.25.
    assert orc.e4m3_from_float(1.0625) == 0x38
    assert orc.e4m3_from_float(1.1875) == 0x3A
    # Subnormal midpoint between 2^-9 (0x01) and 2*2^-9 (0x02) -> 0x02;
    # between 0 and 2^-9 -> 0.
    assert orc.e4m3_from_float(1.5 * 2 ** -9) == 0x02
    assert orc.e4m3_from_float(0.5 * 2 ** -9) == 0x00
    assert orc.e4m3_from_float(-0.5 * 2 ** -9) == 0x80


def test_e4m3_encoder_saturates_and_nan():
    assert orc.e4m3_from_float(448.0) == 0x7E
    assert orc.e4m3_from_float(463.9) == 0x7E
    assert orc.e4m3_from_float(1e6) == 0x7E
    assert orc.e4m3_from_float(-1e6) == 0xFE
    assert orc.e4m3_from_float(float("inf")) == 0x7E
    assert orc.e4m3_from_float(float("nan")) == 0x7F


def test_e4m3_encoder_vs_torch_random():
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x.clamp(-448.0, 448.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_from_float(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(ref, got)
