"""Pins for oracle.numerics: format definitions, library decoders, known values, ties."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import numerics as nm


def test_bf16_decode_matches_torch_for_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ours = nm.bf16_bits_to_f64(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xBF80, -1.0), (0x4000, 2.0), (0x3F81, 1.0 + 2.0 ** -7),
    (0x0080, 2.0 ** -126), (0x0001, 2.0 ** -133), (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127),
    (0x7F80, np.inf), (0xFF80, -np.inf), (0x0000, 0.0),
])
def test_bf16_known_values(bits, value):
    assert nm.bf16_bits_to_f64(np.uint16(bits)) == value


def test_bf16_rne_ties_and_overflow():
    one = 1.0
    q = 2.0 ** -7  # bf16 step in [1, 2)
    cases = {
        one + q / 2: 0x3F80,          # tie -> even (1.0)
        one + 3 * q / 2: 0x3F82,      # tie between 1+q (odd) and 1+2q (even) -> up
        one + q / 2 - 2.0 ** -40: 0x3F80,
        one + q / 2 + 2.0 ** -40: 0x3F81,
        -(one + 3 * q / 2): 0xBF82,
        (2 - 2.0 ** -8) * 2.0 ** 127: 0x7F80,               # tie above max -> even = inf
        (2 - 2.0 ** -8) * 2.0 ** 127 - 2.0 ** 100: 0x7F7F,  # just below the tie -> max
        2.0 ** -134: 0x0000,          # half the smallest subnormal: tie -> 0 (even)
        3 * 2.0 ** -134: 0x0002,      # 1.5 subnormal steps -> 2 (even)
        2.0 ** -126 - 2.0 ** -140: 0x0080,  # rounds up into the normal range
    }
    for x, bits in cases.items():
        assert int(nm.f64_to_bf16_rne(np.float64(x))) == bits, (x, hex(bits))


def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(11)
    x32 = (rng.standard_normal(200_000) * np.exp(rng.uniform(-80, 80, 200_000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(nm.f64_to_bf16_rne(x32.astype(np.float64)), ref)


def test_bf16_rne_roundtrip_and_generator_agree():
    codes = np.arange(65536, dtype=np.uint16)
    vals = nm.bf16_bits_to_f64(codes)
    finite = np.isfinite(vals)
    back = nm.f64_to_bf16_rne(vals[finite])
    # -0 and +0 keep their sign bit
    assert np.array_equal(back, codes[finite])
    rng = np.random.default_rng(12)
    x = rng.standard_normal(100_000) * np.exp(rng.uniform(-95, 88, 100_000))
    assert np.array_equal(nm.f64_to_bf16_rne(x), synthetic.f64_to_bf16_bits(x))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = nm.e4m3fn_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("code,value", [
    (0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6),
    (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x3C, 1.5), (0x00, 0.0),
])
def test_e4m3_known_values(code, value):
    assert nm.e4m3fn_to_f64(np.uint8(code)) == value


def test_e4m3_nan_codes():
    assert np.isnan(nm.e4m3fn_to_f64(np.uint8(0x7F)))
    assert np.isnan(nm.e4m3fn_to_f64(np.uint8(0xFF)))
    assert np.signbit(nm.e4m3fn_to_f64(np.uint8(0x80)))


def test_e4m3_generator_encode_roundtrip_and_rne():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = nm.e4m3fn_to_f64(codes)
    assert np.array_equal(synthetic.f64_to_e4m3_codes(vals), codes)
    # ties: 1 + 1/16 lies halfway between 1.0 (0x38, even) and 1.125 (0x39) -> 0x38
    assert synthetic.f64_to_e4m3_codes(np.float64(1 + 1 / 16)) == 0x38
    assert synthetic.f64_to_e4m3_codes(np.float64(1 + 3 / 16)) == 0x3A
    assert synthetic.f64_to_e4m3_codes(np.float64(1000.0)) == 0x7E  # satfinite


def test_e8m0_decode():
    assert nm.e8m0_to_f64(np.uint8(127)) == 1.0
    assert nm.e8m0_to_f64(np.uint8(0)) == 2.0 ** -127
    assert nm.e8m0_to_f64(np.uint8(254)) == 2.0 ** 127
    assert nm.e8m0_to_f64(np.uint8(123)) == 2.0 ** -4
    assert np.isnan(nm.e8m0_to_f64(np.uint8(255)))
    if hasattr(torch, "float8_e8m0fnu"):
        codes = np.arange(255, dtype=np.uint8)
        ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
        assert np.array_equal(nm.e8m0_to_f64(codes), ref)
