"""Oracle element codecs pinned to independent library routines (numpy float16,
torch bfloat16 and float8_e4m3fn) over every bit pattern, and to values the
OCP E4M3 definition fixes."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, oracle.BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(codes, oracle.E4M3)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_definition_values():
    d = oracle.lib().orc_decode_e4m3
    assert d(0x7E) == 448.0            # largest finite: 1.75 * 2^8
    assert d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6        # smallest normal
    assert d(0x01) == 2.0 ** -9        # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert d(0x38) == 1.0              # exponent field 7 = bias
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    # no infinity: every non-NaN code is finite
    vals = [d(c) for c in range(256) if c & 0x7F != 0x7F]
    assert all(math.isfinite(v) for v in vals)
    assert len(set(vals)) == 253  # 254 non-NaN codes, +0 and -0 compare equal


def test_e4m3_encode_in_range_matches_torch_for_all_bf16():
    # Every finite bf16 value with |x| <= 448: round to nearest, ties to even.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    keep = torch.isfinite(x) & (x.abs() <= 448)
    x = x[keep].contiguous()
    ours = oracle.encode_e4m3(x.numpy())
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_random_floats_match_torch():
    r = np.random.Generator(np.random.PCG64(123))
    x = (r.standard_normal(2_000_000) * np.exp(r.uniform(-14, 6, 2_000_000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ours = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_ties_to_even():
    e = oracle.lib().orc_encode_e4m3
    # 1 + 1/16 lies halfway between 1 (code 0x38, even) and 1.125 (0x39)
    assert e(1.0 + 1.0 / 16) == 0x38
    # 1.125 + 1/16 lies between 0x39 (odd) and 0x3A (even)
    assert e(1.125 + 1.0 / 16) == 0x3A
    # halfway between the two smallest subnormals: 1.5 * 2^-9 -> 2 * 2^-9 (even)
    assert e(1.5 * 2.0 ** -9) == 0x02
    assert e(0.5 * 2.0 ** -9) == 0x00  # ties to zero (even)


@pytest.mark.parametrize("x,code", [(448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E),
                                    (float("inf"), 0x7E), (-500.0, 0xFE),
                                    (float("-inf"), 0xFE)])
def test_e4m3_encode_saturates(x, code):
    assert oracle.lib().orc_encode_e4m3(x) == code


def test_e4m3_encode_nan_and_signed_zero():
    e = oracle.lib().orc_encode_e4m3
    assert e(float("nan")) & 0x7F == 0x7F
    assert e(0.0) == 0x00 and e(-0.0) == 0x80


def test_e4m3_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.decode(codes, oracle.E4M3).astype(np.float32)
    assert np.array_equal(oracle.encode_e4m3(vals), codes)
