"""Pins of the oracle's number formats (bf16 rounding, OCP E4M3FN encode/decode) against library
routines (torch's bfloat16 and float8_e4m3fn conversions) and the format's fixed points."""
import numpy as np
import pytest
import torch

import oracle


def torch_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_e4m3_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_e4m3_value(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).numpy()


def test_bf16_round_matches_torch_random():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),   # tiny and subnormal-adjacent
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
    ])
    assert np.array_equal(oracle.f32_to_bf16_array(x), torch_bf16_bits(x))


def test_bf16_round_ties_to_even():
    # lower 16 bits exactly 0x8000: a tie; the kept part decides (even stays, odd rounds up)
    kept = np.array([0x3F80, 0x3F81, 0xBF80, 0xBF81, 0x0001, 0x7F7F], np.uint32)
    u = (kept << 16) | 0x8000
    x = u.view(np.float32)
    got = oracle.f32_to_bf16_array(x)
    assert np.array_equal(got, torch_bf16_bits(x))
    assert got[0] == 0x3F80 and got[1] == 0x3F82
    assert got[5] == 0x7F80  # carry into the exponent overflows to +inf


def test_bf16_roundtrip_exact():
    rng = np.random.default_rng(12)
    bits = rng.integers(0, 1 << 16, 3000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    for h in bits[:500]:
        assert oracle.f32_to_bf16(oracle.bf16_to_f32(int(h))) == int(h)


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    ref = torch_e4m3_value(codes).astype(np.float64)
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert np.array_equal(nan_o, nan_r)
    assert set(np.flatnonzero(nan_o).tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan_o], ref[~nan_r])


def test_e4m3_format_fixed_points():
    assert oracle.e4m3_decode(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_decode(0x38) == 1.0            # bias 7
    assert oracle.e4m3_encode(1.0) == 0x38
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00


def test_e4m3_encode_sweep_matches_torch():
    x = np.linspace(-500.0, 500.0, 200_001, dtype=np.float32)
    rng = np.random.default_rng(13)
    x = np.concatenate([x, (rng.standard_normal(20000) * 10).astype(np.float32),
                        (rng.standard_normal(20000) * 2.0 ** -7).astype(np.float32)])
    ours = oracle.e4m3_encode_array(x)
    nonsat = np.abs(x) < 464.0   # below the midpoint 448..480: torch and satfinite agree
    assert np.array_equal(ours[nonsat], torch_e4m3_bits(x[nonsat]))
    sat = ~nonsat
    assert np.all((ours[sat] & 0x7F) == 0x7E)
    assert np.array_equal(ours[sat] >> 7, (x[sat] < 0).astype(np.uint8))


def test_e4m3_encode_midpoints_ties_to_even():
    vals = torch_e4m3_value(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float64)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    # only midpoints exactly representable in fp32 are true ties (all are: <= 5 significant bits)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)
    ours = oracle.e4m3_encode_array(mids)
    lo = np.arange(0, 0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(ours, expect)
    assert np.array_equal(ours, torch_e4m3_bits(mids))
    assert np.array_equal(oracle.e4m3_encode_array(-mids), expect | 0x80)


def test_e4m3_saturates_not_nan():
    for v in (448.0, 460.0, 479.9, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F
