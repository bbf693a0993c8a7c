"""Pins for the oracle's number formats: e4m3, e2m1, UE8M0, bf16."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests.refs import E2M1_TABLE, e4m3_decode_torch, e4m3_encode_torch, f32_to_bf16_torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_e4m3_decode_matches_torch_all_codes(orc):
    ref = e4m3_decode_torch(np.arange(256, dtype=np.uint8))
    for c in range(256):
        v = orc.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c


def test_e4m3_landmarks(orc):
    assert orc.e4m3_value(0x7E) == 448.0          # largest finite
    assert orc.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert orc.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert math.isnan(orc.e4m3_value(0x7F)) and math.isnan(orc.e4m3_value(0xFF))


def all_bf16_values():
    u = np.arange(65536, dtype=np.uint32) << 16
    return u.view(np.float32)


def test_e4m3_encode_round_to_nearest_even_matches_torch(orc):
    v = all_bf16_values()
    ok = np.isfinite(v) & (np.abs(v) < 464.0)
    vals = v[ok]
    ref = e4m3_encode_torch(vals)
    got = np.array([orc.e4m3_from_float(float(x)) for x in vals], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_and_nan(orc):
    for x in [448.0, 464.0, 500.0, 1e30, float("inf")]:
        assert orc.e4m3_from_float(x) == 0x7E
        assert orc.e4m3_from_float(-x) == 0xFE
    assert orc.e4m3_from_float(float("nan")) == 0x7F


def test_e4m3_encode_is_nearest(orc):
    """Brute force: the code returned is a nearest finite e4m3 value (ties to
    an even mantissa), for random fp32 inputs in range."""
    rng = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if not math.isnan(orc.e4m3_value(c))], np.uint8)
    vals = np.array([orc.e4m3_value(int(c)) for c in finite])
    xs = np.concatenate([rng.standard_normal(2000) * 20, rng.standard_normal(2000) * 0.01]).astype(np.float32)
    for x in xs:
        c = orc.e4m3_from_float(float(x))
        d = np.abs(vals - float(x))
        best = d.min()
        assert abs(orc.e4m3_value(c) - float(x)) == best
        ties = finite[d == best]
        if len(ties) > 1:
            assert (c & 1) == 0  # even mantissa on ties


def test_e2m1_table(orc):
    got = np.array([orc.e2m1_value(n) for n in range(16)])
    assert np.array_equal(got, E2M1_TABLE)
    assert all(math.copysign(1, got[n]) == math.copysign(1, E2M1_TABLE[n]) for n in range(16))


def test_ue8m0_ceil_is_minimal_power_of_two(orc):
    rng = np.random.default_rng(7)
    specials = [0.0, 1.0, 0.75, 1.5, 2.0 ** -127, 2.0 ** -126, 2.0 ** -149, 3 * 2.0 ** -149,
                2.0 ** -127 + 2.0 ** -149, 2.0 ** 120, 7.6e35, 1.0 / 448.0]
    xs = np.concatenate([
        np.array(specials, np.float32),
        (rng.random(3000) * 2.0 ** rng.integers(-149, 121, 3000)).astype(np.float32),
        np.ldexp(np.ones(200), rng.integers(-140, 120, 200)).astype(np.float32),
    ])
    for s in xs:
        s = float(s)
        b = orc.ue8m0_ceil(s)
        assert b != 0xFF
        if s == 0.0:
            assert b == 0
            continue
        fs = Fraction(s)
        assert Fraction(2) ** (b - 127) >= fs, (s, b)
        assert b == 0 or Fraction(2) ** (b - 128) < fs, (s, b)


def test_ue8m0_value(orc):
    assert orc.ue8m0_value(127) == 1.0
    assert orc.ue8m0_value(0) == 2.0 ** -127
    assert orc.ue8m0_value(254) == 2.0 ** 127
    assert math.isnan(orc.ue8m0_value(255))


def test_bf16_from_float_matches_torch(orc):
    rng = np.random.default_rng(9)
    xs = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                         (rng.standard_normal(2000) * 1e30).astype(np.float32),
                         np.array([0.0, -0.0, 3.4e38, -3.4e38, 1e-40], np.float32)])
    ref = f32_to_bf16_torch(xs)
    got = np.array([orc.bf16_from_float(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def _bf16_exact_round(d):
    """Nearest bf16 (ties to even) of a double, by exact rational search."""
    f = np.float32(d)
    u = int(np.array(f, np.float32).view(np.uint32))
    base = (u >> 16) << 16
    cands = [base - 0x10000, base, base + 0x10000, base + 0x20000]
    best = None
    for c in cands:
        c &= 0xFFFFFFFF
        v = np.array(c, np.uint32).view(np.float32)
        if not np.isfinite(v):
            continue
        err = abs(Fraction(float(v)) - Fraction(d))
        key = (err, (c >> 16) & 1)
        if best is None or key < best[0]:
            best = (key, c >> 16)
    return best[1]


def test_bf16_from_double_single_rounding(orc):
    rng = np.random.default_rng(11)
    xs = list(rng.standard_normal(3000) * 10)
    # values just off a bf16 midpoint, where rounding through fp32 would tie
    for _ in range(500):
        hi = int(rng.integers(0x3F80, 0x4100))
        mid = float(np.array(((hi << 16) | 0x8000), np.uint32).view(np.float32))
        xs += [mid + mid * 2.0 ** -40, mid - mid * 2.0 ** -40, mid]
    for d in xs:
        assert orc.bf16_from_double(d) == _bf16_exact_round(d), d
