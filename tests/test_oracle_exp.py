"""Pins for the exp / SiLU / sigmoid specification against fp64 math."""
import math

import numpy as np
import pytest

from tests.refs import fp32_ulp

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_exp_spec_error_within_2ulp(orc):
    rng = np.random.default_rng(1)
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001), rng.uniform(-87, 88, 5000),
                         rng.uniform(-1, 1, 5000)]).astype(np.float32)
    for x in xs:
        y = orc.exp_spec(float(x))
        ref = math.exp(float(x))
        assert abs(y - ref) <= 2 * fp32_ulp(ref), (x, y, ref)


def test_exp_spec_special_values(orc):
    assert orc.exp_spec(0.0) == 1.0
    assert orc.exp_spec(128.0) == math.inf
    assert orc.exp_spec(100.0) == math.inf       # overflows fp32
    assert orc.exp_spec(-150.0) == 0.0
    assert math.isnan(orc.exp_spec(float("nan")))
    # gradual underflow region stays close in absolute terms
    for x in np.linspace(-103.0, -87.5, 200).astype(np.float32):
        assert abs(orc.exp_spec(float(x)) - math.exp(float(x))) <= 2.0 ** -148


def all_finite_bf16():
    u = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    return u[np.isfinite(u)]


def test_silu_spec_all_bf16(orc):
    for g in all_finite_bf16()[::3]:
        g = float(g)
        y = orc.silu_spec(g)
        if g < -87:
            # exp(-g) overflows fp32, so g / (1 + exp(-g)) flushes to -0;
            # the true value is below 2^-118 in magnitude
            assert abs(y - g * math.exp(g)) <= 2.0 ** -118
            continue
        if g > 100:
            assert y == g
            continue
        ref = g / (1.0 + math.exp(-g))
        assert abs(y - ref) <= 3 * fp32_ulp(ref) + 2.0 ** -149, (g, y, ref)


def test_sigmoid_spec(orc):
    for x in np.linspace(-80, 80, 4001).astype(np.float32):
        x = float(x)
        ref = 1.0 / (1.0 + math.exp(-x))
        assert abs(orc.sigmoid_spec(x) - ref) <= 3 * fp32_ulp(ref) + 2.0 ** -149
