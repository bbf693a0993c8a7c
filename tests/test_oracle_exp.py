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


# ------------------------------------------------------------------ tanh / SiTU
def tanh_sweep():
    rng = np.random.default_rng(7)
    parts = [rng.uniform(2.0 ** -20, 2.0 ** -12, 500), rng.uniform(2.0 ** -12, 0.25, 4000),
             np.linspace(0.2, 0.3, 2001), rng.uniform(0.25, 9.0, 4000), np.linspace(8.5, 12.0, 501)]
    xs = np.concatenate(parts).astype(np.float32)
    return np.concatenate([xs, -xs])


def test_tanh_spec_error_within_4ulp(orc):
    """Each branch of the definition (identity, Taylor polynomial, exp form,
    saturation) against fp64 tanh; a wrong coefficient, sign or threshold in
    any branch moves the error far past 4 ulp."""
    for x in tanh_sweep():
        y = orc.tanh_spec(float(x))
        ref = math.tanh(float(x))
        assert abs(y - ref) <= 4 * fp32_ulp(ref), (x, y, ref)


def test_tanh_spec_odd_monotone_special(orc):
    xs = np.sort(np.abs(tanh_sweep()))
    ys = np.array([orc.tanh_spec(float(x)) for x in xs])
    assert np.all(np.diff(ys) >= 0)
    for x in xs[::7]:
        assert orc.tanh_spec(-float(x)) == -orc.tanh_spec(float(x))
    assert orc.tanh_spec(0.0) == 0.0 and math.copysign(1.0, orc.tanh_spec(-0.0)) == -1.0
    assert orc.tanh_spec(math.inf) == 1.0 and orc.tanh_spec(-math.inf) == -1.0
    assert math.isnan(orc.tanh_spec(math.nan))
    assert orc.tanh_spec(1e-5) == np.float32(1e-5)  # below 2^-12 tanh y rounds to y


def test_situ_specs_against_fp64(orc):
    """gate' = 4 tanh(g/4) sigmoid(g), up' = 25 tanh(u/25): within 6 ulp of the
    fp64 formula over all finite bf16 inputs of moderate size."""
    vals = all_finite_bf16()
    vals = vals[np.abs(vals) < 80]
    for g in vals[::5]:
        g = float(g)
        ref = 4.0 * math.tanh(g / 4.0) / (1.0 + math.exp(-g))
        got = orc.situ_gate_spec(g, 4.0)
        assert abs(got - ref) <= 6 * fp32_ulp(ref) + 1e-40, (g, got, ref)
        ref_u = 25.0 * math.tanh(g / 25.0)
        got_u = orc.situ_up_spec(g, 25.0)
        assert abs(got_u - ref_u) <= 6 * fp32_ulp(ref_u) + 1e-40, (g, got_u, ref_u)
    assert orc.situ_gate_spec(math.inf, 4.0) == 4.0
    assert orc.situ_gate_spec(-math.inf, 4.0) == 0.0
    assert orc.situ_up_spec(math.inf, 25.0) == 25.0 and orc.situ_up_spec(-math.inf, 25.0) == -25.0
