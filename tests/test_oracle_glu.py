"""Pins for the oracle's decode GLU, as far as the pages fix it.

The DeepGEMM FusedMoE page ([DG] §2.4.1, the clamped SiLU-and-mul branch)
clamps the up half on both sides and the gate half from above only; its list
of runner fields ([DG] §2.1.3) calls gemm1_alpha the scale of the SiLU part of
SwiGLU, so the gate factor is SiLU(alpha g) / alpha = g sigmoid(alpha g). Where
beta enters (u + beta) is a reading that no page fixes."""
import math

import numpy as np
import pytest

from tests.refs import fp32_ulp

ALPHA, BETA, LIMIT = 1.702, 1.0, 7.0


def f32(x):
    return float(np.float32(x))


def test_gate_clamped_from_above_only(orc):
    for u in (f32(-3.25), 0.5, f32(2.75)):
        at_limit = orc.glu_oai(LIMIT, u, ALPHA, BETA, LIMIT)
        for g in (7.5, 9.0, 100.0, math.inf):
            assert orc.glu_oai(g, u, ALPHA, BETA, LIMIT) == at_limit
        # below -L the gate keeps its value: the same as with no limit at all
        for g in (-7.5, -9.0, -30.0):
            clamped = orc.glu_oai(g, u, ALPHA, BETA, LIMIT)
            assert clamped == orc.glu_oai(g, u, ALPHA, BETA, 0.0)
            assert clamped != orc.glu_oai(-LIMIT, u, ALPHA, BETA, LIMIT)


def test_up_clamped_on_both_sides(orc):
    for g in (f32(-1.5), 0.25, f32(3.5), 10.0):
        hi = orc.glu_oai(g, LIMIT, ALPHA, BETA, LIMIT)
        lo = orc.glu_oai(g, -LIMIT, ALPHA, BETA, LIMIT)
        for u in (7.25, 50.0, math.inf):
            assert orc.glu_oai(g, u, ALPHA, BETA, LIMIT) == hi
            assert orc.glu_oai(g, -u, ALPHA, BETA, LIMIT) == lo
        for u in (f32(-6.5), 0.0, f32(6.5)):  # inside the limits nothing changes
            if g <= LIMIT:
                assert orc.glu_oai(g, u, ALPHA, BETA, LIMIT) == orc.glu_oai(g, u, ALPHA, BETA, 0.0)


@pytest.mark.parametrize("alpha", [1.0, ALPHA, 0.5])
def test_alpha_scales_the_silu_part(orc, alpha):
    """With u + beta = 1 the GLU is the gate factor alone, which must be
    SiLU(alpha g) / alpha (the SiLU of the pinned spec, fp64 division)."""
    alpha = f32(alpha)
    g_all = np.concatenate([np.linspace(-20.0, 20.0, 4001), [-1e-3, 1e-3, 0.0]]).astype(np.float32)
    for g in g_all:
        g = float(g)
        act = orc.glu_oai(g, 1.0 - BETA, alpha, BETA, 0.0)
        ref = orc.silu_spec(f32(alpha * g)) / alpha
        assert abs(act - ref) <= 4 * fp32_ulp(ref) + 2.0 ** -140, (alpha, g, act, ref)


def test_zero_gate_and_cancelling_up(orc):
    assert orc.glu_oai(0.0, 3.0, ALPHA, BETA, LIMIT) == 0.0
    assert orc.glu_oai(f32(2.5), -BETA, ALPHA, BETA, LIMIT) == 0.0
