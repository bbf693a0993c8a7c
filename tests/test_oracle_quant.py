"""Pins for the group-128 e4m3 / UE8M0 quantisation and the SiLU*mul step."""
import math
from fractions import Fraction

import numpy as np
import pytest

from moe_expert_ffn_scatter_gb300 import synth
from tests.refs import bf16_bits_to_f64, e4m3_decode_torch, e4m3_encode_torch, unpack_scale_bytes

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def ref_group_quant(v32, group=128):
    """Group quantisation written from its definition with numpy/torch:
    s = fl32(amax / 448); b = smallest power-of-two exponent with 2^(b-127) >= s;
    codes = RNE_e4m3(v * 2^(127-b)) saturated to 448."""
    v32 = np.asarray(v32, np.float32)
    K = v32.shape[0]
    G = (K + group - 1) // group
    codes = np.zeros(K, np.uint8)
    sf = np.zeros(G, np.uint8)
    for g in range(G):
        blk = v32[g * group:(g + 1) * group]
        fin = blk[~np.isnan(blk)]
        amax = np.float32(np.max(np.abs(fin))) if fin.size else np.float32(0)
        if np.isinf(amax):
            b = 0xFE
        else:
            s = np.float32(amax) / np.float32(448.0)
            if s == 0:
                b = 0
            else:
                fs = Fraction(float(s))
                b = 0
                while Fraction(2) ** (b - 127) < fs:
                    b += 1
        scale = np.float32(math.ldexp(1.0, 127 - b))
        x = (blk * scale).astype(np.float32)
        sat = np.clip(np.nan_to_num(x, nan=0.0, posinf=448.0, neginf=-448.0), -448.0, 448.0)
        c = e4m3_encode_torch(sat)
        c[np.isnan(x)] = 0x7F
        codes[g * group:(g + 1) * group] = c
        sf[g] = b
    return codes, sf


@pytest.mark.parametrize("group", [128, 32])
@pytest.mark.parametrize("seed,scale", [(0, 1.0), (1, 2.0 ** -20), (2, 2.0 ** 30), (3, 1e-38)])
def test_group_quant_matches_definition(orc, seed, scale, group):
    g = np.random.default_rng(seed)
    v = (g.standard_normal(1024) * scale).astype(np.float32)
    codes, sf = orc.group_quant_row(v, group)
    rc, rsf = ref_group_quant(v, group)
    assert np.array_equal(sf, rsf)
    assert np.array_equal(codes, rc)


def test_group_quant_dequant_error_bound(orc):
    g = np.random.default_rng(4)
    v = (g.standard_normal(4096) * 3).astype(np.float32)
    codes, sf = orc.group_quant_row(v)
    deq = e4m3_decode_torch(codes) * np.repeat(np.ldexp(1.0, sf.astype(int) - 127), 128)
    # e4m3 has 3 mantissa bits: relative error <= 2^-4 for normal codes; the
    # subnormal step is 2^-9 * scale
    step = np.repeat(np.ldexp(1.0, sf.astype(int) - 127 - 9), 128)
    assert np.all(np.abs(deq - v) <= np.maximum(np.abs(v) * 2.0 ** -4, step / 2) + 1e-30)
    assert np.all(np.abs(e4m3_decode_torch(codes)) <= 448)


def test_group_quant_special_cases(orc):
    z = np.zeros(128, np.float32)
    c, s = orc.group_quant_row(z)
    assert s[0] == 0 and np.all(c == 0)
    v = np.full(128, 1e-3, np.float32)
    v[5] = np.inf
    v[6] = np.nan
    c, s = orc.group_quant_row(v)
    assert s[0] == 0xFE           # non-finite amax: largest finite UE8M0
    assert c[5] == 0x7E           # saturated
    assert c[6] == 0x7F           # NaN stays NaN
    assert c[0] == 0              # tiny values flush against the huge scale
    v = np.full(128, -2.0, np.float32)
    v[7] = np.nan                 # NaN does not enter the amax
    c, s = orc.group_quant_row(v)
    assert s[0] == orc.ue8m0_ceil(2.0 / 448.0) and c[7] == 0x7F


def test_act_quant_live_rows_only_and_definition(orc):
    """Tiny live-row act-quant: padding rows keep their sentinel; live rows
    equal silu(g)*u computed in fp64 then quantised by the definition above,
    except where fp32 SiLU rounding moves a code by one step."""
    I = 256
    rows = 640
    gateup, counts = synth.actq_inputs(rows=rows, I=I, E=4, live=300, seed=3)
    start, end = orc.endpoints(counts, 128)
    out, out_sf = orc.act_quant(gateup, end, 128)
    live = np.zeros(rows, bool)
    for e in range(4):
        live[start[e]:end[e]] = True
    assert np.all(out[~live] == 0xAB)
    assert np.all(out_sf.view(np.uint32)[:, :rows][:, ~live] == 0xABABABAB)
    sfb = unpack_scale_bytes(out_sf, rows, I // 128)
    mism = 0
    for r in np.nonzero(live)[0]:
        gg = bf16_bits_to_f64(gateup[r, :I])
        uu = bf16_bits_to_f64(gateup[r, I:])
        h = (gg / (1.0 + np.exp(-gg)) * uu).astype(np.float32)
        rc, rsf = ref_group_quant(h)
        assert np.array_equal(sfb[r], rsf) or np.all(np.abs(sfb[r].astype(int) - rsf) <= 1)
        mism += int(np.sum(out[r] != rc))
    assert mism <= 0.002 * live.sum() * I


def test_act_quant_dense_equals_live_when_full(orc):
    I = 128
    rows = 256
    gateup, counts = synth.actq_inputs(rows=rows, I=I, E=2, full=True, seed=5)
    _, end = orc.endpoints(counts, 128)
    a, asf = orc.act_quant(gateup, end, 128)
    d, dsf = orc.act_quant(gateup, None, 128)
    assert np.array_equal(a, d) and np.array_equal(asf, dsf)


def test_act_quant_clamp_semantics(orc):
    """Gate clamped from above only, up on both sides (limit L)."""
    I = 128
    L = 2.0
    gate = np.array([5.0, -5.0, 1.0] + [0.5] * (I - 3), np.float32)
    up = np.array([5.0, -5.0, -9.0] + [0.25] * (I - 3), np.float32)
    row = synth.f32_to_bf16_bits(np.concatenate([gate, up]))[None, :]
    out, sf = orc.act_quant(row, None, 128, clamp=True, limit=L)
    g = np.minimum(gate.astype(np.float64), L)
    u = np.clip(up.astype(np.float64), -L, L)
    h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
    rc, rsf = ref_group_quant(h)
    assert unpack_scale_bytes(sf, 1, 1)[0, 0] == rsf[0]
    assert np.sum(out[0] != rc) <= 1


def test_act_quant_clamp_nan_gate_and_up(orc):
    """A NaN gate or up value, quiet or signalling, is the missing operand of
    min / max: gate NaN -> L, up NaN -> -L (max(NaN, -L) = -L, then min with L).
    The row with NaNs must equal the row with those values replaced."""
    I = 128
    L = 3.0
    g = np.random.default_rng(2)
    base = synth.f32_to_bf16_bits(g.standard_normal(2 * I).astype(np.float32))
    row = base.copy()
    nan_patterns = [0x7FC0, 0xFFC0, 0x7F81, 0xFF93, 0x7FB3, 0xFFBE]  # quiet and signalling
    for j, p in enumerate(nan_patterns):
        row[j] = p              # gate
        row[I + 40 + j] = p     # up
    repl = base.copy()
    repl[:len(nan_patterns)] = synth.f32_to_bf16_bits(np.array([L], np.float32))[0]
    repl[I + 40:I + 40 + len(nan_patterns)] = synth.f32_to_bf16_bits(np.array([-L], np.float32))[0]
    a, asf = orc.act_quant(row[None, :], None, 128, clamp=True, limit=L)
    b, bsf = orc.act_quant(repl[None, :], None, 128, clamp=True, limit=L)
    assert np.array_equal(a, b) and np.array_equal(asf, bsf)


def test_act_quant_situ_against_fp64(orc):
    """SiTU h = (4 tanh(g/4) sigmoid(g)) (25 tanh(u/25)) through the group
    quantisation: scales equal to the fp64 recipe's, codes equal except where
    the fp64 and fp32 products straddle an e4m3 rounding boundary."""
    I = 256
    rng = np.random.default_rng(12)
    vals = (rng.standard_normal((64, 2 * I)) * 3).astype(np.float32)
    row = synth.f32_to_bf16_bits(vals)
    out, sf = orc.act_quant(row, None, 128, situ=(4.0, 25.0))
    g = (row[:, :I].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    u = (row[:, I:].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    h = (4.0 * np.tanh(g / 4.0) / (1.0 + np.exp(-g))) * (25.0 * np.tanh(u / 25.0))
    bad = 0
    for r in range(h.shape[0]):
        rc, rsf = ref_group_quant(h[r].astype(np.float32))
        assert np.array_equal(unpack_scale_bytes(sf, r + 1, 2)[r], rsf[:2])
        bad += int(np.sum(out[r] != rc))
    assert bad <= 0.005 * out.size


def test_scatter_and_act_quant_group32(orc):
    """The MXFP8 activation recipe (group 32): the scattered rows and the
    act-quant output carry one scale per 32 columns, packed four per word,
    each equal to the recipe applied to that 32-column slice."""
    g = np.random.default_rng(17)
    T, E, k, H, A = 16, 3, 2, 256, 128
    x = synth.bf16_normal(g, (T, H))
    ids = synth.ids_with_counts(g, [10, 0, 22], k)
    cap = synth.align_up(T * k + E * (A - 1), A)
    ends, s2d, a, a_sf = orc.scatter(ids, x, E, A, cap, group=32)
    assert a_sf.shape[0] == H // 128
    xv = (x.astype(np.uint32) << 16).view(np.float32)
    for t in range(T):
        rc, rsf = ref_group_quant(xv[t], 32)
        for j in range(k):
            d = s2d[t, j]
            assert np.array_equal(a[d], rc)
            assert np.array_equal(unpack_scale_bytes(a_sf, d + 1, H // 32)[d], rsf)
    I = 256
    gu = synth.bf16_normal(g, (8, 2 * I))
    out, out_sf = orc.act_quant(gu, None, 128, group=32)
    gate = (gu[:, :I].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    up = (gu[:, I:].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    h = (gate / (1.0 + np.exp(-gate)) * up).astype(np.float32)
    for r in range(8):
        rc, rsf = ref_group_quant(h[r], 32)
        assert np.array_equal(unpack_scale_bytes(out_sf, r + 1, I // 32)[r], rsf)
        assert np.sum(out[r] != rc) <= 2

