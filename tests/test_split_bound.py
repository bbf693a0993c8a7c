"""The error bound of the two-term e4m3 activation split used by the tcgen05
decode GEMMs, checked on the CPU: every bf16 value within 2^13 of its group
maximum is represented exactly by hi + lo, and every other value within
2^-21 of the group maximum. The GPU tests use this bound for the tcgen05
decode path; this file emulates the split as its kernel comment defines it
(hi = e4m3(v 2^(127-sh)), r = v - hi 2^(sh-127), lo = e4m3(r 2^(127-sl)),
sh and sl the UE8M0 ceilings of max|v| / 448 and max|r| / 448)."""
import numpy as np
import torch

from moe_expert_ffn_scatter_gb300 import synth
from tests.refs import bf16_bits_to_f64, e4m3_decode_torch

SPLIT_EXACT_RANGE = 2.0 ** 13
SPLIT_ABS_BOUND = 2.0 ** -21


def e4m3_rne_satfinite(v32):
    v = np.clip(np.asarray(v32, np.float32), -448.0, 448.0)
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def split_two_terms(orc, v32):
    """v32 [n, 32] fp32 (bf16 values) -> (hi value, lo value) per element, fp64."""
    a = np.abs(v32).max(axis=1).astype(np.float32)
    sh = np.array([orc.ue8m0_ceil(np.float32(x) / np.float32(448.0)) for x in a], np.int64)
    up_h = (2.0 ** (127 - sh))[:, None].astype(np.float32)
    hi = e4m3_decode_torch(e4m3_rne_satfinite(v32 * up_h))
    hv = (hi * (2.0 ** (sh - 127))[:, None]).astype(np.float32)  # exact
    r = (v32 - hv).astype(np.float32)  # exact
    mr = np.abs(r).max(axis=1).astype(np.float32)
    sl = np.array([orc.ue8m0_ceil(np.float32(x) / np.float32(448.0)) for x in mr], np.int64)
    up_l = (2.0 ** (127 - sl))[:, None].astype(np.float32)
    lo = e4m3_decode_torch(e4m3_rne_satfinite(r * up_l)) * (2.0 ** (sl - 127))[:, None]
    return hv.astype(np.float64), lo


def test_two_term_split_error_bound(orc):
    g = np.random.default_rng(5)
    n = 4000
    # group maxima anywhere in [2^-20, 2^20); the other values log-uniform down
    # to 2^-40 below the maximum, random signs
    top = 2.0 ** g.integers(-20, 20, size=(n, 1)) * g.uniform(1, 2, size=(n, 1))
    rel = 2.0 ** -g.uniform(0, 40, size=(n, 32))
    rel[:, 0] = 1.0
    v = top * rel * g.choice([-1.0, 1.0], size=(n, 32))
    v32 = bf16_bits_to_f64(synth.f32_to_bf16_bits(v.astype(np.float32))).astype(np.float32)
    hi, lo = split_two_terms(orc, v32)
    err = np.abs(v32.astype(np.float64) - (hi + lo))
    amax = np.abs(v32).max(axis=1, keepdims=True).astype(np.float64)
    near = np.abs(v32) >= amax / SPLIT_EXACT_RANGE
    assert np.all(err[near] == 0.0)
    assert np.all(err <= SPLIT_ABS_BOUND * amax)
    assert (~near).sum() > 1000 and (err[~near] > 0).any()
