"""Sparse decode GEMV path on the GPU against the oracle: FP8-per-expert and
MXFP4 weights, T in {1, 2, 4, 8}, non-local slots never written and skipped."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_scatter_gb300 import binding as B
from moe_expert_ffn_scatter_gb300 import synth
from tests.gpu_util import check_decode_tolerance, dev, dev_bf16, host_u16
from tests.refs import bf16_bits_to_f64, bf16_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx(cuda_lib):
    return B.Context(0)


_CACHE = {}


def inputs(T, seed=synth.DECODE_SEED):
    """Draw the 8-token decode workload once; smaller T use its first rows."""
    if seed not in _CACHE:
        _CACHE[seed] = synth.decode_inputs(8, seed=seed)
    d = _CACHE[seed]
    return synth.DecodeInputs(d.x[:T], d.logits[:T], d.fp8, d.mxfp4)


def run_decode(ctx, d, ids, w, wfmt, H, I, es, nl, fill=0x7FC0):
    T, k = ids.shape
    W = d.fp8 if wfmt == B.MOE_WFMT_FP8_PER_EXPERT else d.mxfp4
    loc = {kk: v[es:es + nl] for kk, v in W.items()}
    nanfill = lambda shape: torch.full(shape, fill, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    y1, act, y2 = nanfill((T, k, 2 * I)), nanfill((T * k, I)), nanfill((T, k, H))
    out = nanfill((T, H))
    kw = dict(w_gu_scale=dev(loc["gu_scale"]), w_d_scale=dev(loc["d_scale"])) if wfmt == 0 else \
        dict(w_gu_sf=dev(loc["gu_sf"]), w_d_sf=dev(loc["d_sf"]))
    B.moe_sparse_gemv_decode(ctx, x=dev_bf16(d.x), topk_ids=dev(ids), topk_w=dev(w), expert_start=es,
                             num_local_experts=nl, wfmt=wfmt, w_gu=dev(loc["w_gu"]), b_gu=dev_bf16(loc["b_gu"]),
                             w_d=dev(loc["w_d"]), b_d=dev_bf16(loc["b_d"]), y1=y1, act=act, y2=y2, out=out,
                             T=T, H=H, I=I, k=k, **kw)
    torch.cuda.synchronize()
    return host_u16(y1), host_u16(act), host_u16(y2), host_u16(out), loc


@pytest.mark.parametrize("wfmt", [B.MOE_WFMT_FP8_PER_EXPERT, B.MOE_WFMT_MXFP4_G32], ids=["fp8", "mxfp4"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_gpt_oss_shape(ctx, orc, wfmt, T):
    d = inputs(T)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E)
    ry1, ract, ry2, rout = orc.decode(d.x, ids, w, loc, wfmt, I)
    # first GEMV: fp32 accumulation against one fp64 sum
    a, b = bf16_bits_to_f64(y1), bf16_bits_to_f64(ry1)
    assert np.mean(np.abs(a - b) <= bf16_ulp(b) * 1.0001) > 0.99
    check_decode_tolerance(out, rout)


@pytest.mark.parametrize("wfmt", [B.MOE_WFMT_FP8_PER_EXPERT, B.MOE_WFMT_MXFP4_G32], ids=["fp8", "mxfp4"])
def test_decode_expert_parallel_slice_skips_nonlocal(ctx, orc, wfmt):
    """This call owns experts 8..23 only: slots routed elsewhere stay NaN in
    y1/act/y2 and do not reach the output."""
    T = 8
    d = inputs(T, seed=21)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    es, nl = 8, 16
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, es, nl)
    nonlocal_ = (ids < es) | (ids >= es + nl)
    assert np.all(y1[nonlocal_] == 0x7FC0) and np.all(y2[nonlocal_] == 0x7FC0)
    assert np.all(act.reshape(T, -1, I)[nonlocal_] == 0x7FC0)
    assert np.all(np.isfinite(bf16_bits_to_f64(out)))
    _, _, _, rout = orc.decode(d.x, ids, w, loc, wfmt, I, expert_start=es, n_local=nl)
    local_any = ~nonlocal_.all(axis=1)
    check_decode_tolerance(out[local_any], rout[local_any])
