"""Grouped block-scaled GEMM, combine and the whole layer on the GPU against
the oracle."""
import os

import numpy as np
import pytest
import torch

from moe_expert_ffn_scatter_gb300 import binding as B
from moe_expert_ffn_scatter_gb300 import synth
from moe_expert_ffn_scatter_gb300.layer import MoEFFNLayer
from tests.gpu_util import check_ffn_tolerance, dev, dev_bf16, filled, host, host_u16
from tests.refs import (bf16_bits_to_f64, bf16_ulp, e2m1_decode, e4m3_decode_torch, e4m3_encode_torch,
                        unpack_scale_bytes)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx(cuda_lib):
    return B.Context(0)


def prepared(ctx, w, w_sf, fmt):
    E, N, K2 = w.shape
    K = 2 * K2
    w_in = dev(w)
    w_out = torch.empty((E, N, K), dtype=torch.uint8, device="cuda") if fmt == B.MOE_GEMM_W_E4M3 else w_in
    sf_out = torch.empty((E, K // 128, N), dtype=torch.int32, device="cuda")
    B.moe_prepare_weights(ctx, w_in, dev(w_sf), E, N, K, fmt, w_out, sf_out)
    return w_out, sf_out


def gemm_case(ctx, orc, counts, N, K, fmt, seed=0, cap=None):
    g = np.random.default_rng(seed)
    E = len(counts)
    counts = np.array(counts, np.int32)
    _, ends = orc.endpoints(counts, 128)
    cap = cap or synth.align_up(max(int(ends[-1]), 128), 128)
    ld = synth.align4(cap)
    a = synth.e4m3_codes(g, (cap, K), exp_lo=1, exp_hi=14)
    sfb = synth.ue8m0_bytes(g, (cap, K // 128), -3, 3)
    a_sf = synth.pack_scale_words(sfb, ld)
    w = synth.e2m1_packed(g, (E, N, K // 2))
    w_sf = synth.ue8m0_bytes(g, (E, N, K // 32))
    wd, wsfd = prepared(ctx, w, w_sf, fmt)
    out = filled((cap, N), 0xAB, torch.int16)
    B.moe_grouped_gemm(ctx, dev(a), dev(a_sf), ld, dev(ends), E, 128, cap, wd, wsfd, fmt, N, K, out)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    got = host_u16(out)
    ref = orc.grouped_gemm(a, a_sf, ends, 128, w, w_sf, out=np.full((cap, N), 0xABAB, np.uint16))
    # sum of |products| per output, for the fp32 accumulation error bound
    ad = np.abs(e4m3_decode_torch(a)) * np.repeat(np.ldexp(1.0, sfb.astype(int) - 127), 128, axis=1)
    wd = np.abs(e2m1_decode(w, K)) * np.repeat(np.ldexp(1.0, w_sf.astype(int) - 127), 32, axis=2)
    start = np.concatenate([[0], (ends[:-1] + 127) // 128 * 128])
    abssum = np.zeros((cap, N))
    for e in range(E):
        abssum[start[e]:ends[e]] = ad[start[e]:ends[e]] @ wd[e].T
    return got, ref, ends, abssum


def live_rows(ends, rows):
    start = np.concatenate([[0], (ends[:-1] + 127) // 128 * 128])
    live = np.zeros(rows, bool)
    for s, e in zip(start, ends):
        live[s:e] = True
    return live


def assert_gemm_close(got, ref, ends, abssum=None, sentinel=0xABAB):
    """fp32 tensor-core accumulation vs one fp64 sum: within one bf16 step of
    the reference plus the fp32 summation bound K * 2^-24 * sum|products|
    (taken as 2^-18 * sum|products|, K <= 4096)."""
    live = live_rows(ends, got.shape[0])
    if sentinel is not None:
        assert np.all(got[~live] == sentinel), "padding rows written"
    g = bf16_bits_to_f64(got[live])
    r = bf16_bits_to_f64(ref[live])
    bound = bf16_ulp(r) * 1.0001 + 1e-30
    if abssum is not None:
        bound = bound + 2.0 ** -18 * abssum[live]
    bad = np.abs(g - r) > bound
    assert not bad.any(), "%d of %d elements outside the bound" % (bad.sum(), bad.size)
    return np.mean(got[live] == ref[live])


@pytest.mark.parametrize("fmt", [B.MOE_GEMM_W_E2M1, B.MOE_GEMM_W_E4M3], ids=["e2m1", "e4m3"])
def test_gemm_single_tile(ctx, orc, fmt):
    got, ref, ends, ab = gemm_case(ctx, orc, [128], 256, 128, fmt)
    assert assert_gemm_close(got, ref, ends, ab) > 0.99


@pytest.mark.parametrize("fmt", [B.MOE_GEMM_W_E2M1, B.MOE_GEMM_W_E4M3], ids=["e2m1", "e4m3"])
def test_gemm_ragged_experts(ctx, orc, fmt):
    # several M tiles per expert, an empty expert, ragged tails, K with a
    # partial group of four 128-blocks (K=640 -> scale words 0 and 1)
    got, ref, ends, ab = gemm_case(ctx, orc, [5, 0, 300, 129, 1], 512, 640, fmt, seed=1)
    assert assert_gemm_close(got, ref, ends, ab) > 0.99


def test_gemm_formats_agree_bitwise(ctx, orc):
    g1 = gemm_case(ctx, orc, [200, 77], 256, 384, B.MOE_GEMM_W_E2M1, seed=3)[0]
    g2 = gemm_case(ctx, orc, [200, 77], 256, 384, B.MOE_GEMM_W_E4M3, seed=3)[0]
    assert np.array_equal(g1, g2)


def test_gemm_many_tiles_persistent(ctx, orc):
    """More tiles than SMs: every CTA loops over several tiles."""
    counts = [700, 650, 0, 900, 810, 333]
    got, ref, ends, ab = gemm_case(ctx, orc, counts, 1024, 256, B.MOE_GEMM_W_E2M1, seed=4)
    assert assert_gemm_close(got, ref, ends, ab) > 0.99


def test_gemm_more_experts_than_the_shared_endpoint_copy(ctx, orc):
    """E = 1100: the tile search reads the endpoints from global memory (the
    shared copy holds 1024); live experts on both sides of index 1024."""
    counts = np.zeros(1100, np.int32)
    counts[[3, 1023, 1024, 1099]] = [40, 130, 1, 77]
    got, ref, ends, ab = gemm_case(ctx, orc, counts, 256, 128, B.MOE_GEMM_W_E2M1, seed=6)
    assert assert_gemm_close(got, ref, ends, ab) > 0.99


def test_gemm_no_live_rows(ctx, orc):
    got = gemm_case(ctx, orc, [0, 0], 256, 128, B.MOE_GEMM_W_E2M1, cap=256)[0]
    assert np.all(got == 0xABAB)


@pytest.mark.parametrize("recipe", ["mxfp8", "fp8_block128"])
def test_gemm_fp8_weight_recipes(ctx, orc, recipe):
    """FP8 weights ([DG] §6 recipes): e4m3 with per-32 scales and group-32 A
    scales (MXFP8), or with 128 x 128 block scales (FP8 block128), prepared
    from their canonical layouts; against the oracle within the fp32
    accumulation bound, padding rows untouched."""
    g = np.random.default_rng(21)
    E, N, K = 3, 512, 512
    counts = np.array([150, 0, 77], np.int32)
    _, ends = orc.endpoints(counts, 128)
    cap = synth.align_up(int(ends[-1]), 128)
    group = 32 if recipe == "mxfp8" else 128
    ld = synth.align4(cap)
    a = synth.e4m3_codes(g, (cap, K), exp_lo=1, exp_hi=14)
    sfb = synth.ue8m0_bytes(g, (cap, K // group), -3, 3)
    a_sf = synth.pack_scale_words(sfb, ld)
    w = synth.e4m3_codes(g, (E, N, K))
    if recipe == "mxfp8":
        w_sf_in = synth.ue8m0_bytes(g, (E, N, K // 32))
        w_sf = w_sf_in
        flags = B.MOE_GEMM_W_IN_E4M3
    else:
        w_sf_in = synth.ue8m0_bytes(g, (E, N // 128, K // 128))
        w_sf = orc.expand_block_scales(w_sf_in, N, K)
        flags = B.MOE_GEMM_W_IN_E4M3 | B.MOE_GEMM_W_SF_BLOCK128
    wd = dev(w)
    sf_out = torch.empty((E, K // 128, N), dtype=torch.int32, device="cuda")
    B.moe_prepare_weights(ctx, wd, dev(w_sf_in), E, N, K, B.MOE_GEMM_W_E4M3 | flags, wd, sf_out)
    out = filled((cap, N), 0xAB, torch.int16)
    fmt = B.MOE_GEMM_W_E4M3 | (B.MOE_GEMM_A_GROUP32 if group == 32 else 0)
    B.moe_grouped_gemm(ctx, dev(a), dev(a_sf), ld, dev(ends), E, 128, cap, wd, sf_out, fmt, N, K, out)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    got = host_u16(out)
    ref = orc.grouped_gemm(a, a_sf, ends, 128, w, w_sf, out=np.full((cap, N), 0xABAB, np.uint16), a_group=group,
                           wfmt=1)
    ad = np.abs(e4m3_decode_torch(a)) * np.repeat(np.ldexp(1.0, sfb.astype(int) - 127), group, axis=1)
    wabs = np.abs(e4m3_decode_torch(w)) * np.repeat(np.ldexp(1.0, w_sf.astype(int) - 127), 32, axis=2)
    start = np.concatenate([[0], (ends[:-1] + 127) // 128 * 128])
    abssum = np.zeros((cap, N))
    for e in range(E):
        abssum[start[e]:ends[e]] = ad[start[e]:ends[e]] @ wabs[e].T
    assert_gemm_close(got, ref, ends, abssum)


def context_with_pairs(n):
    """A context whose grouped GEMM always runs the two-SM kernel with at most
    n CTA pairs (n = 0: always the one-CTA kernel), through
    MOE_GEMM_CTA_PAIRS, read at context creation."""
    old = os.environ.get("MOE_GEMM_CTA_PAIRS")
    os.environ["MOE_GEMM_CTA_PAIRS"] = str(n)
    try:
        return B.Context(0)
    finally:
        if old is None:
            del os.environ["MOE_GEMM_CTA_PAIRS"]
        else:
            os.environ["MOE_GEMM_CTA_PAIRS"] = old


@pytest.mark.parametrize("fmt", [B.MOE_GEMM_W_E2M1, B.MOE_GEMM_W_E4M3], ids=["e2m1", "e4m3"])
def test_pair_kernel_equals_one_cta_kernel(ctx, orc, fmt):
    """The two-SM kernel (cta_group::2, as many pairs as fit, and capped at two
    pairs so that each pair loops over many tiles and wraps its stage ring)
    and the one-CTA kernel give the same bits, within the oracle's bound:
    experts whose last 256-row tile holds 128 rows or fewer (the odd CTA's
    rows past the expert's end), exactly 256 and 257 rows, an empty expert,
    K with a partial group of four 128-blocks."""
    counts = [5, 0, 300, 129, 1, 256, 257, 128, 384]
    outs = []
    for c in (context_with_pairs(1000), context_with_pairs(2), context_with_pairs(0)):
        got, ref, ends, ab = gemm_case(c, orc, counts, 768, 640, fmt, seed=8)
        assert_gemm_close(got, ref, ends, ab)
        outs.append(got)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("act", ["silu", "silu_clamp", "situ"])
def test_pair_kernel_fused_layer_equals_one_cta_kernel(orc, act):
    """The whole layer (fused GEMM1 epilogue, GEMM2) through the two-SM kernel
    and through the one-CTA kernel: codes, scale words and output bit for bit."""
    clamp = act == "silu_clamp"
    kind = {"silu": B.MOE_ACT_SILU, "silu_clamp": B.MOE_ACT_SILU_CLAMP, "situ": B.MOE_ACT_SITU}[act]
    cfg = synth.FFNConfig("pair", T=900, E=7, k=3, H=512, I=512, seed=23, clamp=clamp, limit=2.5 if clamp else 0.0)
    inp = synth.ffn_inputs(cfg)
    res = []
    for n in (1000, 3, 0):
        c = context_with_pairs(n)
        layer = make_layer(c, cfg, inp, act_kind=kind)
        layer.act_fp8.fill_(0xAB)
        layer.act_sf.view(torch.uint8).fill_(0xAB)
        layer.forward(dev_bf16(inp.x), dev(inp.logits))
        torch.cuda.synchronize()
        assert B.moe_get_device_error(c) == 0
        res.append((host(layer.act_fp8).copy(), host(layer.act_sf).copy(), host_u16(layer.out).copy()))
    for r in res[1:]:
        for a_, b_ in zip(res[0], r):
            assert np.array_equal(a_, b_)
    ids, w = oracle_layer(orc, cfg, inp)
    toks = np.arange(0, cfg.T, 7, dtype=np.int32)
    ref = orc.ffn_tokens(inp.x, ids, w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf, toks, clamp=clamp, limit=cfg.limit,
                         situ=(4.0, 25.0) if act == "situ" else None)
    check_ffn_tolerance(res[0][2][toks], ref)


def test_combine_bit_exact(ctx, orc):
    g = np.random.default_rng(6)
    T, k, H, rows = 333, 6, 4096, 2500
    down = synth.bf16_normal(g, (rows, H))
    s2d = g.permutation(rows)[:T * k].reshape(T, k).astype(np.int32)
    s2d[g.random((T, k)) < 0.05] = -1
    w = g.random((T, k)).astype(np.float32)
    down[s2d.max() + 1:] = 0x7FC0  # rows that no slot references are NaN
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    B.moe_combine(ctx, dev_bf16(down), H, dev(w), dev(s2d), T, k, 1.25, out)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), orc.combine(down, w, s2d, rsf=1.25))


# ------------------------------------------------------------ whole layer
def make_layer(ctx, cfg, inp, fmt=B.MOE_GEMM_W_E2M1, fused=True, act_kind=None, recipe="mxfp4"):
    routing = B.MOE_ROUTE_SIGMOID_BIAS_TOPK if cfg.routing == "sigmoid_bias" else B.MOE_ROUTE_SOFTMAX_TOPK
    if act_kind is None:
        act_kind = B.MOE_ACT_SILU_CLAMP if cfg.clamp else B.MOE_ACT_SILU
    layer = MoEFFNLayer(ctx, T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap, routing=routing,
                        act_kind=act_kind, limit=cfg.limit, rsf=cfg.rsf, w_format=fmt, fused=fused, recipe=recipe)
    if recipe == "mxfp8":  # the same values as e4m3 codes with their per-32 scales
        w13 = e4m3_encode_torch(e2m1_decode(inp.w13, cfg.H).astype(np.float32))
        w2 = e4m3_encode_torch(e2m1_decode(inp.w2, cfg.I).astype(np.float32))
        layer.load_weights(w13, inp.w13_sf, w2, inp.w2_sf)
    else:
        layer.load_weights(inp.w13, inp.w13_sf, inp.w2, inp.w2_sf)
    return layer


def oracle_layer(orc, cfg, inp):
    if cfg.routing == "sigmoid_bias":
        ids, w = orc.route_sigmoid_bias_topk(inp.logits, inp.bias, cfg.k)
    else:
        ids, w = orc.route_softmax_topk(inp.logits, cfg.k)
    return ids, w


@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
def test_tiny_layer_vs_oracle(ctx, orc, fused):
    cfg = synth.TINY
    inp = synth.ffn_inputs(cfg)
    layer = make_layer(ctx, cfg, inp, fused=fused)
    bufs = [b for b in (layer.gateup, layer.act_fp8, layer.down, layer.a_fp8) if b is not None]
    for buf in bufs:
        buf.view(torch.uint8).fill_(0xAB)
    out = layer.forward(dev_bf16(inp.x), dev(inp.logits))
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    ids, w = oracle_layer(orc, cfg, inp)
    ends, s2d, a, a_sf = orc.scatter(ids, inp.x, cfg.E, cfg.A, cfg.cap)
    live = live_rows(ends, cfg.cap)
    for buf in bufs:
        assert np.all(host(buf.view(torch.uint8))[~live] == 0xAB), "padding rows written"
    assert np.array_equal(host(layer.expert_ends), ends)
    assert np.array_equal(host(layer.src2dst), s2d)
    gu = orc.grouped_gemm(a, a_sf, ends, cfg.A, inp.w13, inp.w13_sf)
    act, act_sf = orc.act_quant(gu, ends, cfg.A)
    down = orc.grouped_gemm(act, act_sf, ends, cfg.A, inp.w2, inp.w2_sf)
    ref = orc.combine(down, w, s2d, rsf=cfg.rsf)
    if not fused:
        assert_gemm_close(host_u16(layer.gateup), gu, ends, sentinel=None)
    check_ffn_tolerance(host_u16(out), ref)


@pytest.mark.parametrize("act", ["silu", "silu_clamp", "situ", "silu_group32"])
@pytest.mark.parametrize("fmt", [B.MOE_GEMM_W_E2M1, B.MOE_GEMM_W_E4M3], ids=["e2m1", "e4m3"])
def test_fused_act_quant_equals_separate_kernel(ctx, act, fmt):
    """GEMM1 with SiLU*mul + quant in its epilogue gives bit for bit what
    GEMM1 -> bf16 gate/up -> act-quant gives: codes, packed scales (including
    the zero bytes of the last word when I/128 is not a multiple of 4) and the
    layer output. I = 384: three groups of 128."""
    clamp = act == "silu_clamp"
    kind = {"silu": B.MOE_ACT_SILU, "silu_clamp": B.MOE_ACT_SILU_CLAMP, "situ": B.MOE_ACT_SITU,
            "silu_group32": B.MOE_ACT_SILU}[act]
    recipe = "mxfp8" if act == "silu_group32" else "mxfp4"
    cfg = synth.FFNConfig("fused", T=700, E=6, k=3, H=512, I=384, seed=14, clamp=clamp,
                          limit=2.5 if clamp else 0.0)
    inp = synth.ffn_inputs(cfg)
    res = []
    for fused in (False, True):
        layer = make_layer(ctx, cfg, inp, fmt=fmt, fused=fused, act_kind=kind, recipe=recipe)
        layer.act_fp8.fill_(0xAB)
        layer.act_sf.view(torch.uint8).fill_(0xAB)
        layer.forward(dev_bf16(inp.x), dev(inp.logits))
        torch.cuda.synchronize()
        assert B.moe_get_device_error(ctx) == 0
        res.append((host(layer.act_fp8).copy(), host(layer.act_sf).copy(), host_u16(layer.out).copy(),
                    host(layer.expert_ends).copy()))
    (a0, s0, o0, e0), (a1, s1, o1, e1) = res
    assert np.array_equal(e0, e1)
    assert np.array_equal(a0, a1)
    assert np.array_equal(s0, s1)
    assert np.array_equal(o0, o1)
    live = live_rows(e0, cfg.cap)
    assert np.all(a1[~live] == 0xAB)


@pytest.mark.parametrize("act", ["silu", "silu_clamp", "situ"])
def test_fused_silu_across_gate_magnitudes(ctx, act):
    """The fused epilogue reads SiLU from a shared-memory window for
    |g| in [2^-6, 2^6) and from the full table otherwise (SiTU reads its
    tables in global memory). Weight rows scaled by
    2^-24 .. 2^8 put gate values below, inside and above the window; the fused
    layer must still equal the unfused one (GEMM1 -> bf16 -> act-quant) bit for
    bit."""
    clamp = act == "silu_clamp"
    cfg = synth.FFNConfig("gate range", T=512, E=4, k=2, H=256, I=256, seed=21, clamp=clamp,
                          limit=2.5 if clamp else 0.0)
    inp = synth.ffn_inputs(cfg)
    g = np.random.default_rng(22)
    row_exp = g.integers(-24, 9, size=(cfg.E, 2 * cfg.I, 1))
    w13_sf = np.broadcast_to(127 + row_exp, inp.w13_sf.shape).astype(np.uint8).copy()
    inp = type(inp)(inp.x, inp.logits, inp.bias, inp.w13, w13_sf, inp.w2, inp.w2_sf)
    res = []
    for fused in (False, True):
        layer = make_layer(ctx, cfg, inp, fused=fused, act_kind=B.MOE_ACT_SITU if act == "situ" else None)
        layer.act_fp8.fill_(0xAB)
        layer.act_sf.view(torch.uint8).fill_(0xAB)
        layer.forward(dev_bf16(inp.x), dev(inp.logits))
        torch.cuda.synchronize()
        assert B.moe_get_device_error(ctx) == 0
        if not fused:
            ends = host(layer.expert_ends).copy()
            gate = bf16_bits_to_f64(host_u16(layer.gateup)[live_rows(ends, cfg.cap), :cfg.I])
            mag = np.abs(gate[gate != 0])
            assert (mag < 2.0 ** -6).any() and (mag >= 2.0 ** 6).any()
            assert ((mag >= 2.0 ** -6) & (mag < 2.0 ** 6)).any()
        res.append((host(layer.act_fp8).copy(), host(layer.act_sf).copy(), host_u16(layer.out).copy()))
    for a, b in zip(*res):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("recipe", ["mxfp8", "fp8_block128"])
@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
def test_tiny_layer_fp8_recipes_vs_oracle(ctx, orc, recipe, fused):
    """The whole layer under the FP8 recipes of [DG] §6."""
    cfg = synth.FFNConfig("tiny fp8", T=96, E=4, k=2, H=256, I=256, seed=18)
    inp = synth.ffn_inputs(cfg, weights=False)
    g = np.random.default_rng(19)
    w13 = synth.e4m3_codes(g, (cfg.E, 2 * cfg.I, cfg.H))
    w2 = synth.e4m3_codes(g, (cfg.E, cfg.H, cfg.I))
    if recipe == "mxfp8":
        w13_sf = synth.ue8m0_bytes(g, (cfg.E, 2 * cfg.I, cfg.H // 32))
        w2_sf = synth.ue8m0_bytes(g, (cfg.E, cfg.H, cfg.I // 32))
        w13_sf32, w2_sf32 = w13_sf, w2_sf
    else:
        w13_sf = synth.ue8m0_bytes(g, (cfg.E, 2 * cfg.I // 128, cfg.H // 128))
        w2_sf = synth.ue8m0_bytes(g, (cfg.E, cfg.H // 128, cfg.I // 128))
        w13_sf32 = orc.expand_block_scales(w13_sf, 2 * cfg.I, cfg.H)
        w2_sf32 = orc.expand_block_scales(w2_sf, cfg.H, cfg.I)
    layer = MoEFFNLayer(ctx, T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap, recipe=recipe,
                        fused=fused)
    layer.load_weights(w13, w13_sf, w2, w2_sf)
    out = layer.forward(dev_bf16(inp.x), dev(inp.logits))
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    ids, w = orc.route_softmax_topk(inp.logits, cfg.k)
    group = 32 if recipe == "mxfp8" else 128
    ref = orc.ffn_tokens(inp.x, ids, w, w13, w13_sf32, w2, w2_sf32, np.arange(cfg.T, dtype=np.int32), wfmt=1,
                         group=group)
    check_ffn_tolerance(host_u16(out), ref)


def test_fused_layer_with_more_experts_than_the_shared_endpoint_copy(ctx, orc):
    """E = 1100 experts (the GEMM's shared endpoint copy holds 1024, so the tile
    search reads global memory), routing given for experts on both sides of
    index 1024: the fused layer equals the unfused one bit for bit, and its
    output stays within the FFN tolerance of the oracle."""
    E, T, k, H, I = 1100, 64, 2, 256, 128
    g = np.random.default_rng(31)
    pool = np.array([5, 600, 1023, 1024, 1050, 1099], np.int32)
    ids = np.stack([g.choice(pool, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = g.uniform(0.2, 1.0, size=(T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    x = synth.bf16_normal(g, (T, H))
    w13 = synth.e2m1_packed(g, (E, 2 * I, H // 2))
    w13_sf = synth.ue8m0_bytes(g, (E, 2 * I, H // 32))
    w2 = synth.e2m1_packed(g, (E, H, I // 2))
    w2_sf = synth.ue8m0_bytes(g, (E, H, I // 32))
    res = []
    for fused in (False, True):
        layer = MoEFFNLayer(ctx, T=T, E=E, k=k, H=H, I=I, routing=B.MOE_ROUTE_PRECOMPUTED, fused=fused)
        layer.load_weights(w13, w13_sf, w2, w2_sf)
        layer.topk_ids.copy_(torch.from_numpy(ids))
        layer.topk_w.copy_(torch.from_numpy(w))
        layer.act_fp8.fill_(0xAB)
        layer.act_sf.view(torch.uint8).fill_(0xAB)
        out = layer.forward(dev_bf16(x))
        torch.cuda.synchronize()
        assert B.moe_get_device_error(ctx) == 0
        res.append((host(layer.act_fp8).copy(), host(layer.act_sf).copy(), host_u16(out).copy()))
    for a_, b_ in zip(*res):
        assert np.array_equal(a_, b_)
    ref = orc.ffn_tokens(x, ids, w, w13, w13_sf, w2, w2_sf, np.arange(T, dtype=np.int32))
    check_ffn_tolerance(res[1][2], ref)


def test_tiny_layer_situ_vs_oracle(ctx, orc):
    """Layer with the SiTU activation ([DG] §2.4.1), fused GEMM1 epilogue."""
    cfg = synth.FFNConfig("tiny situ", T=64, E=4, k=2, H=256, I=128, seed=16)
    inp = synth.ffn_inputs(cfg)
    layer = make_layer(ctx, cfg, inp, act_kind=B.MOE_ACT_SITU)
    out = layer.forward(dev_bf16(inp.x), dev(inp.logits))
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    ids, w = oracle_layer(orc, cfg, inp)
    ref = orc.ffn_tokens(inp.x, ids, w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf,
                         np.arange(cfg.T, dtype=np.int32), situ=(4.0, 25.0))
    check_ffn_tolerance(host_u16(out), ref)


def sampled_rows_gemm(orc, a, a_sf_words, ends, rows, w, w_sf, K, a_group=128):
    """The oracle's grouped GEMM on selected live rows of a full-size buffer:
    the rows are regrouped by expert into a small endpoint layout (with their
    scale words) and multiplied by their experts' weights. Returns the
    oracle's outputs in the order of `rows` and the sum of |products| of each
    output (the fp32 accumulation bound)."""
    E = ends.shape[0]
    start = np.concatenate([[0], (ends[:-1] + 127) // 128 * 128])
    exp_of = np.searchsorted(ends, rows, side="right")
    assert np.all((rows >= start[exp_of]) & (rows < ends[exp_of]))
    order = np.argsort(exp_of, kind="stable")
    counts = np.bincount(exp_of, minlength=E).astype(np.int32)
    _, ends_s = orc.endpoints(counts, 128)
    start_s = np.concatenate([[0], (ends_s[:-1] + 127) // 128 * 128])
    cap_s = synth.align_up(max(int(ends_s[-1]), 128), 128)
    ld_s = synth.align4(cap_s)
    pos = np.empty(rows.shape[0], np.int64)
    seen = np.zeros(E, np.int64)
    for i in order:
        e = exp_of[i]
        pos[i] = start_s[e] + seen[e]
        seen[e] += 1
    a_s = np.zeros((cap_s, K), np.uint8)
    a_s[pos] = a[rows]
    sf_s = np.zeros((a_sf_words.shape[0], ld_s), np.int32)
    sf_s[:, pos] = a_sf_words[:, rows]
    N = w.shape[1]
    ref = orc.grouped_gemm(a_s, sf_s, ends_s, 128, w, w_sf)[pos]
    G = K // a_group
    sfb = unpack_scale_bytes(sf_s, cap_s, G)[pos].astype(np.int64)
    ad = np.abs(e4m3_decode_torch(a[rows])) * np.repeat(2.0 ** (sfb - 127), a_group, axis=1)
    abssum = np.zeros((rows.shape[0], N))
    for e in np.unique(exp_of):
        sel = exp_of == e
        wd = np.abs(e2m1_decode(w[e], K)) * np.repeat(2.0 ** (w_sf[e].astype(np.int64) - 127), 32, axis=1)
        abssum[sel] = ad[sel] @ wd.T
    return ref, abssum


def assert_rows_close(got, ref, abssum):
    g = bf16_bits_to_f64(got)
    r = bf16_bits_to_f64(ref)
    bad = np.abs(g - r) > bf16_ulp(r) * 1.0001 + 2.0 ** -18 * abssum + 1e-30
    assert not bad.any(), "%d of %d elements outside the bound" % (bad.sum(), bad.size)


def test_deepseek_layer_full_size(ctx, orc):
    """The DeepSeek-style layer (E = 32, top-6, T = 4,096, H = 4,096,
    I = 2,048, capacity 28,672) at full size, unfused and fused:
      - routing, endpoints and src2dst equal the oracle's;
      - every live row's act-quant (e4m3 codes and packed UE8M0 words) equals
        the oracle's act-quant of the GPU's own gate/up buffer, bit for bit
        (all 24,576 live rows);
      - the fused layer (SiLU*mul + quantisation in GEMM1's epilogue) gives
        the unfused layer's codes, scale words and output bit for bit, and
        leaves every padding row's sentinel;
      - GEMM1 and GEMM2 on 256 sampled live rows each: within one bf16 step
        plus the fp32 summation bound of the oracle's GEMM of the GPU's own
        input rows;
      - 256 sampled tokens of the output within the layer tolerance of the
        oracle's whole layer."""
    cfg = synth.DEEPSEEK
    inp = synth.ffn_inputs(cfg)
    res = {}
    for fused in (False, True):
        layer = make_layer(ctx, cfg, inp, fused=fused)
        layer.act_fp8.fill_(0xAB)
        layer.act_sf.view(torch.uint8).fill_(0xAB)
        layer.down.view(torch.uint8).fill_(0xAB)
        out = layer.forward(dev_bf16(inp.x), dev(inp.logits))
        torch.cuda.synchronize()
        assert B.moe_get_device_error(ctx) == 0
        r = dict(act=host(layer.act_fp8).copy(), sf=host(layer.act_sf).copy(), out=host_u16(out).copy(),
                 ends=host(layer.expert_ends).copy(), ids=host(layer.topk_ids).copy(),
                 s2d=host(layer.src2dst).copy(), down=host_u16(layer.down).copy())
        if not fused:
            r["gateup"] = host_u16(layer.gateup).copy()
            r["a"] = host(layer.a_fp8).copy()
            r["a_sf"] = host(layer.a_sf).copy()
        res[fused] = r
        del layer, out
        torch.cuda.empty_cache()
    u, f = res[False], res[True]
    ids, w = oracle_layer(orc, cfg, inp)
    ends, s2d, _, _ = orc.scatter(ids, inp.x, cfg.E, cfg.A, cfg.cap)
    for r in (u, f):
        assert np.array_equal(r["ids"], ids)
        assert np.array_equal(r["ends"], ends)
        assert np.array_equal(r["s2d"], s2d)
    live = live_rows(ends, cfg.cap)
    assert live.sum() == cfg.R
    # act-quant of every live row from the GPU's gate/up
    ract, rsf = orc.act_quant(u["gateup"], ends, cfg.A)
    assert np.array_equal(u["act"][live], ract[live])
    assert np.array_equal(u["sf"][:, :cfg.cap][:, live], rsf[:, :cfg.cap][:, live])
    # fused == unfused, sentinels intact
    for key in ("act", "sf", "out"):
        assert np.array_equal(f[key], u[key]), key
    assert np.all(f["act"][~live] == 0xAB)
    assert np.all(f["sf"].view(np.uint8).reshape(f["sf"].shape[0], -1, 4)[:, :cfg.cap][:, ~live] == 0xAB)
    assert np.all(f["down"][~live] == 0xABAB)
    # the two GEMMs on sampled live rows
    g = np.random.default_rng(11)
    rows = np.sort(g.choice(np.flatnonzero(live), 256, replace=False))
    ref1, ab1 = sampled_rows_gemm(orc, u["a"], u["a_sf"], ends, rows, inp.w13, inp.w13_sf, cfg.H)
    assert_rows_close(u["gateup"][rows], ref1, ab1)
    ref2, ab2 = sampled_rows_gemm(orc, u["act"], u["sf"], ends, rows, inp.w2, inp.w2_sf, cfg.I)
    assert_rows_close(u["down"][rows], ref2, ab2)
    # the whole layer on sampled tokens
    toks = np.sort(g.choice(cfg.T, 256, replace=False)).astype(np.int32)
    ref = orc.ffn_tokens(inp.x, ids, w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf, toks)
    check_ffn_tolerance(u["out"][toks], ref)


def test_kimi_layer_sampled_tokens(ctx, orc):
    """Kimi-shaped layer at full size (E = 896, top-16, sigmoid + bias
    routing, SiLU*mul with clamp 25, capacity 146,560 rows): routing, the
    endpoint tensor, and 256 sampled output rows against the oracle's whole
    layer. The oracle takes the sampled tokens with only the experts those
    tokens use (drawn expert by expert, as the layer's weights were)."""
    cfg = synth.KIMI
    inp = synth.ffn_inputs(cfg)
    layer = MoEFFNLayer(ctx, T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, I=cfg.I, A=cfg.A, cap=cfg.cap,
                        routing=B.MOE_ROUTE_SIGMOID_BIAS_TOPK, act_kind=B.MOE_ACT_SILU_CLAMP,
                        limit=cfg.limit, rsf=cfg.rsf)
    layer.load_expert_weights(lambda e: synth.expert_weights(cfg, e))
    out = layer.forward(dev_bf16(inp.x), dev(inp.logits), dev(inp.bias))
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    ids, w = orc.route_sigmoid_bias_topk(inp.logits, inp.bias, cfg.k)
    assert np.array_equal(host(layer.topk_ids), ids)
    _, ends = orc.endpoints(orc.expert_counts(ids, cfg.E), cfg.A)
    assert np.array_equal(host(layer.expert_ends), ends)
    got = host_u16(out)
    del layer, out
    torch.cuda.empty_cache()
    toks = np.sort(np.random.default_rng(15).choice(cfg.T, 256, replace=False)).astype(np.int32)
    used = np.unique(ids[toks])
    remap = np.full(cfg.E, -1, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    parts = None
    for i, e in enumerate(used):
        p = synth.expert_weights(cfg, int(e))
        if parts is None:
            parts = [np.empty((used.size,) + q.shape, q.dtype) for q in p]
        for dst, q in zip(parts, p):
            dst[i] = q
    ids_c = np.zeros_like(ids)
    ids_c[toks] = remap[ids[toks]]
    ref = orc.ffn_tokens(inp.x, ids_c, w, *parts, toks, clamp=True, limit=cfg.limit)
    check_ffn_tolerance(got[toks], ref)


def test_layer_graph_replay_permuted_routing_deterministic(ctx, orc):
    """Capture route+scatter+FFN once; replay with the logit columns permuted
    (new counts each time): equal to an eager run bit for bit."""
    cfg = synth.FFNConfig("graph", T=512, E=8, k=2, H=512, I=256, seed=12)
    inp = synth.ffn_inputs(cfg)
    layer = make_layer(ctx, cfg, inp)
    x = dev_bf16(inp.x)
    logits = dev(inp.logits)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, logits, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        layer.forward(x, logits, stream=s)
    rng = np.random.default_rng(100)
    for i in range(3):
        perm = rng.permutation(cfg.E)
        logits.copy_(dev(inp.logits[:, perm]))
        graph.replay()
        torch.cuda.synchronize()
        replayed = host_u16(layer.out).copy()
        ends_replayed = host(layer.expert_ends).copy()
        layer.forward(x, logits)
        torch.cuda.synchronize()
        assert np.array_equal(replayed, host_u16(layer.out))
        ids, w = orc.route_softmax_topk(inp.logits[:, perm], cfg.k)
        ends, _, _, _ = orc.scatter(ids, inp.x, cfg.E, cfg.A, cfg.cap)
        assert np.array_equal(ends_replayed, ends)
        toks = np.arange(0, cfg.T, 37, dtype=np.int32)
        ref = orc.ffn_tokens(inp.x, ids, w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf, toks)
        check_ffn_tolerance(replayed[toks], ref)
    assert B.moe_get_device_error(ctx) == 0


def test_layer_three_runs_bitwise_identical(ctx):
    cfg = synth.FFNConfig("det", T=256, E=8, k=4, H=256, I=256, seed=13)
    inp = synth.ffn_inputs(cfg)
    layer = make_layer(ctx, cfg, inp)
    outs = []
    for _ in range(3):
        layer.forward(dev_bf16(inp.x), dev(inp.logits))
        torch.cuda.synchronize()
        outs.append(host_u16(layer.out).copy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
