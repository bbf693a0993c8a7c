"""Pins for the grouped GEMM, the combine, the whole layer (dense twin) and
the decode path."""
import numpy as np
import pytest

from moe_expert_ffn_scatter_gb300 import synth
from tests.refs import (bf16_bits_to_f64, bf16_ulp, e2m1_decode, e4m3_decode_torch, e4m3_encode_torch,
                        unpack_scale_bytes)


def deq_weights(w, w_sf):
    E, N, K2 = w.shape
    K = 2 * K2
    vals = e2m1_decode(w, K)
    scale = np.repeat(np.ldexp(1.0, w_sf.astype(int) - 127), 32, axis=2)
    return vals * scale  # [E, N, K] float64


def random_a(g, cap, K):
    a = synth.e4m3_codes(g, (cap, K), exp_lo=1, exp_hi=14)
    sfb = synth.ue8m0_bytes(g, (cap, K // 128), -3, 3)
    return a, sfb, synth.pack_scale_words(sfb, synth.align4(cap))


def test_grouped_gemm_matches_numpy_matmul(orc):
    g = np.random.default_rng(0)
    E, K, N, A = 3, 256, 64, 128
    counts = np.array([5, 0, 130], np.int32)
    start, end = orc.endpoints(counts, A)
    cap = 512
    a, sfb, a_sf = random_a(g, cap, K)
    w = synth.e2m1_packed(g, (E, N, K // 2))
    w_sf = synth.ue8m0_bytes(g, (E, N, K // 32))
    out = orc.grouped_gemm(a, a_sf, end, A, w, w_sf, out=np.full((cap, N), 0xDEAD, np.uint16))
    wd = deq_weights(w, w_sf)
    ad = e4m3_decode_torch(a) * np.repeat(np.ldexp(1.0, sfb.astype(int) - 127), 128, axis=1)
    live = np.zeros(cap, bool)
    for e in range(E):
        r0, r1 = start[e], end[e]
        live[r0:r1] = True
        ref = ad[r0:r1] @ wd[e].T
        got = bf16_bits_to_f64(out[r0:r1])
        # fp64 sum rounded once to bf16: within half a bf16 ulp of the exact product
        assert np.all(np.abs(got - ref) <= 0.5 * bf16_ulp(ref) + 1e-300)
    assert np.all(out[~live] == 0xDEAD)


@pytest.mark.parametrize("recipe", ["mxfp8", "fp8_block128"])
def test_grouped_gemm_fp8_weight_recipes_match_numpy(orc, recipe):
    """e4m3 weights with per-(row, 32-K) scales (MXFP8, with group-32
    activation scales) or with one scale per 128 x 128 block (FP8 block128,
    group-128 activations): against an fp64 matmul of operands decoded here."""
    g = np.random.default_rng(5)
    E, K, N, A = 2, 256, 256, 128
    counts = np.array([40, 130], np.int32)
    start, end = orc.endpoints(counts, A)
    cap = 384
    group = 32 if recipe == "mxfp8" else 128
    a = synth.e4m3_codes(g, (cap, K), exp_lo=1, exp_hi=14)
    sfb = synth.ue8m0_bytes(g, (cap, K // group), -3, 3)
    a_sf = synth.pack_scale_words(sfb, synth.align4(cap))
    w = synth.e4m3_codes(g, (E, N, K))
    if recipe == "mxfp8":
        w_sf = synth.ue8m0_bytes(g, (E, N, K // 32))
        wscale = np.repeat(np.ldexp(1.0, w_sf.astype(int) - 127), 32, axis=2)
    else:
        blk = synth.ue8m0_bytes(g, (E, N // 128, K // 128))
        w_sf = orc.expand_block_scales(blk, N, K)
        wscale = np.repeat(np.repeat(np.ldexp(1.0, blk.astype(int) - 127), 128, axis=1), 128, axis=2)
    out = orc.grouped_gemm(a, a_sf, end, A, w, w_sf, a_group=group, wfmt=1)
    wd = e4m3_decode_torch(w) * wscale
    ad = e4m3_decode_torch(a) * np.repeat(np.ldexp(1.0, sfb.astype(int) - 127), group, axis=1)
    for e in range(E):
        r0, r1 = start[e], end[e]
        ref = ad[r0:r1] @ wd[e].T
        got = bf16_bits_to_f64(out[r0:r1])
        assert np.all(np.abs(got - ref) <= 0.5 * bf16_ulp(ref) + 1e-300)


def test_e4m3_reencoding_of_e2m1_weights_gives_the_same_gemm(orc):
    """Every e2m1 value is an e4m3 value: the e4m3 path on the re-encoded
    weights equals the packed e2m1 path bit for bit."""
    g = np.random.default_rng(6)
    E, K, N, A = 2, 256, 128, 128
    counts = np.array([7, 99], np.int32)
    _, end = orc.endpoints(counts, A)
    a, _, a_sf = random_a(g, 256, K)
    w = synth.e2m1_packed(g, (E, N, K // 2))
    w_sf = synth.ue8m0_bytes(g, (E, N, K // 32))
    vals = e2m1_decode(w, K)
    w8 = e4m3_encode_torch(vals.astype(np.float32))
    assert np.array_equal(e4m3_decode_torch(w8), vals)
    assert np.array_equal(orc.grouped_gemm(a, a_sf, end, A, w, w_sf),
                          orc.grouped_gemm(a, a_sf, end, A, w8, w_sf, wfmt=1))


def test_grouped_gemm_identity_weights_return_dequantised_a(orc):
    g = np.random.default_rng(1)
    E, K, N, A = 2, 256, 256, 128
    counts = np.array([3, 70], np.int32)
    _, end = orc.endpoints(counts, A)
    a, sfb, a_sf = random_a(g, 256, K)
    w = np.zeros((E, N, K // 2), np.uint8)
    for n in range(N):
        # code 2 is +1.0; put it at k == n
        w[:, n, n // 2] = (0x2 << 4) if n % 2 else 0x2
    w_sf = np.full((E, N, K // 32), 127, np.uint8)
    out = orc.grouped_gemm(a, a_sf, end, A, w, w_sf)
    ad = e4m3_decode_torch(a) * np.repeat(np.ldexp(1.0, sfb.astype(int) - 127), 128, axis=1)
    for r in list(range(0, 3)) + list(range(128, 198)):
        # every dequantised e4m3 value with a power-of-two scale is exact in bf16
        assert np.array_equal(bf16_bits_to_f64(out[r]), ad[r, :N])


def test_combine_closed_forms(orc):
    g = np.random.default_rng(2)
    H = 64
    down = synth.bf16_normal(g, (10, H))
    down[9] = 0x7FC0  # NaN row never referenced
    s2d = np.array([[3, -1], [-1, -1], [5, 5]], np.int32)
    w = np.array([[1.0, 0.3], [0.5, 0.5], [0.25, 0.75]], np.float32)
    out = orc.combine(down, w, s2d, rsf=1.0)
    assert np.array_equal(out[0], down[3])            # single slot, weight 1
    assert np.all(out[1] == 0)                        # no slot at all
    assert np.array_equal(out[2], down[5])            # 0.25 v + 0.75 v == v exactly
    out2 = orc.combine(down, w, s2d, rsf=2.0)
    assert np.array_equal(bf16_bits_to_f64(out2[0]), 2 * bf16_bits_to_f64(down[3]))


def test_combine_vs_fp64(orc):
    g = np.random.default_rng(3)
    T, k, H, rows = 50, 6, 128, 400
    down = synth.bf16_normal(g, (rows, H))
    s2d = g.permutation(rows)[:T * k].reshape(T, k).astype(np.int32)
    s2d[g.random((T, k)) < 0.1] = -1
    w = g.random((T, k)).astype(np.float32)
    out = orc.combine(down, w, s2d, rsf=1.5)
    d = bf16_bits_to_f64(down)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            if s2d[t, j] >= 0:
                ref[t] += float(w[t, j]) * d[s2d[t, j]]
    ref *= 1.5
    got = bf16_bits_to_f64(out)
    assert np.all(np.abs(got - ref) <= bf16_ulp(ref) + 1e-6)


def small_layer(cfg, orc, clamp=False, limit=0.0):
    inp = synth.ffn_inputs(cfg)
    ids, w = orc.route_softmax_topk(inp.logits, cfg.k)
    return inp, ids, w


def layout_path(orc, cfg, inp, ids, w, clamp=False, limit=0.0, rsf=1.0):
    ends, s2d, a, a_sf = orc.scatter(ids, inp.x, cfg.E, cfg.A, cfg.cap)
    gu = orc.grouped_gemm(a, a_sf, ends, cfg.A, inp.w13, inp.w13_sf)
    act, act_sf = orc.act_quant(gu, ends, cfg.A, clamp=clamp, limit=limit)
    down = orc.grouped_gemm(act, act_sf, ends, cfg.A, inp.w2, inp.w2_sf)
    return orc.combine(down, w, s2d, rsf=rsf)


@pytest.mark.parametrize("clamp,limit", [(False, 0.0), (True, 2.0)])
def test_layout_path_equals_dense_twin_bitwise(orc, clamp, limit):
    cfg = synth.FFNConfig("tiny", T=24, E=4, k=2, H=256, I=128, seed=0)
    inp, ids, w = small_layer(cfg, orc)
    ids[3, 1] = -1  # a masked slot
    out = layout_path(orc, cfg, inp, ids, w, clamp, limit, rsf=1.25)
    dense = orc.ffn_dense(inp.x, ids, w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf, clamp, limit, 1.25)
    assert np.array_equal(out, dense)
    toks = np.array([0, 3, 7, 23], np.int32)
    per = orc.ffn_tokens(inp.x, ids, w, inp.w13, inp.w13_sf, inp.w2, inp.w2_sf, toks, clamp, limit, 1.25)
    assert np.array_equal(per, out[toks])


def test_mxfp8_recipe_layout_path_equals_dense_twin_bitwise(orc):
    """MXFP8 recipe (group-32 activations, e4m3 weights with per-32 scales):
    the layout path (scatter -> GEMM -> act-quant -> GEMM -> combine) equals
    the dense twin and the per-token path bit for bit."""
    cfg = synth.FFNConfig("tiny", T=24, E=4, k=2, H=256, I=128, seed=0)
    inp, ids, w = small_layer(cfg, orc)
    g = np.random.default_rng(8)
    w13 = synth.e4m3_codes(g, (cfg.E, 2 * cfg.I, cfg.H))
    w2 = synth.e4m3_codes(g, (cfg.E, cfg.H, cfg.I))
    ends, s2d, a, a_sf = orc.scatter(ids, inp.x, cfg.E, cfg.A, cfg.cap, group=32)
    gu = orc.grouped_gemm(a, a_sf, ends, cfg.A, w13, inp.w13_sf, a_group=32, wfmt=1)
    act, act_sf = orc.act_quant(gu, ends, cfg.A, group=32)
    down = orc.grouped_gemm(act, act_sf, ends, cfg.A, w2, inp.w2_sf, a_group=32, wfmt=1)
    out = orc.combine(down, w, s2d)
    dense = orc.ffn_dense(inp.x, ids, w, w13, inp.w13_sf, w2, inp.w2_sf, wfmt=1, group=32)
    assert np.array_equal(out, dense)
    toks = np.array([0, 5, 23], np.int32)
    per = orc.ffn_tokens(inp.x, ids, w, w13, inp.w13_sf, w2, inp.w2_sf, toks, wfmt=1, group=32)
    assert np.array_equal(per, out[toks])


def test_single_expert_layer_is_textbook_mlp(orc):
    """E=1, k=1: the layer is W2 . act(W13 . x) on dequantised operands."""
    cfg = synth.FFNConfig("one expert", T=8, E=1, k=1, H=256, I=128, seed=6)
    inp = synth.ffn_inputs(cfg)
    ids = np.zeros((cfg.T, 1), np.int32)
    w = np.ones((cfg.T, 1), np.float32)
    out = layout_path(orc, cfg, inp, ids, w)
    x = bf16_bits_to_f64(inp.x).astype(np.float32)
    w13 = deq_weights(inp.w13, inp.w13_sf)[0]
    w2 = deq_weights(inp.w2, inp.w2_sf)[0]
    from tests.test_oracle_quant import ref_group_quant
    for t in range(cfg.T):
        q, s = ref_group_quant(x[t])
        xd = e4m3_decode_torch(q) * np.repeat(np.ldexp(1.0, s.astype(int) - 127), 128)
        gu = xd @ w13.T
        gu_b = bf16_bits_to_f64(synth.f32_to_bf16_bits(gu.astype(np.float32)))
        gg, uu = gu_b[:cfg.I], gu_b[cfg.I:]
        h = (gg / (1 + np.exp(-gg)) * uu).astype(np.float32)
        q2, s2 = ref_group_quant(h)
        hd = e4m3_decode_torch(q2) * np.repeat(np.ldexp(1.0, s2.astype(int) - 127), 128)
        y = hd @ w2.T
        got = bf16_bits_to_f64(out[t])
        # two bf16 roundings and possible one-step e4m3 flips upstream
        err = np.abs(got - y)
        assert np.mean(err) <= 5e-3 * np.mean(np.abs(y)) and np.max(err) <= 2e-2 * np.sqrt(np.mean(y * y)) * 4


@pytest.mark.parametrize("wfmt", [0, 1])
def test_decode_sparse_equals_dense_twin(orc, wfmt):
    T, E, H, I, k = 3, 6, 128, 128, 4
    d = synth.decode_inputs(T, E=E, H=H, I=I, seed=9)
    ids, w = orc.route_softmax_topk(d.logits, k)
    weights = d.fp8 if wfmt == 0 else d.mxfp4
    # two ranks' worth of experts: this "rank" owns experts 2..5
    es, nl = 2, 4
    loc = {kk: v[es:es + nl] for kk, v in weights.items()}
    y1, act, y2, out = orc.decode(d.x, ids, w, loc, wfmt, I, expert_start=es, n_local=nl)
    dense = orc.decode_dense(d.x, ids, w, loc, wfmt, I, expert_start=es, n_local=nl)
    assert np.array_equal(out, dense)
    assert np.all(np.isfinite(bf16_bits_to_f64(out)))
    nonlocal_slots = (ids < es) | (ids >= es + nl)
    assert np.all(y1[nonlocal_slots] == 0x7FC0) and np.all(y2[nonlocal_slots] == 0x7FC0)


@pytest.mark.parametrize("wfmt", [0, 1])
def test_decode_first_gemv_vs_numpy(orc, wfmt):
    T, E, H, I, k = 2, 4, 256, 128, 2
    d = synth.decode_inputs(T, E=E, H=H, I=I, seed=10)
    ids, w = orc.route_softmax_topk(d.logits, k)
    weights = d.fp8 if wfmt == 0 else d.mxfp4
    y1, act, y2, out = orc.decode(d.x, ids, w, weights, wfmt, I)
    x = bf16_bits_to_f64(d.x)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if wfmt == 0:
                W = e4m3_decode_torch(weights["w_gu"][e]) * float(weights["gu_scale"][e])
            else:
                W = deq_weights(weights["w_gu"][e:e + 1], weights["gu_sf"][e:e + 1])[0]
            ref = W @ x[t] + bf16_bits_to_f64(weights["b_gu"][e])
            got = bf16_bits_to_f64(y1[t, j])
            assert np.all(np.abs(got - ref) <= 0.5 * bf16_ulp(ref) * (1 + 1e-9) + 1e-30)


@pytest.mark.parametrize("wfmt", [0, 1])
def test_decode_steps_compose_to_the_whole_path(orc, wfmt):
    """The four decode steps, each run on the previous step's output, give
    the whole path bit for bit (non-local slots included)."""
    T, E, H, I, k = 3, 6, 128, 128, 4
    d = synth.decode_inputs(T, E=E, H=H, I=I, seed=11)
    ids, w = orc.route_softmax_topk(d.logits, k)
    es, nl = 1, 4
    loc = {kk: v[es:es + nl] for kk, v in (d.fp8 if wfmt == 0 else d.mxfp4).items()}
    y1, act, y2, out = orc.decode(d.x, ids, w, loc, wfmt, I, expert_start=es, n_local=nl)
    s1 = orc.decode_gemv1(d.x, ids, loc, wfmt, I, es, nl)
    s2 = orc.decode_glu(s1, ids, I, es, nl)
    s3 = orc.decode_gemv2(s2, ids, loc, wfmt, H, I, es, nl)
    s4 = orc.decode_sum(s3, ids, w, es, nl)
    for a, b in ((s1, y1), (s2, act), (s3, y2), (s4, out)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("wfmt", [0, 1])
def test_decode_second_gemv_vs_numpy(orc, wfmt):
    """The down GEMV on a given act: fp64 numpy matmul on the dequantised
    weights, one rounding to bf16 (within half a bf16 step)."""
    T, E, H, I, k = 2, 4, 128, 256, 2
    d = synth.decode_inputs(T, E=E, H=H, I=I, seed=12)
    ids, _ = orc.route_softmax_topk(d.logits, k)
    weights = d.fp8 if wfmt == 0 else d.mxfp4
    act = synth.bf16_normal(np.random.default_rng(13), (T * k, I))
    y2 = orc.decode_gemv2(act, ids, weights, wfmt, H, I)
    a = bf16_bits_to_f64(act)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if wfmt == 0:
                W = e4m3_decode_torch(weights["w_d"][e]) * float(weights["d_scale"][e])
            else:
                W = deq_weights(weights["w_d"][e:e + 1], weights["d_sf"][e:e + 1])[0]
            ref = W @ a[t * k + j] + bf16_bits_to_f64(weights["b_d"][e])
            got = bf16_bits_to_f64(y2[t, j])
            assert np.all(np.abs(got - ref) <= 0.5 * bf16_ulp(ref) * (1 + 1e-9) + 1e-30)


@pytest.mark.parametrize("interleaved", [True, False])
def test_decode_glu_step_reads_gate_and_up_from_the_layout(orc, interleaved):
    """Interleaved rows pair (2i, 2i+1), halves rows pair (i, I+i); each act
    value is the scalar GLU of its pair rounded to bf16."""
    T, k, I = 2, 2, 64
    ids = np.array([[0, 1], [1, 0]], np.int32)
    y1 = synth.bf16_normal(np.random.default_rng(14), (T, k, 2 * I), std=4.0)
    act = orc.decode_glu(y1, ids, I, 0, 2, interleaved=interleaved)
    for s in range(T * k):
        row = y1.reshape(T * k, 2 * I)[s]
        for i in range(I):
            g, u = (row[2 * i], row[2 * i + 1]) if interleaved else (row[i], row[I + i])
            v = orc.glu_oai(orc.bf16_to_float(g), orc.bf16_to_float(u), 1.702, 1.0, 7.0)
            assert act[s, i] == orc.bf16_from_float(v)


def test_decode_sum_closed_forms(orc):
    """One local slot with weight 1 returns y2; two slots of the same row with
    weights 1/2 return it too (both products exact); a non-local slot adds
    nothing."""
    T, k, H = 2, 3, 32
    y = synth.bf16_normal(np.random.default_rng(15), (T, 1, H))
    y2 = np.repeat(y, k, axis=1)
    ids = np.array([[0, 9, 9], [1, 1, 9]], np.int32)
    w = np.array([[1.0, 5.0, 5.0], [0.5, 0.5, 7.0]], np.float32)
    out = orc.decode_sum(y2, ids, w, 0, 2)
    assert np.array_equal(out, y[:, 0])
