"""Sparse decode path on the GPU against the oracle: FP8-per-expert and MXFP4
weights; the mma.sync path (T in {1, ..., 8}, no workspace) and the tcgen05
path (workspace given, T up to 128); non-local slots never written and
skipped."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_scatter_gb300 import binding as B
from moe_expert_ffn_scatter_gb300 import synth
from tests.gpu_util import check_decode_stages, dev, dev_bf16, host_u16
from tests.refs import bf16_bits_to_f64

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


_CACHE_BIG = {}


def inputs_big(T, seed=synth.DECODE_SEED + 100):
    """A 128-token draw (its own weights); smaller T use its first rows."""
    if seed not in _CACHE_BIG:
        _CACHE_BIG[seed] = synth.decode_inputs(128, seed=seed)
    d = _CACHE_BIG[seed]
    return synth.DecodeInputs(d.x[:T], d.logits[:T], d.fp8, d.mxfp4)


def run_decode(ctx, d, ids, w, wfmt, H, I, es, nl, fill=0x7FC0, ws=False, glu_layout=B.MOE_GLU_INTERLEAVED,
               path=None):
    """ws=True forces the tcgen05 path (with a workspace), ws=False the
    mma.sync path where it applies; path overrides."""
    if path is None:
        path = B.MOE_DECODE_TCGEN05 if ws else B.MOE_DECODE_AUTO
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
                             T=T, H=H, I=I, k=k, glu_layout=glu_layout, path=path,
                             workspace=B.decode_workspace(T, k, H, I, nl) if ws else None, **kw)
    torch.cuda.synchronize()
    return host_u16(y1), host_u16(act), host_u16(y2), host_u16(out), loc


WFMTS = pytest.mark.parametrize("wfmt", [B.MOE_WFMT_FP8_PER_EXPERT, B.MOE_WFMT_MXFP4_G32], ids=["fp8", "mxfp4"])


@WFMTS
@pytest.mark.parametrize("ws", [False, True], ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_gpt_oss_shape(ctx, orc, wfmt, T, ws):
    d = inputs(T)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, ws=ws)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out), split=ws)


@WFMTS
@pytest.mark.parametrize("layout", [B.MOE_GLU_INTERLEAVED, B.MOE_GLU_HALVES], ids=["interleaved", "halves"])
@pytest.mark.parametrize("T", [3, 5, 7])
def test_decode_mma_sync_odd_token_counts(ctx, orc, wfmt, layout, T):
    """The mma.sync path stages min(T, 8) token columns; the MMA's columns
    beyond T read column T - 1 and their outputs are never written. Odd T in
    both GLU layouts, the path forced."""
    d = inputs(T, seed=33)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, glu_layout=layout,
                                       path=B.MOE_DECODE_MMA_SYNC)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out),
                        interleaved=layout == B.MOE_GLU_INTERLEAVED)


@WFMTS
@pytest.mark.parametrize("ws", [False, True], ids=["mma_sync", "tcgen05"])
def test_decode_expert_parallel_slice_skips_nonlocal(ctx, orc, wfmt, ws):
    """This call owns experts 8..23 only: slots routed elsewhere stay NaN in
    y1/act/y2 and do not reach the output."""
    T = 8
    d = inputs(T, seed=21)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    es, nl = 8, 16
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, es, nl, ws=ws)
    nonlocal_ = (ids < es) | (ids >= es + nl)
    assert np.all(y1[nonlocal_] == 0x7FC0) and np.all(y2[nonlocal_] == 0x7FC0)
    assert np.all(act.reshape(T, -1, I)[nonlocal_] == 0x7FC0)
    assert np.all(np.isfinite(bf16_bits_to_f64(out)))
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out), es=es, nl=nl, split=ws)


@WFMTS
@pytest.mark.parametrize("T", [16, 37, 64, 128])
def test_decode_tcgen05_batches(ctx, orc, wfmt, T):
    """Batches past the mma.sync path's 8 tokens: every expert read once for
    all slots that chose it (T = 37 leaves ragged segments)."""
    d = inputs_big(T)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, ws=True)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out), split=True)


@WFMTS
def test_decode_tcgen05_activation_groups_wider_than_the_split_range(ctx, orc, wfmt):
    """Token rows whose groups of 32 hold one value of 2-8 and the rest spread
    log-uniformly down to 2^-30 below it: most values lie beyond the 2^13
    range the two-term e4m3 split reproduces exactly, so the path's y1 carries
    the split's error; every stage must stay within the bound that includes
    it, and the output within the layer tolerance."""
    T = 16
    d = inputs_big(T)
    g = np.random.default_rng(17)
    H = I = synth.DECODE_H
    rel = 2.0 ** -g.uniform(0, 30, size=(T, H // 32, 32))
    rel[:, :, 0] = 1.0
    top = g.uniform(2, 8, size=(T, H // 32, 1))
    v = (top * rel * g.choice([-1.0, 1.0], size=rel.shape)).reshape(T, H)
    for t in range(T):  # the large value's place in each group varies
        v[t] = v[t].reshape(-1, 32)[:, g.permutation(32)].reshape(H)
    x = synth.f32_to_bf16_bits(v.astype(np.float32))
    xv = bf16_bits_to_f64(x).reshape(T, -1, 32)
    ratio = np.abs(xv).max(axis=2, keepdims=True) / np.maximum(np.abs(xv), 1e-300)
    assert np.mean(ratio > 2.0 ** 13) > 0.4
    d = synth.DecodeInputs(x, d.logits, d.fp8, d.mxfp4)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, ws=True)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out), split=True)


@WFMTS
@pytest.mark.parametrize("T", [1, 8, 24])
def test_decode_plain_gemv_path(ctx, orc, wfmt, T):
    """The per-(token, slot) GEMV path ([SD] §3) at the gpt-oss shape: forced
    for T <= 8, and taken by AUTO for T = 24 without a workspace."""
    d = inputs(T) if T <= 8 else inputs_big(T)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    path = B.MOE_DECODE_GEMV if T <= 8 else B.MOE_DECODE_AUTO
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, path=path)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out))


@WFMTS
@pytest.mark.parametrize("layout", [B.MOE_GLU_INTERLEAVED, B.MOE_GLU_HALVES], ids=["interleaved", "halves"])
def test_decode_plain_gemv_small_odd_shape(ctx, orc, wfmt, layout):
    """H = I = 160 (a multiple of 32, not of 64): only the plain GEMV path
    applies and AUTO takes it; both GLU layouts; 5 tokens over 8 experts."""
    T, E, k, H = 5, 8, 4, 160
    d = synth.decode_inputs(T, E=E, H=H, I=H, seed=77)
    ids, w = orc.route_softmax_topk(d.logits, k)
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, H, 0, E, glu_layout=layout)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, H, (y1, act, y2, out),
                        interleaved=layout == B.MOE_GLU_INTERLEAVED)


@WFMTS
def test_decode_tcgen05_halves_layout(ctx, orc, wfmt):
    """GLU halves layout: gate rows [0, I), up rows [I, 2I) of w_gu."""
    T = 24
    d = inputs_big(T)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, ws=True,
                                       glu_layout=B.MOE_GLU_HALVES)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out), interleaved=False, split=True)


@WFMTS
def test_decode_tcgen05_hot_expert_two_chunks(ctx, orc, wfmt):
    """Every one of 100 tokens picks expert 5 (100 slots: two 64-column chunks
    of one weight block) and three others; expert-parallel slice 0..23."""
    T, k = 100, synth.DECODE_K
    d = inputs_big(T)
    g = np.random.default_rng(7)
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        others = g.choice([e for e in range(synth.DECODE_E) if e != 5], size=k - 1, replace=False)
        ids[t] = np.concatenate([[5], others])
        g.shuffle(ids[t])
    w = g.random((T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    H = I = synth.DECODE_H
    es, nl = 0, 24
    y1, act, y2, out, loc = run_decode(ctx, d, ids, w, wfmt, H, I, es, nl, ws=True)
    local = ids < es + nl
    assert np.all(y1[~local] == 0x7FC0) and np.all(y2[~local] == 0x7FC0)
    check_decode_stages(orc, d.x, ids, w, loc, wfmt, H, I, (y1, act, y2, out), es=es, nl=nl, split=True)


def test_decode_tcgen05_graph_replay_new_routing(ctx, orc):
    """Captured once, replayed with other routing written into the same id and
    weight buffers: equal to an eager call on that routing."""
    wfmt = B.MOE_WFMT_MXFP4_G32
    T, k = 48, synth.DECODE_K
    H = I = synth.DECODE_H
    d = inputs_big(T)
    ids_a, w_a = orc.route_softmax_topk(d.logits, k)
    ids_b, w_b = orc.route_softmax_topk(d.logits[::-1].copy(), k)
    W = d.mxfp4
    x, ids_t, w_t = dev_bf16(d.x), dev(ids_a), dev(w_a)
    args = dict(expert_start=0, num_local_experts=synth.DECODE_E, wfmt=wfmt, w_gu=dev(W["w_gu"]),
                w_gu_sf=dev(W["gu_sf"]), b_gu=dev_bf16(W["b_gu"]), w_d=dev(W["w_d"]), w_d_sf=dev(W["d_sf"]),
                b_d=dev_bf16(W["b_d"]), T=T, H=H, I=I, k=k)
    bufs = dict(y1=torch.empty((T, k, 2 * I), dtype=torch.bfloat16, device="cuda"),
                act=torch.empty((T * k, I), dtype=torch.bfloat16, device="cuda"),
                y2=torch.empty((T, k, H), dtype=torch.bfloat16, device="cuda"),
                out=torch.empty((T, H), dtype=torch.bfloat16, device="cuda"))
    ws = B.decode_workspace(T, k, H, I, synth.DECODE_E)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.moe_sparse_gemv_decode(ctx, x=x, topk_ids=ids_t, topk_w=w_t, workspace=ws, **args, **bufs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        B.moe_sparse_gemv_decode(ctx, x=x, topk_ids=ids_t, topk_w=w_t, workspace=ws, **args, **bufs)
    ids_t.copy_(dev(ids_b))
    w_t.copy_(dev(w_b))
    graph.replay()
    torch.cuda.synchronize()
    got = {kk: host_u16(v).copy() for kk, v in bufs.items()}
    eager = {kk: torch.empty_like(v) for kk, v in bufs.items()}
    B.moe_sparse_gemv_decode(ctx, x=x, topk_ids=dev(ids_b), topk_w=dev(w_b), workspace=ws, **args, **eager)
    torch.cuda.synchronize()
    assert np.array_equal(got["out"], host_u16(eager["out"]))
    check_decode_stages(orc, d.x, ids_b, w_b, W, wfmt, H, I, (got["y1"], got["act"], got["y2"], got["out"]),
                        split=True)


def test_decode_tcgen05_workspace_checks(ctx):
    """A workspace smaller than moe_decode_workspace_size or misaligned is an
    invalid argument for the tcgen05 path."""
    T, k, H, I, nl = 16, 4, 256, 128, 8
    need = B.moe_decode_workspace_size(T, k, H, I, nl)
    assert need > 0 and B.moe_decode_workspace_size(0, k, H, I, nl) == 0
    z = lambda *shape: torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    u8 = lambda n: torch.zeros(n, dtype=torch.uint8, device="cuda")
    args = dict(x=z(T, H), topk_ids=torch.zeros((T, k), dtype=torch.int32, device="cuda"),
                topk_w=torch.zeros((T, k), dtype=torch.float32, device="cuda"), expert_start=0,
                num_local_experts=nl, wfmt=B.MOE_WFMT_FP8_PER_EXPERT, w_gu=u8(nl * 2 * I * H),
                w_gu_scale=torch.ones(nl, device="cuda"), b_gu=z(nl, 2 * I), w_d=u8(nl * H * I),
                w_d_scale=torch.ones(nl, device="cuda"), b_d=z(nl, H), y1=z(T, k, 2 * I), act=z(T * k, I),
                y2=z(T, k, H), out=z(T, H), T=T, H=H, I=I, k=k)
    tc5 = B.MOE_DECODE_TCGEN05
    with pytest.raises(B.MoeError):
        B.moe_sparse_gemv_decode(ctx, workspace=u8(need - 1024), path=tc5, **args)
    with pytest.raises(B.MoeError):
        B.moe_sparse_gemv_decode(ctx, workspace=u8(need + 1024)[16:], path=tc5, **args)
    B.moe_sparse_gemv_decode(ctx, workspace=u8(need), path=tc5, **args)
    torch.cuda.synchronize()


@WFMTS
@pytest.mark.parametrize("T", [1, 16])
def test_decode_auto_path_matches_forced(ctx, orc, wfmt, T):
    """AUTO with a workspace: T = 1 takes the mma.sync path, T = 16 the tcgen05
    path, bit for bit the forced results."""
    d = inputs_big(T)
    ids, w = orc.route_softmax_topk(d.logits, synth.DECODE_K)
    H = I = synth.DECODE_H
    forced = B.MOE_DECODE_MMA_SYNC if T <= 8 else B.MOE_DECODE_TCGEN05
    auto = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, ws=True, path=B.MOE_DECODE_AUTO)
    ref = run_decode(ctx, d, ids, w, wfmt, H, I, 0, synth.DECODE_E, ws=True, path=forced)
    for a_, b_ in zip(auto[:4], ref[:4]):
        assert np.array_equal(a_, b_)


def test_decode_forced_path_checks(ctx):
    """A forced path that does not apply is an invalid argument."""
    T, k, H, I, nl = 16, 4, 256, 128, 8
    z = lambda *shape: torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    u8 = lambda n: torch.zeros(n, dtype=torch.uint8, device="cuda")
    args = dict(x=z(T, H), topk_ids=torch.zeros((T, k), dtype=torch.int32, device="cuda"),
                topk_w=torch.zeros((T, k), dtype=torch.float32, device="cuda"), expert_start=0,
                num_local_experts=nl, wfmt=B.MOE_WFMT_FP8_PER_EXPERT, w_gu=u8(nl * 2 * I * H),
                w_gu_scale=torch.ones(nl, device="cuda"), b_gu=z(nl, 2 * I), w_d=u8(nl * H * I),
                w_d_scale=torch.ones(nl, device="cuda"), b_d=z(nl, H), y1=z(T, k, 2 * I), act=z(T * k, I),
                y2=z(T, k, H), out=z(T, H), T=T, H=H, I=I, k=k)
    with pytest.raises(B.MoeError):  # tcgen05 without a workspace
        B.moe_sparse_gemv_decode(ctx, path=B.MOE_DECODE_TCGEN05, **args)
    with pytest.raises(B.MoeError):  # mma.sync takes T <= 8
        B.moe_sparse_gemv_decode(ctx, path=B.MOE_DECODE_MMA_SYNC, **args)
    with pytest.raises(B.MoeError):
        B.moe_sparse_gemv_decode(ctx, path=7, **args)
    B.moe_sparse_gemv_decode(ctx, path=B.MOE_DECODE_GEMV, **args)
    torch.cuda.synchronize()
