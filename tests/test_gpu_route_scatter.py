"""Routing, endpoints and the token scatter on the GPU against the oracle:
ids and weights, expert_ends, src2dst, e4m3 rows and packed scales bit-exact;
padding rows untouched."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_scatter_gb300 import binding as B
from moe_expert_ffn_scatter_gb300 import synth
from tests.gpu_util import dev, dev_bf16, filled, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx(cuda_lib):
    return B.Context(0)


def gpu_route_scatter(ctx, x, E, k, A, cap, mode, logits=None, bias=None, ids=None, group=128):
    T, H = x.shape
    ids_d = dev(ids) if ids is not None else torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    w_d = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    ends = torch.full((E,), -9, dtype=torch.int32, device="cuda")
    s2d = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    a = filled((cap, H), 0xAB)
    a_sf = filled(((H // group + 3) // 4, synth.align4(cap)), 0xAB, torch.int32)
    ws = torch.empty((B.moe_route_scatter_workspace_size(T, E, k),), dtype=torch.uint8, device="cuda")
    B.moe_route_scatter(ctx, routing_mode=mode, x=dev_bf16(x), logits=None if logits is None else dev(logits),
                        corr_bias=None if bias is None else dev(bias), topk_ids=ids_d,
                        topk_w=w_d if mode != B.MOE_ROUTE_PRECOMPUTED else None, expert_ends=ends, src2dst=s2d,
                        a_fp8=a, a_sf=a_sf, workspace=ws, T=T, E=E, k=k, H=H, A=A, cap=cap, quant_group=group)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    return host(ids_d), host(w_d), host(ends), host(s2d), host(a), host(a_sf)


def check_against_oracle(orc, res, ids_ref, x, E, A, cap, w_ref=None, group=128):
    ids, w, ends, s2d, a, a_sf = res
    assert np.array_equal(ids, ids_ref)
    if w_ref is not None:
        assert np.array_equal(w.view(np.uint32), w_ref.view(np.uint32))  # bit-exact weights
    r_ends, r_s2d, r_a, r_sf = orc.scatter(ids_ref, x, E, A, cap, group=group)
    assert np.array_equal(ends, r_ends)
    assert np.array_equal(s2d, r_s2d)
    assert np.array_equal(a, r_a)
    assert np.array_equal(a_sf, r_sf)


@pytest.mark.parametrize("cfg", [synth.TINY, synth.DEEPSEEK], ids=["tiny", "deepseek"])
def test_softmax_routing_and_scatter(ctx, orc, cfg):
    inp = synth.ffn_inputs(cfg, weights=False)
    ids_ref, w_ref = orc.route_softmax_topk(inp.logits, cfg.k)
    res = gpu_route_scatter(ctx, inp.x, cfg.E, cfg.k, cfg.A, cfg.cap, B.MOE_ROUTE_SOFTMAX_TOPK, logits=inp.logits)
    check_against_oracle(orc, res, ids_ref, inp.x, cfg.E, cfg.A, cfg.cap, w_ref)


def test_sigmoid_bias_routing_and_scatter_kimi_shape(ctx, orc):
    cfg = synth.KIMI
    inp = synth.ffn_inputs(cfg, weights=False)
    ids_ref, w_ref = orc.route_sigmoid_bias_topk(inp.logits, inp.bias, cfg.k)
    res = gpu_route_scatter(ctx, inp.x, cfg.E, cfg.k, cfg.A, cfg.cap, B.MOE_ROUTE_SIGMOID_BIAS_TOPK,
                            logits=inp.logits, bias=inp.bias)
    check_against_oracle(orc, res, ids_ref, inp.x, cfg.E, cfg.A, cfg.cap, w_ref)


def test_precomputed_page_counts(ctx, orc):
    """[LR] §2 worked example: A=128, counts=[96,0,129,1] -> end=[96,128,257,385]."""
    g = np.random.default_rng(0)
    ids = synth.ids_with_counts(g, [96, 0, 129, 1], k=2)
    x = synth.bf16_normal(g, (ids.shape[0], 256))
    cap = synth.align_up(ids.size + 4 * 127, 128)
    res = gpu_route_scatter(ctx, x, 4, 2, 128, cap, B.MOE_ROUTE_PRECOMPUTED, ids=ids)
    assert res[2].tolist() == [96, 128, 257, 385]
    check_against_oracle(orc, res, ids, x, 4, 128, cap)


@pytest.mark.parametrize("H", [128, 384, 3584])
def test_precomputed_masked_slots_ragged_hidden(ctx, orc, H):
    g = np.random.default_rng(H)
    T, k, E = 300, 3, 7
    ids = g.integers(-1, E, size=(T, k)).astype(np.int32)
    ids[5] = -1
    ids[ids == 4] = -1  # expert 4 empty
    x = synth.bf16_normal(g, (T, H))
    cap = synth.align_up(T * k + E * 127, 128)
    res = gpu_route_scatter(ctx, x, E, k, 128, cap, B.MOE_ROUTE_PRECOMPUTED, ids=ids)
    check_against_oracle(orc, res, ids, x, E, 128, cap)


def test_all_masked_and_empty_batch(ctx, orc):
    ids = np.full((70, 2), -1, np.int32)
    x = synth.bf16_normal(np.random.default_rng(1), (70, 256))
    res = gpu_route_scatter(ctx, x, 5, 2, 128, 1024, B.MOE_ROUTE_PRECOMPUTED, ids=ids)
    assert res[2].tolist() == [0] * 5 and np.all(res[3] == -1)
    assert np.all(res[4] == 0xAB)


def topk_edge_cases():
    g = np.random.default_rng(31)
    cases = []
    l = synth.fp32_normal(g, (8, 896))
    l[:, 5::32] += 10.0  # every winner in one lane: its sorted list runs dry and is rebuilt
    cases.append(("one_lane", l, 16, None))
    l = g.integers(-3, 4, size=(64, 700)).astype(np.float32)  # ties inside and across lanes
    l[g.random(l.shape) < 0.05] = np.nan
    l[g.random(l.shape) < 0.01] = np.inf
    l[g.random(l.shape) < 0.01] = -np.inf
    cases.append(("ties_nan_inf", l, 16, None))
    l = g.integers(-2, 3, size=(64, 200)).astype(np.float32)
    cases.append(("sigmoid_ties", l, 8, np.zeros(200, np.float32)))
    l = np.array([[np.nan, 1.0, np.nan, -np.inf, 2.0, np.inf, -0.0, 0.0] * 4,
                  [-0.0, 0.0] * 16, [np.nan] * 32], np.float32)
    cases.append(("k_equals_E", l, 32, None))
    cases.append(("E1024_k32", synth.fp32_normal(g, (40, 1024)), 32, None))
    return cases


@pytest.mark.parametrize("name,logits,k,bias", topk_edge_cases(), ids=[c[0] for c in topk_edge_cases()])
def test_topk_selection_edge_cases(ctx, orc, name, logits, k, bias):
    """Selection order bit-exact against the oracle with ties, NaN, +-inf,
    signed zeros, all winners in one lane, k = E and E = 1024; weights
    bit-exact on the rows whose selected logits are all finite."""
    T, E = logits.shape
    x = synth.bf16_normal(np.random.default_rng(1), (T, 128))
    cap = synth.align_up(T * k + E * 127, 128)
    if bias is None:
        ids_ref, w_ref = orc.route_softmax_topk(logits, k)
        mode = B.MOE_ROUTE_SOFTMAX_TOPK
    else:
        ids_ref, w_ref = orc.route_sigmoid_bias_topk(logits, bias, k)
        mode = B.MOE_ROUTE_SIGMOID_BIAS_TOPK
    res = gpu_route_scatter(ctx, x, E, k, 128, cap, mode, logits=logits, bias=bias)
    check_against_oracle(orc, res, ids_ref, x, E, 128, cap)
    finite = np.all(np.isfinite(np.take_along_axis(logits, ids_ref, axis=1)), axis=1)
    assert np.array_equal(res[1][finite].view(np.uint32), w_ref[finite].view(np.uint32))


@pytest.mark.parametrize("H", [256, 384, 4096])
def test_scatter_group32_mxfp8_recipe(ctx, orc, H):
    """Input quantisation with group 32 (MXFP8 recipe, [DG] §6): codes and
    the four-bytes-a-word scale array bit-exact, padding untouched; H = 384
    leaves half a 256-column pass."""
    g = np.random.default_rng(H)
    T, E, k = 300, 8, 3
    logits = synth.fp32_normal(g, (T, E))
    x = synth.bf16_normal(g, (T, H))
    x[5, :40] = 0x7FC0  # NaN values in one group
    x[6] = 0            # an all-zero row
    cap = synth.align_up(T * k + E * 127, 128)
    ids_ref, w_ref = orc.route_softmax_topk(logits, k)
    res = gpu_route_scatter(ctx, x, E, k, 128, cap, B.MOE_ROUTE_SOFTMAX_TOPK, logits=logits, group=32)
    check_against_oracle(orc, res, ids_ref, x, E, 128, cap, w_ref, group=32)


def test_skewed_routing_one_hot_expert(ctx, orc):
    """Every token prefers expert 3: one long segment, the rest small."""
    g = np.random.default_rng(5)
    T, E, k = 1000, 16, 4
    logits = synth.fp32_normal(g, (T, E))
    logits[:, 3] += 10.0
    x = synth.bf16_normal(g, (T, 512))
    cap = synth.align_up(T * k + E * 127, 128)
    ids_ref, w_ref = orc.route_softmax_topk(logits, k)
    res = gpu_route_scatter(ctx, x, E, k, 128, cap, B.MOE_ROUTE_SOFTMAX_TOPK, logits=logits)
    check_against_oracle(orc, res, ids_ref, x, E, 128, cap, w_ref)


def test_capacity_checked_on_host(ctx):
    x = torch.zeros((10, 128), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(4096, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_route_scatter(ctx, routing_mode=B.MOE_ROUTE_PRECOMPUTED, x=x, topk_ids=t, expert_ends=t, src2dst=t,
                            a_fp8=t, a_sf=t, workspace=t, T=10, E=2, k=1, H=128, A=128, cap=100)
    assert ei.value.status == -2
