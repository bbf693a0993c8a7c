"""moe_route_scatter_noalloc: routing + endpoints + scatter for callers that
cannot allocate device memory (a host framework that owns every device buffer
and hands the library only the operation's tensors, or a latency-critical path
where an allocation is not allowed). It uses the library's built-in scratch
array instead of a caller workspace, and must give exactly what
moe_route_scatter gives. Collected last on purpose."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_scatter_gb300 import binding as B
from moe_expert_ffn_scatter_gb300 import synth

pytestmark = pytest.mark.gpu


def outputs(T, E, k, H, cap):
    def full(shape, val, dt):
        return torch.full(shape, val, dtype=dt, device="cuda")
    return dict(topk_ids=full((T, k), -9, torch.int32), topk_w=full((T, k), -1.0, torch.float32),
                expert_ends=full((E,), -9, torch.int32), src2dst=full((T, k), -9, torch.int32),
                a_fp8=full((cap, H), 0xAB, torch.uint8),
                a_sf=full(((H // 128 + 3) // 4, synth.align4(cap)), -0x54545455, torch.int32))


def run(ctx, noalloc, cfg, inp, mode):
    o = outputs(cfg.T, cfg.E, cfg.k, cfg.H, cfg.cap)
    kw = dict(routing_mode=mode, x=torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda(),
              logits=torch.from_numpy(inp.logits).cuda(),
              corr_bias=None if inp.bias is None else torch.from_numpy(inp.bias).cuda(),
              T=cfg.T, E=cfg.E, k=cfg.k, H=cfg.H, A=cfg.A, cap=cfg.cap, **o)
    if noalloc:
        B.moe_route_scatter_noalloc(ctx, **kw)
    else:
        ws = torch.empty((B.moe_route_scatter_workspace_size(cfg.T, cfg.E, cfg.k),), dtype=torch.uint8,
                         device="cuda")
        B.moe_route_scatter(ctx, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    return {key: v.cpu().numpy() for key, v in o.items()}


def test_noalloc_equals_workspace_entry_point_on_two_calls_in_a_row(cuda_lib):
    ctx = B.Context(0)
    cases = [(synth.DEEPSEEK, B.MOE_ROUTE_SOFTMAX_TOPK), (synth.KIMI, B.MOE_ROUTE_SIGMOID_BIAS_TOPK)]
    refs = []
    for cfg, mode in cases:
        refs.append(run(ctx, False, cfg, synth.ffn_inputs(cfg, weights=False), mode))
    # two no-allocation calls back to back: the second finds the first one's
    # leftovers in the shared scratch array and must not depend on them
    for (cfg, mode), ref in zip(cases, refs):
        got = run(ctx, True, cfg, synth.ffn_inputs(cfg, weights=False), mode)
        for key in ref:
            assert np.array_equal(got[key], ref[key]), key
    ctx.close()


def run_given_routing(ctx, noalloc, ids, x, E, H, A, cap):
    """Routing given (MOE_ROUTE_PRECOMPUTED): the completion count in the
    scratch is zeroed by a 4-byte memset instead of by the routing kernel.
    T = 0 takes the endpoint kernel alone, which reads the scratch as its
    workspace."""
    T, k = ids.shape
    o = outputs(T, E, k, H, cap)
    o["topk_ids"] = torch.from_numpy(ids).cuda()
    kw = dict(routing_mode=B.MOE_ROUTE_PRECOMPUTED, x=torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda(),
              T=T, E=E, k=k, H=H, A=A, cap=cap, **o)
    if noalloc:
        B.moe_route_scatter_noalloc(ctx, **kw)
    else:
        ws = torch.empty((max(16, B.moe_route_scatter_workspace_size(T, E, k)),), dtype=torch.uint8, device="cuda")
        B.moe_route_scatter(ctx, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    return {key: v.cpu().numpy() for key, v in o.items()}


def test_noalloc_given_routing_and_no_tokens_after_a_large_call(cuda_lib):
    """Each case runs right after a full-size no-allocation call, so the
    shared array holds that call's histograms and completion count."""
    ctx = B.Context(0)
    big = synth.DEEPSEEK
    big_inp = synth.ffn_inputs(big, weights=False)
    g = np.random.default_rng(41)
    E, k, H, A = 4, 2, 256, 128
    counts = np.array([96, 0, 129, 1], np.int64)  # the endpoint example of the live-row page
    ids = synth.ids_with_counts(g, counts, k)
    x = synth.bf16_normal(g, (ids.shape[0], H))
    cap = synth.align_up(ids.size + E * (A - 1), A)
    ref_given = run_given_routing(ctx, False, ids, x, E, H, A, cap)
    T0_ids = np.zeros((0, 6), np.int32)
    T0_x = np.zeros((0, 4096), np.uint16)
    ref_empty = run_given_routing(ctx, False, T0_ids, T0_x, 32, 4096, 128, 32 * 127 + 128)
    for case in ("given", "empty"):
        run(ctx, True, big, big_inp, B.MOE_ROUTE_SOFTMAX_TOPK)
        if case == "given":
            got, ref = run_given_routing(ctx, True, ids, x, E, H, A, cap), ref_given
            assert np.array_equal(got["expert_ends"], [96, 128, 257, 385])
        else:
            got, ref = run_given_routing(ctx, True, T0_ids, T0_x, 32, 4096, 128, 32 * 127 + 128), ref_empty
            assert np.array_equal(got["expert_ends"], np.zeros(32, np.int32))
        for key in ref:
            assert np.array_equal(got[key], ref[key]), (case, key)
    ctx.close()


def test_noalloc_rejects_sizes_beyond_the_scratch_array(cuda_lib):
    ctx = B.Context(0)
    T, E, k, H = 65536 + 64, 256, 1, 128  # ceil(T/64) * E * 4 bytes just above 1 MiB
    cap = synth.align_up(T * k + E * 127, 128)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_route_scatter_noalloc(ctx, routing_mode=B.MOE_ROUTE_PRECOMPUTED, x=x, topk_ids=ids,
                                    expert_ends=torch.zeros((E,), dtype=torch.int32, device="cuda"),
                                    src2dst=torch.zeros((T, k), dtype=torch.int32, device="cuda"),
                                    a_fp8=torch.zeros((16,), dtype=torch.uint8, device="cuda"),
                                    a_sf=torch.zeros((16,), dtype=torch.int32, device="cuda"),
                                    T=T, E=E, k=k, H=H, A=128, cap=cap)
    assert ei.value.status == -3
    ctx.close()
