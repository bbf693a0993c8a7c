"""Live-row SiLU*mul + e4m3/UE8M0 quantisation on the GPU against the oracle:
bit-exact codes and packed scales, padding outputs untouched, dense fallback,
graph capture replayed with reversed counts, edge cases."""
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


def nan_padding(orc, gateup, counts, A=128):
    g = gateup.copy()
    start, end = orc.endpoints(counts, A)
    live = np.zeros(g.shape[0], bool)
    for s, e in zip(start, end):
        live[s:e] = True
    g[~live] = 0x7FC0
    return g, live


def run_gpu(ctx, gateup_u16, counts, I, A=128, dense=False, kind=B.MOE_ACT_SILU, limit=0.0, situ=(4.0, 25.0),
            group=128):
    M = gateup_u16.shape[0]
    E = len(counts)
    g = dev_bf16(gateup_u16)
    out = filled((M, I), 0xAB)
    out_sf = filled((((I // group) + 3) // 4, synth.align4(M)), 0xAB, torch.int32)
    ends = None
    if not dense:
        ends = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        B.moe_expert_ends_from_counts(ctx, dev(np.asarray(counts, np.int32)), A, ends)
    B.moe_act_quant(ctx, g, out, out_sf, ends, E, A, M, I, kind, limit, situ=situ, group=group)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) == 0
    return out, out_sf, ends


def test_microbench_shape_bit_exact(ctx, orc):
    gateup, counts = synth.actq_inputs()
    gateup, live = nan_padding(orc, gateup, counts)
    out, out_sf, ends = run_gpu(ctx, gateup, counts, synth.ACTQ_I)
    _, ref_end = orc.endpoints(counts, 128)
    assert np.array_equal(host(ends), ref_end)
    ref, ref_sf = orc.act_quant(gateup, ref_end, 128)
    assert np.array_equal(host(out), ref)           # live rows bit-exact, padding still 0xAB
    assert np.array_equal(host(out_sf), ref_sf)
    assert np.all(host(out)[~live] == 0xAB)


def test_full_buffer_metadata_equals_dense(ctx, orc):
    gateup, counts = synth.actq_inputs(full=True)
    out, out_sf, _ = run_gpu(ctx, gateup, counts, synth.ACTQ_I)
    dout, dsf, _ = run_gpu(ctx, gateup, counts, synth.ACTQ_I, dense=True)
    assert np.array_equal(host(out), host(dout)) and np.array_equal(host(out_sf), host(dsf))
    rows = np.random.default_rng(0).choice(gateup.shape[0], 512, replace=False)
    ref, ref_sf = orc.act_quant(gateup[rows], None, 128)
    assert np.array_equal(host(dout)[rows], ref)
    assert np.array_equal(host(dsf)[:, rows], ref_sf[:, :512])


@pytest.mark.parametrize("counts", [[0, 0, 0, 0], [0, 300, 0, 5], [129, 1, 0, 128], [1, 1, 1, 1]])
def test_empty_and_ragged_counts(ctx, orc, counts):
    I = 384  # three groups: the last packed word has an unused byte
    rows = 1024
    gateup, _ = synth.actq_inputs(rows=rows, I=I, E=4, live=1, seed=7)
    gateup, live = nan_padding(orc, gateup, np.array(counts, np.int32))
    out, out_sf, _ = run_gpu(ctx, gateup, counts, I)
    _, end = orc.endpoints(np.array(counts, np.int32), 128)
    ref, ref_sf = orc.act_quant(gateup, end, 128)
    assert np.array_equal(host(out), ref) and np.array_equal(host(out_sf), ref_sf)


@pytest.mark.parametrize("limit", [25.0, 0.75])
def test_clamp(ctx, orc, limit):
    I = 128
    gateup, counts = synth.actq_inputs(rows=512, I=I, E=2, live=300, seed=9)
    gateup = (synth.f32_to_bf16_bits(orc.bf16_to_f32_array(gateup) * 8)).astype(np.uint16)
    gateup, _ = nan_padding(orc, gateup, counts)
    out, out_sf, _ = run_gpu(ctx, gateup, counts, I, kind=B.MOE_ACT_SILU_CLAMP, limit=limit)
    _, end = orc.endpoints(counts, 128)
    ref, ref_sf = orc.act_quant(gateup, end, 128, clamp=True, limit=limit)
    assert np.array_equal(host(out), ref) and np.array_equal(host(out_sf), ref_sf)


def test_special_values(ctx, orc):
    """Zero rows, a row with inf (scale stays 0xFE), huge and tiny values."""
    I = 256
    rows = 128
    g = np.random.default_rng(3)
    vals = g.standard_normal((rows, 2 * I)).astype(np.float32)
    vals[0] = 0.0
    vals[1, 5] = np.inf
    vals[2] *= 1e30
    vals[3] *= 1e-30
    vals[4, I + 3] = np.nan  # NaN in up: its code is NaN, the amax ignores it
    gateup = synth.f32_to_bf16_bits(vals)
    out, out_sf, _ = run_gpu(ctx, gateup, [rows], I)
    ref, ref_sf = orc.act_quant(gateup, np.array([rows], np.int32), 128)
    assert np.array_equal(host(out), ref) and np.array_equal(host(out_sf), ref_sf)


@pytest.mark.parametrize("kind,limit", [(B.MOE_ACT_SILU, 0.0), (B.MOE_ACT_SILU_CLAMP, 7.0)], ids=["silu", "clamp"])
def test_every_gate_bit_pattern(ctx, orc, kind, limit):
    """Each of the 65,536 bf16 gate patterns once (NaN, inf, subnormal, both
    zeros, every exponent inside and outside the shared-memory window), up
    drawn N(0,1): codes and scales bit-exact."""
    I = 2048
    rows = 65536 // I
    g = np.random.default_rng(9)
    gate = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g.shuffle(gate)
    up = synth.bf16_normal(g, (rows, I))
    gateup = np.concatenate([gate.reshape(rows, I), up], axis=1)
    out, out_sf, _ = run_gpu(ctx, gateup, [rows], I, kind=kind, limit=limit)
    ref, ref_sf = orc.act_quant(gateup, np.array([rows], np.int32), 128, clamp=kind == B.MOE_ACT_SILU_CLAMP,
                                limit=limit)
    got = host(out)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, [(int(r), int(c), hex(gateup[r, c]), hex(gateup[r, I + c]), int(got[r, c]),
                            int(ref[r, c])) for r, c in bad[:8]]
    assert np.array_equal(host(out_sf), ref_sf)


@pytest.mark.parametrize("betas", [(4.0, 25.0), (1.5, 7.0)], ids=["kimi", "other"])
def test_situ_microbench_shape_bit_exact(ctx, orc, betas):
    """SiTU ([DG] §2.4.1) over the live rows: codes and scales bit-exact, the
    padding untouched; a second beta pair refills the context's tables."""
    gateup, counts = synth.actq_inputs()
    gateup, live = nan_padding(orc, gateup, counts)
    out, out_sf, ends = run_gpu(ctx, gateup, counts, synth.ACTQ_I, kind=B.MOE_ACT_SITU, situ=betas)
    _, ref_end = orc.endpoints(counts, 128)
    ref, ref_sf = orc.act_quant(gateup, ref_end, 128, situ=betas)
    assert np.array_equal(host(out), ref)
    assert np.array_equal(host(out_sf), ref_sf)
    assert np.all(host(out)[~live] == 0xAB)


@pytest.mark.parametrize("half", ["gate", "up"])
def test_situ_every_bit_pattern(ctx, orc, half):
    """Each of the 65,536 bf16 patterns once in the gate (or the up) half
    under SiTU, the other half N(0,1): bit-exact."""
    I = 2048
    rows = 65536 // I
    g = np.random.default_rng(10)
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g.shuffle(pat)
    other = synth.bf16_normal(g, (rows, I))
    halves = [pat.reshape(rows, I), other] if half == "gate" else [other, pat.reshape(rows, I)]
    gateup = np.concatenate(halves, axis=1)
    out, out_sf, _ = run_gpu(ctx, gateup, [rows], I, kind=B.MOE_ACT_SITU)
    ref, ref_sf = orc.act_quant(gateup, np.array([rows], np.int32), 128, situ=(4.0, 25.0))
    got = host(out)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, [(int(r), int(c), int(got[r, c]), int(ref[r, c])) for r, c in bad[:8]]
    assert np.array_equal(host(out_sf), ref_sf)


@pytest.mark.parametrize("kind,I", [(B.MOE_ACT_SILU, 2048), (B.MOE_ACT_SILU_CLAMP, 384), (B.MOE_ACT_SITU, 640)],
                         ids=["silu", "clamp_I384", "situ_I640"])
def test_group32_mxfp8_recipe_bit_exact(ctx, orc, kind, I):
    """Group-32 e4m3 output (MXFP8 recipe, [DG] §6): one scale per 32
    columns, four per word; live rows only, padding untouched."""
    g = np.random.default_rng(I)
    counts = np.array([100, 0, 37, 260], np.int32)
    _, end = orc.endpoints(counts, 128)
    M = int(synth.align_up(end[-1], 128))
    gateup = synth.bf16_normal(g, (M, 2 * I))
    gateup[5, :20] = 0x7FC0
    gateup, live = nan_padding(orc, gateup, counts)
    limit = 1.5 if kind == B.MOE_ACT_SILU_CLAMP else 0.0
    out, out_sf, _ = run_gpu(ctx, gateup, counts, I, kind=kind, limit=limit, group=32)
    ref, ref_sf = orc.act_quant(gateup, end, 128, clamp=kind == B.MOE_ACT_SILU_CLAMP, limit=limit,
                                situ=(4.0, 25.0) if kind == B.MOE_ACT_SITU else None, group=32)
    assert np.array_equal(host(out), ref)
    assert np.array_equal(host(out_sf), ref_sf)
    assert np.all(host(out)[~live] == 0xAB)


def test_graph_replay_with_reversed_counts(ctx, orc):
    """Capture endpoints + act-quant once; replay after reversing the counts
    (and refreshing the inputs in place): live outputs bit-exact, padding of
    the new layout untouched ([LR] §3 test recipe)."""
    I = synth.ACTQ_I
    rows = synth.ACTQ_ROWS
    E = synth.ACTQ_E
    gateup0, counts0 = synth.actq_inputs()
    counts1 = counts0[::-1].copy()
    g_dev = dev_bf16(nan_padding(orc, gateup0, counts0)[0])
    c_dev = dev(counts0)
    ends = torch.zeros((E,), dtype=torch.int32, device="cuda")
    out = filled((rows, I), 0xAB)
    out_sf = filled((I // 512, rows), 0xAB, torch.int32)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        B.moe_expert_ends_from_counts(ctx, c_dev, 128, ends, stream=s)
        B.moe_act_quant(ctx, g_dev, out, out_sf, ends, E, 128, rows, I, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        B.moe_expert_ends_from_counts(ctx, c_dev, 128, ends, stream=s)
        B.moe_act_quant(ctx, g_dev, out, out_sf, ends, E, 128, rows, I, stream=s)
    for counts in (counts1, counts0, counts1):
        gateup, live = nan_padding(orc, gateup0, counts)
        g_dev.copy_(dev_bf16(gateup))
        c_dev.copy_(dev(counts))
        out.fill_(0xAB)
        out_sf.view(torch.uint8).fill_(0xAB)
        graph.replay()
        torch.cuda.synchronize()
        _, end = orc.endpoints(counts, 128)
        ref, ref_sf = orc.act_quant(gateup, end, 128)
        assert np.array_equal(host(ends), end)
        assert np.array_equal(host(out), ref) and np.array_equal(host(out_sf), ref_sf)
        assert np.all(host(out)[~live] == 0xAB)
    assert B.moe_get_device_error(ctx) == 0


def test_bad_endpoints_set_error_bit_and_write_nothing(ctx):
    I = 128
    M = 256
    g = dev_bf16(np.zeros((M, 2 * I), np.uint16))
    out = filled((M, I), 0xAB)
    out_sf = filled((1, M), 0xAB, torch.int32)
    ends = dev(np.array([100, 5000], np.int32))  # beyond the buffer
    B.moe_act_quant(ctx, g, out, out_sf, ends, 2, 128, M, I)
    torch.cuda.synchronize()
    assert B.moe_get_device_error(ctx) & B.MOE_DEVERR_ENDPOINTS
    assert np.all(host(out)[100:] == 0xAB)
    assert B.moe_get_device_error(ctx) == 0  # reading clears the word


def test_invalid_arguments_rejected(ctx):
    t = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoeError):
        B.moe_act_quant(ctx, t, t, t, None, 1, 128, 4, 100)  # I not a multiple of 128
    for bad_limit in (0.0, -1.0, float("nan")):  # the clamp needs L > 0
        with pytest.raises(B.MoeError):
            B.moe_act_quant(ctx, t, t, t, None, 1, 128, 4, 128, B.MOE_ACT_SILU_CLAMP, bad_limit)
    for bad in ((0.0, 25.0), (4.0, -1.0), (float("inf"), 25.0), (4.0, float("nan"))):  # SiTU betas
        with pytest.raises(B.MoeError):
            B.moe_act_quant(ctx, t, t, t, None, 1, 128, 4, 128, B.MOE_ACT_SITU, situ=bad)
    with pytest.raises(B.MoeError):
        B.moe_act_quant(ctx, t, t, t, None, 1, 128, 4, 128, 7)  # unknown kind
