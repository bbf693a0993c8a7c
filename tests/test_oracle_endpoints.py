"""Pins for the aligned prefix-sum endpoints, the scatter permutation and the
routing, against the page's worked example, closed forms and brute force."""
import numpy as np
import pytest

from moe_expert_ffn_scatter_gb300 import synth
from tests.refs import golden, e4m3_decode_torch, unpack_scale_bytes
from tests.test_oracle_quant import ref_group_quant


def test_worked_example_from_page(orc):
    gx = golden("endpoints_worked_example.json")
    start, end = orc.endpoints(np.array(gx["counts"], np.int32), gx["A"])
    assert start.tolist() == gx["start"]
    assert end.tolist() == gx["end"]


def closed_form(counts, A):
    """end[e] = sum_{i<e} align_up(count_i, A) + count_e (numpy cumsum)."""
    aligned = (counts + A - 1) // A * A
    start = np.concatenate([[0], np.cumsum(aligned)[:-1]])
    return start, start + counts


def count_vectors(n=2004, seed=0):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(g.integers(1, 65))
        kind = i % 6
        if kind == 0:
            c = g.integers(0, 400, E)
        elif kind == 1:
            c = np.zeros(E, np.int64)                     # all empty
        elif kind == 2:
            c = g.integers(0, 3, E) * g.integers(0, 2, E)  # mostly empty
        elif kind == 3:
            c = np.zeros(E, np.int64); c[g.integers(0, E)] = g.integers(1, 5000)  # one hot expert
        elif kind == 4:
            c = g.integers(0, 4, E) * 128                 # exact multiples of A
        else:
            c = g.integers(0, 4, E) * 128 + g.integers(-1, 2, E).clip(0)
        out.append(c.astype(np.int32))
    return out


def test_endpoint_recurrence_equals_closed_form(orc):
    checks = 0
    for A in (128, 64, 1):
        for c in count_vectors(2004 if A == 128 else 300, seed=A):
            s, e = orc.endpoints(c, A)
            rs, re = closed_form(c.astype(np.int64), A)
            assert np.array_equal(s, rs) and np.array_equal(e, re)
            assert np.all(s % A == 0) and np.all(e - s == c)
            checks += 2 * len(c)
    assert checks > 24048


def test_counts_skip_masked_and_out_of_range(orc):
    ids = np.array([[0, -1], [3, 3], [7, 1], [1, -5]], np.int32)
    assert orc.expert_counts(ids, 4).tolist() == [1, 2, 0, 2]


def check_scatter(orc, ids, x, E, A, cap):
    ends, s2d, a, sf = orc.scatter(ids, x, E, A, cap)
    T, k = ids.shape
    H = x.shape[1]
    counts = np.array([np.sum(ids == e) for e in range(E)], np.int64)
    rs, re = closed_form(counts, A)
    assert np.array_equal(ends, re)
    live = np.zeros(cap, bool)
    for e in range(E):
        live[rs[e]:re[e]] = True
    # permutation: injective onto the live rows, each route inside its segment,
    # row-major (token, slot) order kept inside a segment
    flat = s2d.reshape(-1)
    ok = (ids.reshape(-1) >= 0) & (ids.reshape(-1) < E)
    assert np.all(flat[~ok] == -1)
    dsts = flat[ok]
    assert len(np.unique(dsts)) == len(dsts)
    assert np.array_equal(np.sort(dsts), np.nonzero(live)[0])
    for e in range(E):
        d = flat[ids.reshape(-1) == e]
        assert np.all((d >= rs[e]) & (d < re[e]))
        assert np.all(np.diff(d) == 1)
    # copied rows are the token's quantised row; padding keeps the sentinel
    assert np.all(a[~live] == 0xAB)
    assert np.all(sf.view(np.uint32)[:, :cap][:, ~live] == 0xABABABAB)
    G = H // 128
    sfb = unpack_scale_bytes(sf, cap, G)
    qcache = {}
    for i, dst in enumerate(flat):
        if dst < 0:
            continue
        t = i // k
        if t not in qcache:
            xv = (x[t].astype(np.uint32) << 16).view(np.float32)
            qcache[t] = ref_group_quant(xv)
        rc, rsf = qcache[t]
        assert np.array_equal(a[dst], rc)
        assert np.array_equal(sfb[dst], rsf)
    # unused bytes of the last packed word are zero for live rows
    if G % 4:
        w = sf.view(np.uint32)[G // 4, :cap][live]
        assert np.all((w >> (8 * (G % 4))) == 0)
    return ends, s2d


def test_scatter_page_counts(orc):
    g = np.random.default_rng(0)
    ids = synth.ids_with_counts(g, [96, 0, 129, 1], k=2)
    x = synth.bf16_normal(g, (ids.shape[0], 256))
    ends, _ = check_scatter(orc, ids, x, 4, 128, 640)
    assert ends.tolist() == [96, 128, 257, 385]


def test_scatter_tiny_softmax_routing(orc):
    cfg = synth.TINY
    inp = synth.ffn_inputs(cfg, weights=False)
    ids, w = orc.route_softmax_topk(inp.logits, cfg.k)
    check_scatter(orc, ids, inp.x, cfg.E, cfg.A, cfg.cap)


def test_scatter_masked_slots_and_empty(orc):
    g = np.random.default_rng(2)
    ids = g.integers(-1, 6, size=(40, 3)).astype(np.int32)
    ids[ids == 2] = -1  # expert 2 empty
    x = synth.bf16_normal(g, (40, 384))
    check_scatter(orc, ids, x, 6, 128, 120 + 6 * 128)
    allmasked = np.full((8, 2), -1, np.int32)
    ends, s2d = check_scatter(orc, allmasked, synth.bf16_normal(g, (8, 128)), 3, 128, 128)
    assert ends.tolist() == [0, 0, 0] and np.all(s2d == -1)


def test_scatter_capacity_overflow(orc):
    ids = np.zeros((200, 1), np.int32)
    with pytest.raises(ValueError):
        orc.scatter(ids, np.zeros((200, 128), np.uint16), 1, 128, 128)


# --------------------------------------------------------------- routing
def softmax64(l):
    z = l.astype(np.float64) - l.max(axis=1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=1, keepdims=True)


@pytest.mark.parametrize("T,E,k", [(64, 4, 2), (300, 32, 6), (50, 896, 16)])
def test_softmax_topk_matches_full_softmax(orc, T, E, k):
    g = np.random.default_rng(T + E)
    logits = synth.fp32_normal(g, (T, E))
    ids, w = orc.route_softmax_topk(logits, k)
    p = softmax64(logits)
    ref_ids = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)
    sel = np.take_along_axis(p, ref_ids, axis=1)
    ref_w = sel / sel.sum(axis=1, keepdims=True)
    assert np.max(np.abs(w - ref_w)) < 4e-7
    assert np.max(np.abs(w.astype(np.float64).sum(axis=1) - 1)) < 1e-6


def test_topk_ties_prefer_lower_index(orc):
    logits = np.array([[1.0, 3.0, 3.0, 0.0, 3.0]], np.float32)
    ids, w = orc.route_softmax_topk(logits, 3)
    assert ids.tolist() == [[1, 2, 4]]
    assert np.allclose(w, 1 / 3, atol=1e-7)


def brute_topk(scores, k):
    """Top-k by enumeration: order experts by (score descending, index
    ascending) with every NaN after every number; +0 and -0 are equal."""
    out = []
    for row in scores:
        key = [(1, 0.0, e) if np.isnan(v) else (0, -float(v) + 0.0, e) for e, v in enumerate(row)]
        out.append([e for _, _, e in sorted(key)[:k]])
    return np.array(out, np.int32)


def test_topk_nan_inf_and_signed_zero(orc):
    nan, inf = np.nan, np.inf
    logits = np.array([
        [nan, 1.0, nan, -inf, 2.0, inf, -0.0, 0.0],
        [nan, nan, nan, nan, -inf, nan, nan, nan],
        [-0.0, 0.0, -0.0, 0.0, nan, -1.0, 1.0, -0.0],
        [nan, nan, nan, nan, nan, nan, nan, nan],
    ], np.float32)
    for k in (1, 3, 5, 8):
        ids, _ = orc.route_softmax_topk(logits, k)
        assert np.array_equal(ids, brute_topk(logits, k)), k
    ids, _ = orc.route_softmax_topk(logits, 8)
    assert ids[0].tolist() == [5, 4, 1, 6, 7, 3, 0, 2]
    assert ids[2].tolist()[:6] == [6, 0, 1, 2, 3, 7]


def test_topk_random_ties_match_enumeration(orc):
    g = np.random.default_rng(21)
    logits = g.integers(-3, 4, size=(40, 100)).astype(np.float32)  # many ties
    logits[g.random((40, 100)) < 0.05] = np.nan
    for k in (1, 7, 16, 100):
        ids, _ = orc.route_softmax_topk(logits, k)
        assert np.array_equal(ids, brute_topk(logits, k))


def test_sigmoid_bias_selects_biased_weights_unbiased(orc):
    g = np.random.default_rng(4)
    T, E, k = 200, 896, 16
    logits = synth.fp32_normal(g, (T, E))
    bias = synth.fp32_normal(g, (E,), 0.1)
    ids, w = orc.route_sigmoid_bias_topk(logits, bias, k)
    sig = 1.0 / (1.0 + np.exp(-logits.astype(np.float64)))
    score = sig + bias.astype(np.float64)
    order = np.argsort(-score, axis=1, kind="stable")
    checked = 0
    for t in range(T):
        srt = np.sort(score[t])[::-1]
        if srt[k - 1] - srt[k] < 1e-5:
            continue  # fp32 vs fp64 may order a near tie differently
        assert set(ids[t]) == set(order[t, :k])
        ref_w = sig[t, ids[t]] / sig[t, ids[t]].sum()
        assert np.max(np.abs(w[t] - ref_w)) < 4e-7
        checked += 1
    assert checked > T * 0.8
    # the bias matters for selection: with it removed the selection changes
    ids0, _ = orc.route_sigmoid_bias_topk(logits, np.zeros(E, np.float32), k)
    assert not np.array_equal(np.sort(ids, axis=1), np.sort(ids0, axis=1))
