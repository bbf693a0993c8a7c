"""Helpers shared by the GPU tests: numpy <-> torch transfers and tolerances."""
import numpy as np
import torch

from tests.refs import bf16_bits_to_f64, bf16_ulp, e2m1_decode, e4m3_decode_torch


def dev_bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    return t.contiguous().cpu().numpy()


def filled(shape, byte, dtype=torch.uint8):
    """Device tensor whose every byte is `byte` (a sentinel)."""
    nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    t = torch.full((nbytes,), byte, dtype=torch.uint8, device="cuda")
    return t.view(dtype).view(shape)


def check_ffn_tolerance(got_u16, ref_u16):
    """The layer-output tolerance: max|err| <= 2e-2 * rms(ref) and
    mean(|err|) / mean(|ref|) <= 5e-3."""
    g = bf16_bits_to_f64(got_u16)
    r = bf16_bits_to_f64(ref_u16)
    assert np.all(np.isfinite(g))
    err = np.abs(g - r)
    rms = np.sqrt(np.mean(r * r))
    max_ratio = err.max() / rms
    mean_rel = err.mean() / np.mean(np.abs(r))
    assert max_ratio <= 2e-2, (max_ratio, mean_rel)
    assert mean_rel <= 5e-3, (max_ratio, mean_rel)
    return max_ratio, mean_rel


# fp32 summation bound of a tensor-core dot product over K <= 4096 terms,
# relative to the sum of |products| (as in the grouped GEMM tests); twice that
# where every activation enters as two terms.
FP32_SUM_BOUND = 2.0 ** -18
# two-term e4m3 split of the tcgen05 decode path: values within 2^13 of their
# group-of-32 maximum exact, the rest within 2^-21 of that maximum
# (tests/test_split_bound.py)
SPLIT_ABS_BOUND = 2.0 ** -21


def _abs_weights(W, wfmt, key, e, K):
    """|dequantised weight matrix| of local expert e, fp64 [N, K] (without
    the per-expert fp32 scale of the FP8 format)."""
    if wfmt == 0:
        return np.abs(e4m3_decode_torch(W["w_" + key][e]))
    sf = W[key + "_sf"][e].astype(np.int64)
    return np.abs(e2m1_decode(W["w_" + key][e], K)) * np.repeat(2.0 ** (sf - 127), 32, axis=1)


def _gemv_bound(inp_rows, W, wfmt, key, slots_of, K, split):
    """Per-element bound of |got - exact| for y = W v * scale + b on every slot:
    the fp32 summation bound, plus the split's error when the activation
    enters as two e4m3 terms. inp_rows: bf16 bits [n_slots, K]."""
    v = np.abs(bf16_bits_to_f64(inp_rows))
    gmax = np.repeat(v.reshape(v.shape[0], -1, 32).max(axis=2), 32, axis=1)
    out = {}
    for e, slots in slots_of.items():
        aw = _abs_weights(W, wfmt, key, e, K)
        sc = float(W[key + "_scale"][e]) if wfmt == 0 else 1.0
        b = (2 * FP32_SUM_BOUND if split else FP32_SUM_BOUND) * (v[slots] @ aw.T)
        if split:
            b = b + SPLIT_ABS_BOUND * (gmax[slots] @ aw.T)
        out[e] = b * sc
    return out


def check_decode_stages(orc, x, ids, w, W, wfmt, H, I, got, es=0, nl=None, interleaved=True, split=False):
    """Stage-wise check of one decode call against the oracle, each stage fed
    the GPU's own output of the stage before:
      y1  every local element within one bf16 step of the oracle's GEMV of x
          plus the fp32 summation bound (plus the split bound with split=True,
          the tcgen05 path);
      act bit for bit the oracle's GLU of the GPU's y1;
      y2  every local element within the same kind of bound of the oracle's
          GEMV of the GPU's act;
      out bit for bit the oracle's slot-ordered weighted sum of the GPU's y2.
    Then the whole output against the oracle's whole path: mean relative
    error <= 5e-3. (A max|err| <= 2e-2 rms bound on the whole path does not
    hold for any implementation whose GEMV sums differ from the oracle's
    single fp64 sums: a bf16 output above 2.56 rms has a step larger than
    2e-2 rms, and a one-step difference in y1 or y2 now and then moves such
    an output by one step; the stage checks above bound every step instead.)
    Returns (max|err| / rms, mean relative error) of the whole path."""
    y1, act, y2, out = got
    T, k = ids.shape
    nl = W["b_gu"].shape[0] if nl is None else nl
    lid = ids - es
    local = (lid >= 0) & (lid < nl)
    slots_of = {}
    for s in np.flatnonzero(local.ravel()):
        slots_of.setdefault(int(lid.ravel()[s]), []).append(int(s))

    def close(got_rows, ref_rows, bounds, name):
        for e, slots in slots_of.items():
            g = bf16_bits_to_f64(got_rows[slots])
            r = bf16_bits_to_f64(ref_rows[slots])
            lim = bf16_ulp(r) * 1.0001 + 2.0 ** -22 * np.abs(r) + bounds[e]
            bad = ~(np.abs(g - r) <= lim)
            assert not bad.any(), "%s: %d of %d elements of expert %d outside the bound" % (
                name, bad.sum(), bad.size, e)

    ry1 = orc.decode_gemv1(x, ids, W, wfmt, I, es, nl).reshape(T * k, 2 * I)
    y1f = y1.reshape(T * k, 2 * I)
    xs = np.repeat(x, k, axis=0)  # slot rows of x
    close(y1f, ry1, _gemv_bound(xs, W, wfmt, "gu", slots_of, H, split), "y1")
    ract = orc.decode_glu(y1, ids, I, es, nl, interleaved=interleaved)
    lf = local.ravel()
    assert np.array_equal(act[lf], ract[lf]), "act differs from the oracle GLU of the GPU's y1"
    ry2 = orc.decode_gemv2(act, ids, W, wfmt, H, I, es, nl).reshape(T * k, H)
    close(y2.reshape(T * k, H), ry2, _gemv_bound(act, W, wfmt, "d", slots_of, I, split), "y2")
    rout = orc.decode_sum(y2, ids, w, es, nl)
    assert np.array_equal(out, rout), "out differs from the oracle's weighted sum of the GPU's y2"
    _, _, _, full = orc.decode(x, ids, w, W, wfmt, I, expert_start=es, n_local=nl, interleaved=interleaved)
    rows = local.any(axis=1)
    g = bf16_bits_to_f64(out[rows])
    r = bf16_bits_to_f64(full[rows])
    assert np.all(np.isfinite(g))
    err = np.abs(g - r)
    mean_rel = err.mean() / np.mean(np.abs(r))
    assert mean_rel <= 5e-3, mean_rel
    return err.max() / np.sqrt(np.mean(r * r)), mean_rel
