"""CPU oracle for the routed MoE expert FFN: numpy-facing wrappers over liboracle.so.

TEST INFRASTRUCTURE ONLY. This package is imported by the test suite, by the
smoke check and by the benchmark's CPU-baseline leg, and by nothing in the
product path (the CUDA library and its Python binding never import it). It
shares no code with the GPU side: only the seeded input generators are common.

Every function is a direct wrapper over the C function of the same name
without the ``orc_`` prefix; see oracle/moe_oracle.c for the definitions and
the page sections they restate.

Parity partly unpinned: ``glu_oai`` (the gpt-oss GLU of the decode path). Its
clamp and the place of alpha are pinned by ``tests/test_oracle_glu.py``; where
beta enters is a reading that no page fixes.
"""
import ctypes
import os

import numpy as np

from ._build import LIB, build_oracle

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle()
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_long
_F = ctypes.c_float


def _declare(L):
    sig = {
        "orc_bf16_to_float": (_F, [ctypes.c_uint16]),
        "orc_bf16_from_float": (ctypes.c_uint16, [_F]),
        "orc_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_e4m3_from_float": (ctypes.c_uint8, [_F]),
        "orc_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_ue8m0_value": (ctypes.c_double, [ctypes.c_uint8]),
        "orc_ue8m0_ceil": (ctypes.c_uint8, [_F]),
        "orc_exp_spec": (_F, [_F]),
        "orc_silu_spec": (_F, [_F]),
        "orc_sigmoid_spec": (_F, [_F]),
        "orc_tanh_spec": (_F, [_F]),
        "orc_situ_gate_spec": (_F, [_F, _F]),
        "orc_situ_up_spec": (_F, [_F, _F]),
        "orc_glu_oai": (_F, [_F, _F, _F, _F, _F]),
        "orc_group_quant_row": (None, [_P, _I, _I, _P, _P]),
        "orc_route_softmax_topk": (None, [_P, _I, _I, _I, _P, _P]),
        "orc_route_sigmoid_bias_topk": (None, [_P, _P, _I, _I, _I, _P, _P]),
        "orc_expert_counts": (None, [_P, _L, _I, _P]),
        "orc_endpoints": (None, [_P, _I, _I, _P, _P]),
        "orc_scatter": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
        "orc_grouped_gemm": (None, [_P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _I, _I, _P]),
        "orc_expand_block_scales": (None, [_P, _I, _I, _I, _P]),
        "orc_act_quant": (None, [_P, _I, _I, _P, _I, _I, _I, _F, _F, _F, _I, _P, _P, _I]),
        "orc_combine": (None, [_P, _I, _P, _P, _I, _I, _F, _P]),
        "orc_ffn_tokens": (None, [_P, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _F, _F, _F, _F, _P, _I,
                                   _P]),
        "orc_ffn_dense": (None, [_P, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _F, _F, _F, _F, _P]),
        "orc_decode": (None, [_P, _I, _I, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                              _I, _F, _F, _F, _P, _P, _P, _P]),
        "orc_decode_gemv1": (None, [_P, _I, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
        "orc_decode_glu": (None, [_P, _I, _I, _P, _I, _I, _I, _I, _F, _F, _F, _P]),
        "orc_decode_gemv2": (None, [_P, _I, _I, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
        "orc_decode_sum": (None, [_P, _I, _I, _P, _P, _I, _I, _I, _P]),
        "orc_decode_dense": (None, [_P, _I, _I, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _I, _F, _F, _F, _P]),
        "orc_num_threads": (_I, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _p(a):
    """Pointer to a C-contiguous numpy array (or None)."""
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- scalars
def bf16_to_float(h): return lib().orc_bf16_to_float(int(h))
def bf16_from_float(f): return lib().orc_bf16_from_float(float(f))
def bf16_from_double(d): return lib().orc_bf16_from_double(float(d))
def e4m3_value(c): return lib().orc_e4m3_value(int(c))
def e4m3_from_float(x): return lib().orc_e4m3_from_float(float(x))
def e2m1_value(n): return lib().orc_e2m1_value(int(n))
def ue8m0_value(b): return lib().orc_ue8m0_value(int(b))
def ue8m0_ceil(s): return lib().orc_ue8m0_ceil(float(s))
def exp_spec(x): return lib().orc_exp_spec(float(x))
def silu_spec(x): return lib().orc_silu_spec(float(x))
def sigmoid_spec(x): return lib().orc_sigmoid_spec(float(x))
def tanh_spec(x): return lib().orc_tanh_spec(float(x))
def situ_gate_spec(g, beta_s=4.0): return lib().orc_situ_gate_spec(float(g), float(beta_s))
def situ_up_spec(u, beta_l=25.0): return lib().orc_situ_up_spec(float(u), float(beta_l))


def _act(clamp, limit, situ):
    """(kind, limit, beta_s, beta_l): SiLU, SiLU with the clamp, or SiTU when
    situ = (beta_s, beta_l) is given."""
    if situ is not None:
        return 2, 0.0, float(situ[0]), float(situ[1])
    return (1 if clamp else 0), float(limit), 0.0, 0.0
def glu_oai(g, u, alpha, beta, limit): return lib().orc_glu_oai(g, u, alpha, beta, limit)
def num_threads(): return lib().orc_num_threads()


def bf16_to_f32_array(u16):
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ arrays
def group_quant_row(v, group=128):
    v = _c(v, np.float32)
    K = v.shape[0]
    codes = np.zeros(K, np.uint8)
    sf = np.zeros((K + group - 1) // group, np.uint8)
    lib().orc_group_quant_row(_p(v), K, group, _p(codes), _p(sf))
    return codes, sf


def route_softmax_topk(logits, k):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    lib().orc_route_softmax_topk(_p(logits), T, E, k, _p(ids), _p(w))
    return ids, w


def route_sigmoid_bias_topk(logits, bias, k):
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    lib().orc_route_sigmoid_bias_topk(_p(logits), _p(bias), T, E, k, _p(ids), _p(w))
    return ids, w


def expert_counts(ids, E):
    ids = _c(ids, np.int32)
    counts = np.zeros(E, np.int32)
    lib().orc_expert_counts(_p(ids), ids.size, E, _p(counts))
    return counts


def endpoints(counts, A):
    counts = _c(counts, np.int32)
    E = counts.shape[0]
    start = np.zeros(E, np.int32)
    end = np.zeros(E, np.int32)
    lib().orc_endpoints(_p(counts), E, A, _p(start), _p(end))
    return start, end


def align4(n):
    return (n + 3) // 4 * 4


def scatter(ids, x_bf16, E, A, cap, fp8_fill=0xAB, sf_fill=None, group=128):
    """Returns expert_ends, src2dst, a_fp8 [cap,H], a_sf [G4, align4(cap)]
    (G4 = ceil(H/group/4)). Non-live rows keep the fill value (the oracle only
    writes live rows)."""
    ids = _c(ids, np.int32)
    x = _c(x_bf16, np.uint16)
    T, k = ids.shape
    H = x.shape[1]
    G4 = (H // group + 3) // 4
    ld = align4(cap)
    ends = np.zeros(E, np.int32)
    s2d = np.zeros((T, k), np.int32)
    a = np.full((cap, H), fp8_fill, np.uint8)
    sf = np.full((G4, ld), fp8_fill * 0x01010101 if sf_fill is None else sf_fill, np.uint32).view(np.int32)
    rc = lib().orc_scatter(_p(ids), _p(x), T, k, E, H, A, cap, ld, group, _p(ends), _p(s2d), _p(a), _p(sf))
    if rc != 0:
        raise ValueError("capacity exceeded")
    return ends, s2d, a, sf


def grouped_gemm(a, a_sf, expert_ends, A, w, w_sf, out=None, a_group=128, wfmt=0):
    """wfmt 0: w packed e2m1 [E,N,K/2]; 1: w e4m3 [E,N,K]. w_sf [E,N,K/32]."""
    a = _c(a, np.uint8)
    a_sf = _c(a_sf, np.int32)
    ends = _c(expert_ends, np.int32)
    w = _c(w, np.uint8)
    w_sf = _c(w_sf, np.uint8)
    cap, K = a.shape
    E, N = w.shape[0], w.shape[1]
    if out is None:
        out = np.zeros((cap, N), np.uint16)
    lib().orc_grouped_gemm(_p(a), _p(a_sf), a_sf.shape[1], K, a_group, _p(ends), E, A, _p(w), _p(w_sf), wfmt, N,
                           _p(out))
    return out


def expand_block_scales(sf_blk, N, K):
    """FP8-block128 scales [E, ceil(N/128), K/128] -> per-(row, 32-K) [E, N, K/32]."""
    sf_blk = _c(sf_blk, np.uint8)
    E = sf_blk.shape[0]
    out = np.zeros((E, N, K // 32), np.uint8)
    lib().orc_expand_block_scales(_p(sf_blk), E, N, K, _p(out))
    return out


def act_quant(gateup, expert_ends, A, clamp=False, limit=0.0, out=None, out_sf=None, fill=0xAB, situ=None,
              group=128):
    gateup = _c(gateup, np.uint16)
    M, I2 = gateup.shape
    I = I2 // 2
    G4 = ((I + group - 1) // group + 3) // 4
    ld = align4(M)
    if out is None:
        out = np.full((M, I), fill, np.uint8)
    if out_sf is None:
        out_sf = np.full((G4, ld), fill * 0x01010101, np.uint32).view(np.int32)
    ends = None if expert_ends is None else _c(expert_ends, np.int32)
    E = 0 if ends is None else ends.shape[0]
    lib().orc_act_quant(_p(gateup), M, I, _p(ends), E, A, *_act(clamp, limit, situ), group, _p(out), _p(out_sf),
                        ld)
    return out, out_sf


def combine(down, topk_w, src2dst, rsf=1.0):
    down = _c(down, np.uint16)
    topk_w = _c(topk_w, np.float32)
    s2d = _c(src2dst, np.int32)
    T, k = s2d.shape
    H = down.shape[1]
    out = np.zeros((T, H), np.uint16)
    lib().orc_combine(_p(down), H, _p(topk_w), _p(s2d), T, k, float(rsf), _p(out))
    return out


def ffn_tokens(x, ids, topk_w, w13, w13_sf, w2, w2_sf, tokens, clamp=False, limit=0.0, rsf=1.0, situ=None,
               wfmt=0, group=128):
    """wfmt 0: packed e2m1 weights, 1: e4m3; group: activation quantisation
    group (input and act-quant) 128, or 32 for the MXFP8 recipe."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    tokens = _c(tokens, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    E, I2 = w13.shape[0], w13.shape[1]
    out = np.zeros((tokens.shape[0], H), np.uint16)
    lib().orc_ffn_tokens(_p(x), H, I2 // 2, _p(ids), _p(topk_w), k, E, _p(_c(w13, np.uint8)),
                         _p(_c(w13_sf, np.uint8)), _p(_c(w2, np.uint8)), _p(_c(w2_sf, np.uint8)),
                         wfmt, group, *_act(clamp, limit, situ), float(rsf), _p(tokens), tokens.shape[0], _p(out))
    return out


def ffn_dense(x, ids, topk_w, w13, w13_sf, w2, w2_sf, clamp=False, limit=0.0, rsf=1.0, situ=None, wfmt=0,
              group=128):
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    T, H = x.shape
    k = ids.shape[1]
    E, I2 = w13.shape[0], w13.shape[1]
    out = np.zeros((T, H), np.uint16)
    lib().orc_ffn_dense(_p(x), T, H, I2 // 2, _p(ids), _p(topk_w), k, E, _p(_c(w13, np.uint8)),
                        _p(_c(w13_sf, np.uint8)), _p(_c(w2, np.uint8)), _p(_c(w2_sf, np.uint8)),
                        wfmt, group, *_act(clamp, limit, situ), float(rsf), _p(out))
    return out


def _decode_args(w):
    """Returns pointer tuple for a decode weight set dict."""
    def g(key, dt):
        return None if w.get(key) is None else _c(w[key], dt)
    arrs = dict(w_gu=g("w_gu", np.uint8), gu_scale=g("gu_scale", np.float32), gu_sf=g("gu_sf", np.uint8),
                b_gu=g("b_gu", np.uint16), w_d=g("w_d", np.uint8), d_scale=g("d_scale", np.float32),
                d_sf=g("d_sf", np.uint8), b_d=g("b_d", np.uint16))
    return arrs


def decode(x, ids, topk_w, weights, wfmt, I, expert_start=0, n_local=None, interleaved=True,
           alpha=1.702, beta=1.0, limit=7.0, fill=0x7FC0):
    """Sparse decode path. Returns (y1 [T,k,2I], act [T*k,I], y2 [T,k,H], out [T,H]);
    slots of non-local experts keep `fill` (bf16 NaN by default) in y1/act/y2."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    T, H = x.shape
    k = ids.shape[1]
    a = _decode_args(weights)
    if n_local is None:
        n_local = a["b_gu"].shape[0]
    y1 = np.full((T, k, 2 * I), fill, np.uint16)
    act = np.full((T * k, I), fill, np.uint16)
    y2 = np.full((T, k, H), fill, np.uint16)
    out = np.zeros((T, H), np.uint16)
    lib().orc_decode(_p(x), T, H, I, _p(ids), _p(topk_w), k, expert_start, n_local, wfmt,
                     _p(a["w_gu"]), _p(a["gu_scale"]), _p(a["gu_sf"]), _p(a["b_gu"]),
                     _p(a["w_d"]), _p(a["d_scale"]), _p(a["d_sf"]), _p(a["b_d"]),
                     int(bool(interleaved)), float(alpha), float(beta), float(limit),
                     _p(y1), _p(act), _p(y2), _p(out))
    return y1, act, y2, out


def decode_gemv1(x, ids, weights, wfmt, I, expert_start=0, n_local=None, fill=0x7FC0):
    """Step 1 of the decode path alone: y1 [T, k, 2I] of the local slots."""
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    a = _decode_args(weights)
    if n_local is None:
        n_local = a["b_gu"].shape[0]
    y1 = np.full((T, k, 2 * I), fill, np.uint16)
    lib().orc_decode_gemv1(_p(x), T, H, I, _p(ids), k, expert_start, n_local, wfmt, _p(a["w_gu"]),
                           _p(a["gu_scale"]), _p(a["gu_sf"]), _p(a["b_gu"]), _p(y1))
    return y1


def decode_glu(y1, ids, I, expert_start=0, n_local=None, interleaved=True, alpha=1.702, beta=1.0, limit=7.0,
               fill=0x7FC0):
    """Step 2 alone: act [T*k, I] from y1 [T, k, 2I]."""
    y1 = _c(y1, np.uint16)
    ids = _c(ids, np.int32)
    T, k = ids.shape
    if n_local is None:
        n_local = int(ids.max()) + 1 - expert_start
    act = np.full((T * k, I), fill, np.uint16)
    lib().orc_decode_glu(_p(y1), T, I, _p(ids), k, expert_start, n_local, int(bool(interleaved)), float(alpha),
                         float(beta), float(limit), _p(act))
    return act


def decode_gemv2(act, ids, weights, wfmt, H, I, expert_start=0, n_local=None, fill=0x7FC0):
    """Step 3 alone: y2 [T, k, H] from act [T*k, I]."""
    act = _c(act, np.uint16)
    ids = _c(ids, np.int32)
    T, k = ids.shape
    a = _decode_args(weights)
    if n_local is None:
        n_local = a["b_gu"].shape[0]
    y2 = np.full((T, k, H), fill, np.uint16)
    lib().orc_decode_gemv2(_p(act), T, H, I, _p(ids), k, expert_start, n_local, wfmt, _p(a["w_d"]),
                           _p(a["d_scale"]), _p(a["d_sf"]), _p(a["b_d"]), _p(y2))
    return y2


def decode_sum(y2, ids, topk_w, expert_start=0, n_local=None):
    """Step 4 alone: out [T, H] from y2 [T, k, H]."""
    y2 = _c(y2, np.uint16)
    ids = _c(ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    T, k = ids.shape
    H = y2.shape[2]
    if n_local is None:
        n_local = int(ids.max()) + 1 - expert_start
    out = np.zeros((T, H), np.uint16)
    lib().orc_decode_sum(_p(y2), T, H, _p(ids), _p(topk_w), k, expert_start, n_local, _p(out))
    return out


def decode_dense(x, ids, topk_w, weights, wfmt, I, expert_start=0, n_local=None, interleaved=True,
                 alpha=1.702, beta=1.0, limit=7.0):
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    topk_w = _c(topk_w, np.float32)
    T, H = x.shape
    k = ids.shape[1]
    a = _decode_args(weights)
    if n_local is None:
        n_local = a["b_gu"].shape[0]
    out = np.zeros((T, H), np.uint16)
    lib().orc_decode_dense(_p(x), T, H, I, _p(ids), _p(topk_w), k, expert_start, n_local, wfmt,
                           _p(a["w_gu"]), _p(a["gu_scale"]), _p(a["gu_sf"]), _p(a["b_gu"]),
                           _p(a["w_d"]), _p(a["d_scale"]), _p(a["d_sf"]), _p(a["b_d"]),
                           int(bool(interleaved)), float(alpha), float(beta), float(limit), _p(out))
    return out
