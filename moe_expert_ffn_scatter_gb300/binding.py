"""Thin Python binding of libmoe_gb300.so (the C ABI in include/moe_gb300.h).

Each function carries the name of its C entry point and only marshals
arguments: torch tensors become device pointers, the current torch stream
becomes the cudaStream_t, a non-zero status becomes a MoeError. Every step of
the path runs in the library's CUDA kernels; there is no fallback of any kind:
if the library is missing or fails to load, load() raises.
"""
import ctypes
import os

import torch

from . import build as _build

MOE_OK = 0
MOE_ROUTE_SOFTMAX_TOPK = 0
MOE_ROUTE_SIGMOID_BIAS_TOPK = 1
MOE_ROUTE_PRECOMPUTED = 2
MOE_ACT_SILU = 0
MOE_ACT_SILU_CLAMP = 1
MOE_ACT_SITU = 2
MOE_WFMT_FP8_PER_EXPERT = 0
MOE_WFMT_MXFP4_G32 = 1
MOE_GLU_HALVES = 0
MOE_GLU_INTERLEAVED = 1
MOE_DECODE_AUTO = 0
MOE_DECODE_TCGEN05 = 1
MOE_DECODE_MMA_SYNC = 2
MOE_DECODE_GEMV = 3
MOE_GEMM_W_E2M1 = 0
MOE_GEMM_W_E4M3 = 1
MOE_GEMM_W_GATEUP_BLOCK128 = 2
MOE_GEMM_W_IN_E4M3 = 4
MOE_GEMM_W_SF_BLOCK128 = 8
MOE_GEMM_A_GROUP32 = 16
MOE_DEVERR_EXPERT_ID = 0x1
MOE_DEVERR_CAPACITY = 0x2
MOE_DEVERR_WAIT_TIMEOUT = 0x4
MOE_DEVERR_ENDPOINTS = 0x8

_P = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_F = ctypes.c_float


class MoeError(RuntimeError):
    def __init__(self, name, status, msg):
        super().__init__("%s failed: status %d (%s)" % (name, status, msg))
        self.status = status


class moe_route_args(ctypes.Structure):
    _fields_ = [("routing_mode", _I32), ("logits", _P), ("corr_bias", _P), ("topk_ids", _P), ("topk_w", _P),
                ("x", _P), ("a_fp8", _P), ("a_sf", _P), ("expert_ends", _P), ("src2dst", _P),
                ("workspace", _P), ("workspace_bytes", ctypes.c_size_t),
                ("T", _I32), ("E", _I32), ("k", _I32), ("H", _I32), ("A", _I32), ("cap", _I32),
                ("quant_group", _I32)]


class moe_act_params(ctypes.Structure):
    _fields_ = [("kind", _I32), ("limit", _F), ("situ_beta_s", _F), ("situ_beta_l", _F), ("quant_group", _I32)]


def act_params(kind=0, limit=0.0, situ=(4.0, 25.0), group=128):
    """moe_act_params for SiLU / SiLU with clamp limit / SiTU (situ = (beta_s,
    beta_l)); group: quantisation group of the result, 128 or 32 (MXFP8)."""
    return moe_act_params(kind, limit, float(situ[0]), float(situ[1]), group)


class moe_ffn_args(ctypes.Structure):
    _fields_ = [("a_fp8", _P), ("a_sf", _P), ("expert_ends", _P), ("w13", _P), ("w13_sf", _P), ("w2", _P),
                ("w2_sf", _P), ("gateup", _P), ("act_fp8", _P), ("act_sf", _P), ("down", _P), ("topk_w", _P),
                ("src2dst", _P), ("out", _P),
                ("T", _I32), ("E", _I32), ("k", _I32), ("H", _I32), ("I", _I32), ("A", _I32), ("cap", _I32),
                ("w_format", _I32), ("act", moe_act_params), ("rsf", _F)]


class moe_decode_args(ctypes.Structure):
    _fields_ = [("x", _P), ("topk_ids", _P), ("topk_w", _P),
                ("expert_start", _I32), ("num_local_experts", _I32), ("wfmt", _I32),
                ("w_gu", _P), ("w_gu_scale", _P), ("w_gu_sf", _P), ("b_gu", _P),
                ("w_d", _P), ("w_d_scale", _P), ("w_d_sf", _P), ("b_d", _P),
                ("glu_layout", _I32), ("glu_alpha", _F), ("glu_beta", _F), ("glu_limit", _F),
                ("y1", _P), ("act", _P), ("y2", _P), ("out", _P),
                ("T", _I32), ("H", _I32), ("I", _I32), ("k", _I32),
                ("workspace", _P), ("workspace_bytes", ctypes.c_size_t), ("path", _I32)]


_SIGS = {
    "moe_version": (_I, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_ctx_create": (_I, [ctypes.POINTER(_P), _I]),
    "moe_ctx_destroy": (_I, [_P]),
    "moe_get_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "moe_expert_ends_from_counts": (_I, [_P, _P, _I, _I, _P, _P]),
    "moe_route_scatter_workspace_size": (ctypes.c_size_t, [_I, _I, _I]),
    "moe_route_scatter": (_I, [_P, ctypes.POINTER(moe_route_args), _P]),
    "moe_route_scatter_noalloc": (_I, [_P, ctypes.POINTER(moe_route_args), _P]),
    "moe_prepare_weights": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_gemm": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P]),
    "moe_grouped_gemm_act_quant": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _P, _P, _I, _I, _I,
                                        ctypes.POINTER(moe_act_params), _P, _P, _P]),
    "moe_act_quant": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.POINTER(moe_act_params), _P]),
    "moe_combine": (_I, [_P, _P, _I, _P, _P, _I, _I, _F, _P, _P]),
    "moe_ffn_forward": (_I, [_P, ctypes.POINTER(moe_ffn_args), _P]),
    "moe_decode_workspace_size": (ctypes.c_size_t, [_I32, _I32, _I32, _I32, _I32]),
    "moe_sparse_gemv_decode": (_I, [_P, ctypes.POINTER(moe_decode_args), _P]),
}

_lib = None


def lib_path():
    return _build.LIB


def load(build_if_missing=True):
    """Load the CUDA library (building it in-tree first if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError("libmoe_gb300.so not built: run __graft_entry__.build()")
        _build.build()
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(name, status):
    if status != MOE_OK:
        raise MoeError(name, status, load().moe_status_string(status).decode())


def ptr(t):
    """Device pointer of a CUDA tensor; None passes NULL.

    Every buffer the library takes is a dense device array, so a host tensor
    (whose address a kernel cannot dereference) or a strided view (whose
    elements are not where the library reads them) is refused here, before
    anything is enqueued."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got shape {tuple(t.shape)} strides {t.stride()}")
    return t.data_ptr()


def cur_stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Context:
    """Owns a moe_ctx (the device error word and device facts)."""

    def __init__(self, device=0):
        self.device = device
        h = ctypes.c_void_p()
        _check("moe_ctx_create", load().moe_ctx_create(ctypes.byref(h), device))
        self.handle = h

    def close(self):
        if self.handle:
            load().moe_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_version():
    return load().moe_version()


def moe_get_device_error(ctx, stream=None):
    bits = ctypes.c_uint32(0)
    _check("moe_get_device_error", load().moe_get_device_error(ctx.handle, ctypes.byref(bits), cur_stream(stream)))
    return bits.value


def moe_expert_ends_from_counts(ctx, counts, A, expert_ends, stream=None):
    _check("moe_expert_ends_from_counts",
           load().moe_expert_ends_from_counts(ctx.handle, ptr(counts), counts.numel(), A, ptr(expert_ends),
                                              cur_stream(stream)))


def moe_route_scatter_workspace_size(T, E, k):
    return load().moe_route_scatter_workspace_size(T, E, k)


def moe_route_scatter(ctx, *, routing_mode, x, topk_ids, expert_ends, src2dst, a_fp8, a_sf, workspace,
                      T, E, k, H, A, cap, logits=None, corr_bias=None, topk_w=None, stream=None, quant_group=128):
    a = moe_route_args(routing_mode, ptr(logits), ptr(corr_bias), ptr(topk_ids), ptr(topk_w), ptr(x),
                       ptr(a_fp8), ptr(a_sf), ptr(expert_ends), ptr(src2dst), ptr(workspace),
                       workspace.numel() * workspace.element_size(), T, E, k, H, A, cap, quant_group)
    _check("moe_route_scatter", load().moe_route_scatter(ctx.handle, ctypes.byref(a), cur_stream(stream)))


def moe_route_scatter_noalloc(ctx, *, routing_mode, x, topk_ids, expert_ends, src2dst, a_fp8, a_sf,
                              T, E, k, H, A, cap, logits=None, corr_bias=None, topk_w=None, stream=None,
                              quant_group=128):
    """moe_route_scatter without a caller workspace: the library's built-in
    scratch array is used (for callers that cannot allocate device memory)."""
    a = moe_route_args(routing_mode, ptr(logits), ptr(corr_bias), ptr(topk_ids), ptr(topk_w), ptr(x),
                       ptr(a_fp8), ptr(a_sf), ptr(expert_ends), ptr(src2dst), None, 0, T, E, k, H, A, cap,
                       quant_group)
    _check("moe_route_scatter_noalloc",
           load().moe_route_scatter_noalloc(ctx.handle, ctypes.byref(a), cur_stream(stream)))


def moe_prepare_weights(ctx, w_in, sf_in, E, N, K, w_format, w_out, sf_out, stream=None):
    _check("moe_prepare_weights",
           load().moe_prepare_weights(ctx.handle, ptr(w_in), ptr(sf_in), E, N, K, w_format, ptr(w_out),
                                      ptr(sf_out), cur_stream(stream)))


def moe_grouped_gemm(ctx, a, a_sf, ld_sf, expert_ends, E, A, cap, w, w_sf, w_format, N, K, out, stream=None):
    _check("moe_grouped_gemm",
           load().moe_grouped_gemm(ctx.handle, ptr(a), ptr(a_sf), ld_sf, ptr(expert_ends), E, A, cap, ptr(w),
                                   ptr(w_sf), w_format, N, K, ptr(out), cur_stream(stream)))


def moe_grouped_gemm_act_quant(ctx, a, a_sf, ld_sf, expert_ends, E, A, cap, w13, w13_sf, w_format, I, K,
                               out_fp8, out_sf, kind=MOE_ACT_SILU, limit=0.0, stream=None, situ=(4.0, 25.0),
                               group=128):
    p = act_params(kind, limit, situ, group)
    _check("moe_grouped_gemm_act_quant",
           load().moe_grouped_gemm_act_quant(ctx.handle, ptr(a), ptr(a_sf), ld_sf, ptr(expert_ends), E, A, cap,
                                             ptr(w13), ptr(w13_sf), w_format, I, K, ctypes.byref(p), ptr(out_fp8),
                                             ptr(out_sf), cur_stream(stream)))


def moe_act_quant(ctx, gateup, out, out_sf, expert_ends, E, A, M_alloc, I, kind=MOE_ACT_SILU, limit=0.0,
                  stream=None, situ=(4.0, 25.0), group=128):
    p = act_params(kind, limit, situ, group)
    _check("moe_act_quant",
           load().moe_act_quant(ctx.handle, ptr(gateup), ptr(out), ptr(out_sf), ptr(expert_ends), E, A, M_alloc,
                                I, ctypes.byref(p), cur_stream(stream)))


def moe_combine(ctx, down, H, topk_w, src2dst, T, k, rsf, out, stream=None):
    _check("moe_combine",
           load().moe_combine(ctx.handle, ptr(down), H, ptr(topk_w), ptr(src2dst), T, k, float(rsf), ptr(out),
                              cur_stream(stream)))


def moe_ffn_forward(ctx, *, a_fp8, a_sf, expert_ends, w13, w13_sf, w2, w2_sf, gateup, act_fp8, act_sf, down,
                    topk_w, src2dst, out, T, E, k, H, I, A, cap, w_format=MOE_GEMM_W_E2M1, act_kind=MOE_ACT_SILU,
                    limit=0.0, rsf=1.0, stream=None, situ=(4.0, 25.0), act_group=128):
    a = moe_ffn_args(ptr(a_fp8), ptr(a_sf), ptr(expert_ends), ptr(w13), ptr(w13_sf), ptr(w2), ptr(w2_sf),
                     ptr(gateup), ptr(act_fp8), ptr(act_sf), ptr(down), ptr(topk_w), ptr(src2dst), ptr(out),
                     T, E, k, H, I, A, cap, w_format, act_params(act_kind, limit, situ, act_group), rsf)
    _check("moe_ffn_forward", load().moe_ffn_forward(ctx.handle, ctypes.byref(a), cur_stream(stream)))


def moe_sparse_gemv_decode(ctx, *, x, topk_ids, topk_w, expert_start, num_local_experts, wfmt, w_gu, b_gu, w_d,
                           b_d, y1, act, y2, out, T, H, I, k, w_gu_scale=None, w_gu_sf=None, w_d_scale=None,
                           w_d_sf=None, glu_layout=MOE_GLU_INTERLEAVED, glu_alpha=1.702, glu_beta=1.0,
                           glu_limit=7.0, workspace=None, path=None, stream=None):
    """workspace: a uint8 device tensor of at least moe_decode_workspace_size()
    bytes enables the tcgen05 path (T <= 128); path: MOE_DECODE_* (default
    AUTO: tcgen05 from T >= 8 (FP8) / T >= 4 (MXFP4) when it applies, else
    mma.sync, else GEMV)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a = moe_decode_args(ptr(x), ptr(topk_ids), ptr(topk_w), expert_start, num_local_experts, wfmt,
                        ptr(w_gu), ptr(w_gu_scale), ptr(w_gu_sf), ptr(b_gu), ptr(w_d), ptr(w_d_scale), ptr(w_d_sf),
                        ptr(b_d), glu_layout, glu_alpha, glu_beta, glu_limit, ptr(y1), ptr(act), ptr(y2), ptr(out),
                        T, H, I, k, ptr(workspace), ws_bytes, MOE_DECODE_AUTO if path is None else path)
    _check("moe_sparse_gemv_decode", load().moe_sparse_gemv_decode(ctx.handle, ctypes.byref(a), cur_stream(stream)))


def moe_decode_workspace_size(T, k, H, I, num_local_experts):
    return int(load().moe_decode_workspace_size(T, k, H, I, num_local_experts))


def decode_workspace(T, k, H, I, num_local_experts, device="cuda"):
    """Device workspace of the tcgen05 decode path (uint8 tensor)."""
    n = moe_decode_workspace_size(T, k, H, I, num_local_experts)
    if n == 0:
        raise ValueError("decode sizes out of range")
    return torch.empty(n, dtype=torch.uint8, device=device)
