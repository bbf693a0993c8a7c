"""One routed MoE FFN layer on one GPU: fixed-capacity buffers plus the two
C-ABI calls of the hot path (moe_route_scatter, moe_ffn_forward).

PyTorch only allocates device memory and supplies the stream; all arithmetic
runs in the library's kernels. Every buffer is allocated once at capacity and
keeps its address, so `forward` can be captured into a CUDA graph and replayed
with new routing (the endpoint tensor's contents change, its address does not).
"""
from collections import deque
from concurrent.futures import ThreadPoolExecutor

import torch

from . import binding as B
from .synth import align4


def ceil_div(a, b):
    return (a + b - 1) // b


def _expect(name, t, shape, dtype, device):
    """The library sees only pointers, so a caller buffer of the wrong size or
    type would be read or written past its end on the device: refuse it here."""
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{name}: expected {tuple(shape)} {dtype} on {device}, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device}")


class MoEFFNLayer:
    def __init__(self, ctx, *, T, E, k, H, I, A=128, cap=None, routing=B.MOE_ROUTE_SOFTMAX_TOPK,
                 act_kind=B.MOE_ACT_SILU, limit=0.0, rsf=1.0, w_format=B.MOE_GEMM_W_E2M1, fused=True,
                 situ=(4.0, 25.0), recipe="mxfp4", device="cuda"):
        """fused: run SiLU*mul and the quantisation in GEMM1's epilogue (w13 is
        prepared with gate/up rows interleaved in blocks of 128); otherwise
        GEMM1 writes the bf16 gate/up buffer and the act-quant kernel follows.
        recipe: "mxfp4" (e2m1 weights, per-32 scales; group-128 e4m3
        activations; w_format E4M3 widens the weights), "mxfp8" (e4m3 weights
        with per-32 scales, group-32 activations) or "fp8_block128" (e4m3
        weights with one scale per 128 x 128 block, group-128 activations)."""
        if recipe not in ("mxfp4", "mxfp8", "fp8_block128"):
            raise ValueError(f"unknown recipe {recipe!r}")
        self.ctx = ctx
        self.T, self.E, self.k, self.H, self.I, self.A = T, E, k, H, I, A
        if cap is None:
            cap = ceil_div(T * k + E * (A - 1), A) * A
        self.cap = cap
        self.routing = routing
        self.act_kind, self.limit, self.rsf, self.situ = act_kind, limit, rsf, situ
        self.recipe = recipe
        self.group = 32 if recipe == "mxfp8" else 128
        if recipe != "mxfp4":
            w_format = B.MOE_GEMM_W_E4M3
        self.w_format = w_format
        self.fused = fused
        self.w13_format = w_format | (B.MOE_GEMM_W_GATEUP_BLOCK128 if fused else 0)
        # the input-side flags moe_prepare_weights needs for this recipe
        self.prep_flags = {"mxfp4": 0, "mxfp8": B.MOE_GEMM_W_IN_E4M3,
                           "fp8_block128": B.MOE_GEMM_W_IN_E4M3 | B.MOE_GEMM_W_SF_BLOCK128}[recipe]
        # GEMM1 reads group-32 input scales in the MXFP8 recipe
        self.gemm1_format = self.w13_format | (B.MOE_GEMM_A_GROUP32 if self.group == 32 else 0)
        words = lambda K: ceil_div(K, 4 * self.group)
        dev = torch.device(device)
        u8, i32, f32, bf16 = torch.uint8, torch.int32, torch.float32, torch.bfloat16
        self.topk_ids = torch.empty((T, k), dtype=i32, device=dev)
        self.topk_w = torch.empty((T, k), dtype=f32, device=dev)
        self.src2dst = torch.empty((T, k), dtype=i32, device=dev)
        self.expert_ends = torch.zeros((E,), dtype=i32, device=dev)
        self.a_fp8 = torch.empty((cap, H), dtype=u8, device=dev)
        self.a_sf = torch.empty((words(H), align4(cap)), dtype=i32, device=dev)
        self.ws = torch.empty((max(16, B.moe_route_scatter_workspace_size(T, E, k)),), dtype=u8, device=dev)
        self.gateup = None if fused else torch.empty((cap, 2 * I), dtype=bf16, device=dev)
        self.act_fp8 = torch.empty((cap, I), dtype=u8, device=dev)
        self.act_sf = torch.empty((words(I), align4(cap)), dtype=i32, device=dev)
        self.down = torch.empty((cap, H), dtype=bf16, device=dev)
        self.out = torch.empty((T, H), dtype=bf16, device=dev)
        self.w13 = self.w13_sf = self.w2 = self.w2_sf = None

    # ---------------------------------------------------------------- weights
    def load_weights(self, w13, w13_sf, w2, w2_sf, stream=None):
        """Upload canonical weights and prepare them for the grouped GEMM (scale
        re-layout, optional e4m3 widening, gate/up interleave). mxfp4: packed
        e2m1 [E,N,K/2] + UE8M0 [E,N,K/32]; mxfp8: e4m3 [E,N,K] + UE8M0
        [E,N,K/32]; fp8_block128: e4m3 [E,N,K] + UE8M0 [E,N/128,K/128]."""
        dev = self.out.device
        E, H, I = self.E, self.H, self.I

        def prep(w, sf, N, K, fmt):
            w_in = torch.as_tensor(w).to(dev).contiguous()
            sf_in = torch.as_tensor(sf).to(dev).contiguous()
            if self.recipe != "mxfp4" and not fmt & B.MOE_GEMM_W_GATEUP_BLOCK128:
                w_out = w_in  # e4m3 input used as is
            elif fmt & B.MOE_GEMM_W_E4M3:
                w_out = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
            elif fmt & B.MOE_GEMM_W_GATEUP_BLOCK128:
                w_out = torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev)
            else:
                w_out = w_in
            sf_out = torch.empty((E, K // 128, N), dtype=torch.int32, device=dev)
            B.moe_prepare_weights(self.ctx, w_in, sf_in, E, N, K, fmt | self.prep_flags, w_out, sf_out,
                                  stream=stream)
            return w_out, sf_out

        self.w13, self.w13_sf = prep(w13, w13_sf, 2 * I, H, self.w13_format)
        self.w2, self.w2_sf = prep(w2, w2_sf, H, I, self.w_format)

    def load_expert_weights(self, get_expert, stream=None, threads=8, window=16):
        """Like load_weights, with the canonical arrays uploaded one expert at
        a time: get_expert(e) -> (w13 [2I,H/2], w13_sf [2I,H/32], w2 [H,I/2],
        w2_sf [H,I/32]) as host arrays, called from a few host threads; at most
        `window` experts are held on the host at a time. The canonical device
        copy of w13 is dropped once prepared."""
        dev = self.out.device
        E, H, I = self.E, self.H, self.I
        u8 = torch.uint8
        w13 = torch.empty((E, 2 * I, H // 2), dtype=u8, device=dev)
        w13_sf = torch.empty((E, 2 * I, H // 32), dtype=u8, device=dev)
        w2 = torch.empty((E, H, I // 2), dtype=u8, device=dev)
        w2_sf = torch.empty((E, H, I // 32), dtype=u8, device=dev)
        with ThreadPoolExecutor(threads) as ex:
            pending = deque(ex.submit(get_expert, e) for e in range(min(window, E)))
            for e in range(E):
                parts = pending.popleft().result()
                if e + window < E:
                    pending.append(ex.submit(get_expert, e + window))
                for dst, src in zip((w13, w13_sf, w2, w2_sf), parts):
                    dst[e].copy_(torch.from_numpy(src))
        self.load_weights(w13, w13_sf, w2, w2_sf, stream=stream)

    # ------------------------------------------------------------------ steps
    def route_scatter(self, x, logits=None, bias=None, stream=None):
        """x [T,H] bf16; logits [T,E] fp32 unless the routing is precomputed
        (then topk_ids / topk_w are filled by the caller); bias [E] fp32 for
        sigmoid routing with correction bias."""
        dev = self.out.device
        _expect("x", x, (self.T, self.H), torch.bfloat16, dev)
        if self.routing != B.MOE_ROUTE_PRECOMPUTED:
            _expect("logits", logits, (self.T, self.E), torch.float32, dev)
        if self.routing == B.MOE_ROUTE_SIGMOID_BIAS_TOPK and bias is not None:
            _expect("bias", bias, (self.E,), torch.float32, dev)
        B.moe_route_scatter(self.ctx, routing_mode=self.routing, x=x, logits=logits, corr_bias=bias,
                            topk_ids=self.topk_ids, topk_w=self.topk_w, expert_ends=self.expert_ends,
                            src2dst=self.src2dst, a_fp8=self.a_fp8, a_sf=self.a_sf, workspace=self.ws,
                            T=self.T, E=self.E, k=self.k, H=self.H, A=self.A, cap=self.cap, stream=stream,
                            quant_group=self.group)

    def ffn(self, stream=None, out=None):
        """out: [T,H] bf16 device buffer for the result (default self.out)."""
        if out is None:
            out = self.out
        _expect("out", out, (self.T, self.H), torch.bfloat16, self.out.device)
        if self.w13 is None:
            raise RuntimeError("load_weights() has not been called")
        B.moe_ffn_forward(self.ctx, a_fp8=self.a_fp8, a_sf=self.a_sf, expert_ends=self.expert_ends, w13=self.w13,
                          w13_sf=self.w13_sf, w2=self.w2, w2_sf=self.w2_sf, gateup=self.gateup,
                          act_fp8=self.act_fp8, act_sf=self.act_sf, down=self.down, topk_w=self.topk_w,
                          src2dst=self.src2dst, out=out, T=self.T, E=self.E, k=self.k, H=self.H, I=self.I,
                          A=self.A, cap=self.cap, w_format=self.gemm1_format, act_kind=self.act_kind,
                          limit=self.limit, rsf=self.rsf, stream=stream, situ=self.situ, act_group=self.group)

    def forward(self, x, logits=None, bias=None, stream=None, out=None):
        """x [T,H] bf16, logits [T,E] fp32 (device) -> out (default self.out)
        [T,H] bf16. A caller that overlaps the read-back of one step's output
        with the next step passes alternating `out` buffers."""
        self.route_scatter(x, logits, bias, stream=stream)
        self.ffn(stream=stream, out=out)
        return self.out if out is None else out
