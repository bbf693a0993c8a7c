"""Seeded synthetic inputs for the routed MoE expert FFN workloads.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no routing, no quantisation, no GEMM). The same bytes feed
the CUDA path and the CPU oracle. Every workload below is named by what it is
and its sizes; the draw order inside each generator is fixed.

Value recipes
  bf16 activations   fp32 N(0, std^2) rounded to bf16 (round to nearest even)
  router logits      fp32 N(0, 1); correction bias fp32 N(0, 0.1^2)
  MXFP4 weights      uniform random bytes: both e2m1 nibbles uniform over all
                     16 codes (low nibble = even K index); the Kimi-shaped
                     layer draws each expert from its own stream
  UE8M0 weight scale 127 + uniform integer exponent in [-6, -2]
  FP8 weights        e4m3 codes with random sign, exponent field uniform in
                     [4, 8] (magnitudes 2^-3 .. 2^1.9) and random mantissa --
                     a stand-in for e4m3(N(0,1)) drawn as raw code bits
"""
from dataclasses import dataclass, field

import numpy as np


def rng(seed):
    return np.random.default_rng(seed)


def f32_to_bf16_bits(a):
    """fp32 array -> bf16 bit patterns (round to nearest even)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_normal(g, shape, std=1.0):
    return f32_to_bf16_bits(g.standard_normal(shape, dtype=np.float32) * np.float32(std))


def fp32_normal(g, shape, std=1.0):
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def e2m1_packed(g, shape_bytes):
    return g.integers(0, 256, size=shape_bytes, dtype=np.uint8)


def ue8m0_bytes(g, shape, lo=-6, hi=-2):
    return (127 + g.integers(lo, hi + 1, size=shape)).astype(np.uint8)


def e4m3_codes(g, shape, exp_lo=4, exp_hi=8):
    sign = g.integers(0, 2, size=shape, dtype=np.uint8) << 7
    ex = g.integers(exp_lo, exp_hi + 1, size=shape).astype(np.uint8) << 3
    man = g.integers(0, 8, size=shape, dtype=np.uint8)
    return (sign | ex | man).astype(np.uint8)


def pack_scale_words(scale_bytes, ld):
    """Lay per-(row, group) scale bytes [rows, G] out as the MN-major packed
    int32 array [ceil(G/4), ld]: byte (g % 4) of word [g/4][row]."""
    rows, G = scale_bytes.shape
    G4 = (G + 3) // 4
    padded = np.zeros((rows, G4 * 4), np.uint8)
    padded[:, :G] = scale_bytes
    words = padded.view(np.uint32).reshape(rows, G4).T  # [G4, rows]
    out = np.zeros((G4, ld), np.uint32)
    out[:, :rows] = words
    return out.view(np.int32)


def ids_with_counts(g, counts, k):
    """Routing ids [T, k] realising the given per-expert route counts (sum must
    be a multiple of k); routes are shuffled, a token may repeat an expert."""
    counts = np.asarray(counts, np.int64)
    flat = np.repeat(np.arange(counts.shape[0], dtype=np.int32), counts)
    g.shuffle(flat)
    assert flat.shape[0] % k == 0
    return flat.reshape(-1, k).astype(np.int32)


def align_up(x, a):
    return (x + a - 1) // a * a


def align4(n):
    return align_up(n, 4)


# ------------------------------------------------------------------ workloads
@dataclass
class FFNConfig:
    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    A: int = 128
    seed: int = 0
    routing: str = "softmax"      # "softmax" | "sigmoid_bias"
    clamp: bool = False
    limit: float = 0.0
    rsf: float = 1.0
    # weights drawn expert by expert (expert_weights) instead of in one block,
    # so that a consumer holds only the experts it needs on the host
    per_expert_weights: bool = False

    @property
    def R(self):
        return self.T * self.k

    @property
    def cap(self):
        # every route plus the worst-case alignment gap of each expert, rounded
        # up to whole A-row tiles
        return align_up(self.R + self.E * (self.A - 1), self.A)


TINY = FFNConfig("tiny MoE FFN: E=4 top-2 T=64 H=256 I=128", T=64, E=4, k=2, H=256, I=128, seed=0)
DEEPSEEK = FFNConfig("DeepSeek-style W4A8 layer: E=32 top-6 T=4096 H=4096 I=2048",
                     T=4096, E=32, k=6, H=4096, I=2048, seed=2)
KIMI = FFNConfig("Kimi-K3-shaped layer: E=896 top-16 T=2048 H=3584 I=3072 clamp 25",
                 T=2048, E=896, k=16, H=3584, I=3072, seed=4, routing="sigmoid_bias",
                 clamp=True, limit=25.0, per_expert_weights=True)

# The live-row activation-quant microbenchmark shape.
ACTQ_ROWS = 28672
ACTQ_I = 2048
ACTQ_E = 32
ACTQ_LIVE = 3072
ACTQ_SEED = 1


@dataclass
class FFNInputs:
    x: np.ndarray            # bf16 bits [T, H]
    logits: np.ndarray       # fp32 [T, E]
    bias: np.ndarray         # fp32 [E] (sigmoid routing) or None
    w13: np.ndarray          # uint8 [E, 2I, H/2]
    w13_sf: np.ndarray       # uint8 [E, 2I, H/32]
    w2: np.ndarray           # uint8 [E, H, I/2]
    w2_sf: np.ndarray        # uint8 [E, H, I/32]


def ffn_inputs(cfg: FFNConfig, weights=True):
    """Activations, router logits (+ correction bias) and, unless the config
    draws its weights per expert, the four weight arrays."""
    g = rng(cfg.seed)
    x = bf16_normal(g, (cfg.T, cfg.H))
    logits = fp32_normal(g, (cfg.T, cfg.E))
    bias = fp32_normal(g, (cfg.E,), 0.1) if cfg.routing == "sigmoid_bias" else None
    if not weights or cfg.per_expert_weights:
        return FFNInputs(x, logits, bias, None, None, None, None)
    w13 = e2m1_packed(g, (cfg.E, 2 * cfg.I, cfg.H // 2))
    w13_sf = ue8m0_bytes(g, (cfg.E, 2 * cfg.I, cfg.H // 32))
    w2 = e2m1_packed(g, (cfg.E, cfg.H, cfg.I // 2))
    w2_sf = ue8m0_bytes(g, (cfg.E, cfg.H, cfg.I // 32))
    return FFNInputs(x, logits, bias, w13, w13_sf, w2, w2_sf)


def expert_weights(cfg: FFNConfig, e):
    """MXFP4 weights of expert e alone, from its own stream (seed, 1, e):
    w13 [2I, H/2], w13_sf [2I, H/32], w2 [H, I/2], w2_sf [H, I/32]. The byte
    draws use Generator.bytes (uniform bytes, so both nibbles uniform)."""
    g = rng([cfg.seed, 1, e])

    def nibbles(shape):
        return np.frombuffer(g.bytes(int(np.prod(shape))), np.uint8).reshape(shape).copy()

    w13 = nibbles((2 * cfg.I, cfg.H // 2))
    w13_sf = ue8m0_bytes(g, (2 * cfg.I, cfg.H // 32))
    w2 = nibbles((cfg.H, cfg.I // 2))
    w2_sf = ue8m0_bytes(g, (cfg.H, cfg.I // 32))
    return w13, w13_sf, w2, w2_sf


def stacked_expert_weights(cfg: FFNConfig, experts):
    """expert_weights of the listed experts stacked along a new first axis."""
    parts = [expert_weights(cfg, int(e)) for e in experts]
    return tuple(np.stack([p[i] for p in parts]) for i in range(4))


def actq_inputs(rows=ACTQ_ROWS, I=ACTQ_I, E=ACTQ_E, live=ACTQ_LIVE, seed=ACTQ_SEED, full=False):
    """gate/up buffer [rows, 2I] of bf16 N(0,1) values (gate = columns [0, I),
    up = [I, 2I)) and per-expert live-row counts: multinomial over E equally
    likely experts, or rows/E each when `full`. Which rows are live follows
    from the counts through the endpoint layout; callers overwrite the other
    rows with NaN."""
    g = rng(seed)
    if full:
        counts = np.full(E, rows // E, np.int32)
    else:
        counts = g.multinomial(live, np.full(E, 1.0 / E)).astype(np.int32)
    gateup = bf16_normal(g, (rows, 2 * I))
    return gateup, counts


@dataclass
class DecodeInputs:
    x: np.ndarray
    logits: np.ndarray
    fp8: dict = field(default_factory=dict)
    mxfp4: dict = field(default_factory=dict)


DECODE_E = 32
DECODE_K = 4
DECODE_H = 2880
DECODE_I = 2880
DECODE_SEED = 3


def decode_inputs(T, E=DECODE_E, H=DECODE_H, I=DECODE_I, seed=DECODE_SEED, fp8=True, mxfp4=True):
    g = rng(seed)
    x = bf16_normal(g, (T, H))
    logits = fp32_normal(g, (T, E))
    out = DecodeInputs(x, logits)
    if fp8:
        out.fp8 = dict(
            w_gu=e4m3_codes(g, (E, 2 * I, H)),
            gu_scale=(np.float32(2.0 ** -6) * (1 + g.random(E, dtype=np.float32))).astype(np.float32),
            b_gu=bf16_normal(g, (E, 2 * I), 0.1),
            w_d=e4m3_codes(g, (E, H, I)),
            d_scale=(np.float32(2.0 ** -6) * (1 + g.random(E, dtype=np.float32))).astype(np.float32),
            b_d=bf16_normal(g, (E, H), 0.1),
        )
    if mxfp4:
        out.mxfp4 = dict(
            w_gu=e2m1_packed(g, (E, 2 * I, H // 2)),
            gu_sf=ue8m0_bytes(g, (E, 2 * I, H // 32)),
            b_gu=bf16_normal(g, (E, 2 * I), 0.1),
            w_d=e2m1_packed(g, (E, H, I // 2)),
            d_sf=ue8m0_bytes(g, (E, H, I // 32)),
            b_d=bf16_normal(g, (E, H), 0.1),
        )
    return out
