"""Independent reference pieces for pinning the oracle: library routines and
tables written from the format definitions, never the oracle's own code."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


E2M1_TABLE = np.array(golden("e2m1_values.json")["values"], dtype=np.float64)


def e4m3_decode_torch(codes):
    """e4m3 codes -> float64 through PyTorch's float8_e4m3fn type."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e4m3_encode_torch(v32):
    """fp32 -> e4m3 codes via PyTorch (round to nearest even; it does not
    saturate, so only valid for |v| < 464)."""
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def bf16_bits_to_f64(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_torch(v32):
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def e2m1_decode(packed, K):
    """packed e2m1 [..., K/2] (low nibble = even k) -> float64 [..., K]."""
    p = np.asarray(packed, np.uint8)
    lo = p & 0xF
    hi = p >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(p.shape[:-1] + (K,))
    return E2M1_TABLE[nib]


def bf16_ulp(x64):
    """Spacing of bf16 numbers at |x| (normal range)."""
    ax = np.maximum(np.abs(x64), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def fp32_ulp(x64):
    ax = np.maximum(np.abs(x64), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 23)


def unpack_scale_bytes(words, rows, G):
    """MN-major packed int32 [ceil(G/4), ld] -> bytes [rows, G]."""
    w = np.asarray(words).view(np.uint32)[:, :rows]
    b = w.T.copy().view(np.uint8).reshape(rows, -1)
    return b[:, :G]
