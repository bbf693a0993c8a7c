"""Helpers shared by the GPU tests: numpy <-> torch transfers and tolerances."""
import numpy as np
import torch

from tests.refs import bf16_bits_to_f64


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


def check_decode_tolerance(got_u16, ref_u16):
    """Decode output: the layer tolerance plus one bf16 step of the element.
    The path rounds to bf16 four times (y1, act, y2, out); summing the fp32
    dot products in another order than the oracle's single fp64 sum moves a
    value across a rounding boundary now and then, and one such flip on an
    output of 4-5 rms is already 2e-2 rms. Mean relative error <= 5e-3."""
    g = bf16_bits_to_f64(got_u16)
    r = bf16_bits_to_f64(ref_u16)
    assert np.all(np.isfinite(g))
    err = np.abs(g - r)
    rms = np.sqrt(np.mean(r * r))
    ulp = np.ldexp(1.0, np.frexp(np.abs(r))[1] - 8)
    worst = np.max(err - ulp)
    mean_rel = err.mean() / np.mean(np.abs(r))
    assert worst <= 2e-2 * rms, (worst / rms, mean_rel)
    assert mean_rel <= 5e-3, (worst / rms, mean_rel)
    return worst / rms, mean_rel

