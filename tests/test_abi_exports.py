"""The C ABI library loads on a machine without a GPU, exports every symbol
that include/*.h declares, and rejects invalid arguments on the host before
touching the device."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from moe_expert_ffn_scatter_gb300 import binding as B
from moe_expert_ffn_scatter_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_exports_only_declared_symbols():
    out = os.popen("nm -D --defined-only %s" % build_mod.LIB).read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == declared_symbols()


def test_binding_names_match_abi():
    for n in declared_symbols():
        if n in ("moe_ctx_create", "moe_ctx_destroy", "moe_status_string"):
            continue
        assert hasattr(B, n), n


def test_host_validation_without_device(lib):
    """Invalid arguments are rejected before any CUDA call (so this runs on
    CPU-only machines): NULL context, NULL args, bad sizes."""
    assert lib.moe_version() == 10000
    assert lib.moe_status_string(-1) == b"invalid argument"
    assert lib.moe_route_scatter(None, None, None) == -1
    assert lib.moe_ffn_forward(None, None, None) == -1
    assert lib.moe_sparse_gemv_decode(None, None, None) == -1
    assert lib.moe_grouped_gemm(None, None, None, 0, None, 1, 128, 128, None, None, 0, 256, 128, None, None) == -1
    p = B.moe_act_params(0, 0.0)
    assert lib.moe_act_quant(None, None, None, None, None, 1, 128, 10, 128, ctypes.byref(p), None) == -1
    assert lib.moe_combine(None, None, 8, None, None, 1, 1, 1.0, None, None) == -1
    assert lib.moe_expert_ends_from_counts(None, None, 4, 128, None, None) == -1
    # chunk histograms + the 4-byte completion count, rounded up to 16 bytes
    assert lib.moe_route_scatter_workspace_size(4096, 32, 6) == 64 * 32 * 4 + 16
    assert lib.moe_route_scatter_workspace_size(-1, 32, 6) == 0


def test_struct_layouts_match_header(tmp_path):
    """The ctypes mirrors of the argument structs have the sizes and field
    offsets that a C compiler gives the header's structs."""
    structs = {"moe_route_args": B.moe_route_args, "moe_act_params": B.moe_act_params,
               "moe_ffn_args": B.moe_ffn_args, "moe_decode_args": B.moe_decode_args}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_gb300.h"', 'int main(void) {']
    for name, cls in structs.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (name, name))
        for fname, _ in cls._fields_:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (name, fname, name, fname))
    lines += ['return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for fname, _ in cls._fields_:
            assert int(got["%s.%s" % (name, fname)]) == getattr(cls, fname).offset, (name, fname)


def test_binding_refuses_host_and_strided_tensors():
    """The binding hands only device pointers into dense buffers to the
    library: a host tensor or a strided view is refused before any call."""
    import torch

    assert B.ptr(None) is None
    with pytest.raises(ValueError, match="CUDA tensor"):
        B.ptr(torch.zeros(16, dtype=torch.int32))


def test_layer_buffer_checks():
    """The layer checks caller tensors' shapes and dtypes (the library sees
    only pointers, so a short buffer would be overrun on the device)."""
    import torch
    from moe_expert_ffn_scatter_gb300.layer import _expect

    cpu = torch.device("cpu")
    _expect("x", torch.zeros((4, 8), dtype=torch.bfloat16), (4, 8), torch.bfloat16, cpu)
    for bad in (torch.zeros((4, 7), dtype=torch.bfloat16), torch.zeros((4, 8), dtype=torch.float32)):
        with pytest.raises(ValueError, match="x: expected"):
            _expect("x", bad, (4, 8), torch.bfloat16, cpu)
    with pytest.raises(ValueError, match="required"):
        _expect("logits", None, (4, 2), torch.float32, cpu)
