"""The C-ABI library on the host: it loads, exports every symbol include/moe.h
declares, and rejects bad arguments before touching a GPU (no compute calls)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_20_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_forward_ex", "moe_workspace_size", "moe_get_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    from mixture_experts_layer_20_gb300 import binding
    for n in declared_functions():
        assert n in binding._SIGS, n


def test_host_side_validation(lib):
    from mixture_experts_layer_20_gb300 import binding as b
    L = b._lib
    vp = ctypes.c_void_p
    fake = vp(1 << 20)  # never dereferenced: every case below fails before any CUDA call
    # bad shapes
    assert L.moe_forward(fake, fake, fake, fake, 16, 100, 8, 128, 2, fake, fake, 1 << 30, None) == b.MOE_ERR_UNSUPPORTED
    assert L.moe_forward(fake, fake, fake, fake, 16, 256, 300, 128, 2, fake, fake, 1 << 30, None) == b.MOE_ERR_UNSUPPORTED
    assert L.moe_forward(fake, fake, fake, fake, 16, 256, 8, 128, 9, fake, fake, 1 << 30, None) == b.MOE_ERR_INVALID_ARG
    assert L.moe_forward(fake, fake, fake, fake, 16, 256, 4, 128, 5, fake, fake, 1 << 30, None) == b.MOE_ERR_INVALID_ARG
    assert L.moe_forward(fake, fake, fake, fake, -1, 256, 8, 128, 2, fake, fake, 1 << 30, None) == b.MOE_ERR_INVALID_ARG
    # T == 0 is a no-op
    assert L.moe_forward(None, None, None, None, 0, 256, 8, 128, 2, None, None, 0, None) == b.MOE_OK
    # null and unaligned pointers
    assert L.moe_forward(None, fake, fake, fake, 16, 256, 8, 128, 2, fake, fake, 1 << 30, None) == b.MOE_ERR_INVALID_ARG
    assert L.moe_forward(vp((1 << 20) + 8), fake, fake, fake, 16, 256, 8, 128, 2, fake, fake, 1 << 30, None) == b.MOE_ERR_INVALID_ARG
    # workspace too small
    need = b.moe_workspace_size(16, 256, 8, 128, 2)
    assert L.moe_forward(fake, fake, fake, fake, 16, 256, 8, 128, 2, fake, fake, need - 1, None) == b.MOE_ERR_WORKSPACE
    assert b"workspace" in b._lib.moe_last_error()
    assert L.moe_expert_ffn(fake, fake, fake, fake, 100, 256, 8, 96, fake, fake, 1 << 30, None) == b.MOE_ERR_UNSUPPORTED
    assert L.moe_permute(fake, None, 10, 256, 8, 2, fake, fake, fake, fake, None, fake, 256, None) == b.MOE_ERR_WORKSPACE


def test_workspace_layout():
    from mixture_experts_layer_20_gb300 import binding as b
    T, d, E, I, k, Is = 6000, 4096, 128, 1536, 8, 0
    lay = b.moe_workspace_layout(T, d, E, I, k, Is)
    assert lay["total"] == b.moe_workspace_size(T, d, E, I, k, Is)
    offs = sorted(v for n, v in lay.items() if n != "total")
    assert all(o % 256 == 0 for o in offs)
    n = T * k
    assert lay["x_perm"] + n * d * 2 <= lay["h"]
    assert lay["y"] + n * d * 2 <= lay["x_stage"]          # y: fp16
    lay5 = b.moe_workspace_layout(8192, 7168, 256, 2048, 8, 2048)
    assert lay5["y_shared"] + 8192 * 7168 * 2 <= lay5["x_stage"]
    assert lay5["out_stage"] + 8192 * 7168 * 2 == lay5["total"]


def test_status_strings():
    from mixture_experts_layer_20_gb300 import binding as b
    assert b._lib.moe_status_string(b.MOE_ERR_TIMEOUT) == b"MOE_ERR_TIMEOUT"
    assert b._lib.moe_status_string(b.MOE_ERR_RANGE) == b"MOE_ERR_RANGE"
    assert b._lib.moe_status_string(b.MOE_OK) == b"MOE_OK"
