"""The C-ABI library builds, loads and exports every declared entry point.

No compute call is made here (no GPU on this machine): only symbol lookup and
argument checks that return before any CUDA call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "while", "return"):
                names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import moe_layers_gb300 as M
    M.build()
    return M._load()


def test_header_declares_the_api():
    names = declared_functions()
    for required in ("dec_create", "dec_linear", "dec_linear_residual", "moe_route_topk", "moe_experts",
                     "decode_layer", "dec_status_string", "dec_check_device_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(lib):
    for s in range(5):
        assert lib.dec_status_string(s)
    assert lib.dec_status_string(99) == b"unknown status"


def test_null_handle_is_rejected_before_any_cuda_call(lib):
    INVALID = 1
    assert lib.dec_linear(None, None, 0, None, None, 1, 1, 8, None, 0, None) == INVALID
    assert lib.dec_linear_residual(None, None, 0, None, None, None, 1, 1, 8, None, 0, None) == INVALID
    assert lib.dec_rmsnorm(None, None, None, None, 1, 8, ctypes.c_float(1e-6), None) == INVALID
    assert lib.moe_route_topk(None, None, None, 1, 8, 8, 1, None, None, None, None, 0, None) == INVALID
    assert lib.dec_set_force_variant(None, 0) == INVALID
    assert lib.dec_last_variant(None) == 0
    assert lib.dec_destroy(None) == 0
    assert lib.dec_create(None, 0) == INVALID
