"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point that include/w4a8.h declares, and rejects bad arguments
before touching the device.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from int4_weight_quantized_gb300.build import build
    build()
    import int4_weight_quantized_gb300 as w4
    return w4.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "w4a8.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4a8_pack", "w4a8_linear", "w4a8_linear_ex", "w4a8_packed_bytes",
                     "w4a8_debug_quantize_act", "w4a8_debug_block_dots", "w4a8_select_path",
                     "w4a8_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/w4a8.h but not exported"


def test_status_strings(L):
    for s in range(8):
        assert L.w4a8_status_string(s)
    assert L.w4a8_status_string(99) == b"unknown status"


def test_packed_bytes(L):
    assert L.w4a8_packed_bytes(512, 256) == 512 * 128
    assert L.w4a8_packed_bytes(8192, 2048) == 8192 * 1024
    assert L.w4a8_packed_bytes(0, 256) == 0
    assert L.w4a8_packed_bytes(1, 48) == 0
    assert L.w4a8_packed_bytes(1, 16) == 0


def test_stage_aware_dispatch(L):
    # decode for a handful of tokens, prefill for a sequence
    for M in range(1, 9):
        assert L.w4a8_select_path(M, 8192, 2048) == 1
    for M in (9, 16, 64, 512):
        assert L.w4a8_select_path(M, 8192, 2048) == 2
    assert L.w4a8_select_path(0, 8192, 2048) == 0
    assert L.w4a8_select_path(1, 8192, 2000) == 0


def test_workspace_sizes(L):
    assert L.w4a8_workspace_bytes(1, 8192, 2048, 1) == 0
    assert L.w4a8_workspace_bytes(1, 8192, 2048, 0) == 0
    assert L.w4a8_workspace_bytes(0, 8192, 2048, 2) == 0


def test_bad_arguments_rejected_before_launch(L):
    P = ctypes.c_void_p
    good = P(4096)
    # shapes
    assert L.w4a8_linear(good, good, good, 0, 8, 64, good, None) == 1
    assert L.w4a8_linear(good, good, good, 1, 0, 64, good, None) == 1
    assert L.w4a8_linear(good, good, good, 1, 8, 48, good, None) == 1
    assert L.w4a8_linear(good, good, good, 1, 8, 16, good, None) == 1
    assert L.w4a8_pack(good, 8, 40, good, None) == 1
    assert L.w4a8_debug_quantize_act(good, 1, 33, good, good, None) == 1
    # pointers
    assert L.w4a8_linear(P(4100), good, good, 1, 8, 64, good, None) == 2
    assert L.w4a8_linear(good, P(0), good, 1, 8, 64, good, None) == 2
    assert L.w4a8_linear(good, good, good, 1, 8, 64, P(4104), None) == 2
    assert L.w4a8_pack(P(3), 8, 64, good, None) == 2
    assert L.w4a8_debug_quantize_act(good, 1, 64, good, P(2), None) == 2
    # path argument
    assert L.w4a8_set_wait_budget(-1) == 1
