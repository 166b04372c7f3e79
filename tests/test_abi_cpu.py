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
    # decode for a few tokens, the short-sequence tensor-core kernel up to
    # 64 tokens, prefill for a sequence
    for M in (1, 2, 3, 4):
        assert L.w4a8_select_path(M, 8192, 2048) == 1
    assert L.w4a8_select_path(4, 4096, 14336) == 3          # long rows: 4 tokens already favour the tensor cores
    assert L.w4a8_select_path(2, 4096, 14336) == 3          # K > 8192: the GEMV's codes leave registers
    assert L.w4a8_select_path(1, 4096, 14336) == 1
    assert L.w4a8_select_path(3, 2048, 8192) == 1
    assert L.w4a8_select_path(4, 2048, 8192) == 3
    assert L.w4a8_select_path(3, 14336, 4096) == 1
    assert L.w4a8_select_path(4, 14336, 4096) == 3
    for M in (5, 8, 9, 16, 33, 64):
        assert L.w4a8_select_path(M, 8192, 2048) == 3
    for M in (65, 128, 512):
        assert L.w4a8_select_path(M, 8192, 2048) == 2
    # the mid path needs K % 256 == 0; decode keeps up to 8 tokens otherwise
    assert L.w4a8_select_path(6, 8192, 2080) == 1
    assert L.w4a8_select_path(16, 8192, 2080) == 2
    assert L.w4a8_select_path(0, 8192, 2048) == 0
    assert L.w4a8_select_path(1, 8192, 2000) == 0
    # splits of the mid path: K spread over more CTAs when there are few tiles
    assert L.w4a8_mid_splits(8, 4096, 14336) >= 2
    assert L.w4a8_mid_splits(8, 8192, 2080) == 0


def test_workspace_sizes(L):
    L.w4a8_workspace_bytes.restype = ctypes.c_size_t
    assert L.w4a8_workspace_bytes(1, 8192, 2048, 1) == 0
    assert L.w4a8_workspace_bytes(1, 8192, 2048, 0) == 0
    assert L.w4a8_workspace_bytes(0, 8192, 2048, 2) == 0
    # mid path: fp16 codes [Mp][K] + fp32 scales [K/32][Mp], Mp = 16, 32 or 64
    assert L.w4a8_workspace_bytes(5, 8192, 2048, 3) == 16 * 2048 * 2 + 64 * 16 * 4
    assert L.w4a8_workspace_bytes(40, 8192, 2048, 0) == 64 * 2048 * 2 + 64 * 64 * 4


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
    # read-ceiling probe: sizes, mode and pointers are checked before any launch
    L.w4a8_debug_stream_read.argtypes = [P, ctypes.c_size_t, ctypes.c_int, P, P]
    assert L.w4a8_debug_stream_read(good, 0, 0, good, None) == 1
    assert L.w4a8_debug_stream_read(good, 24, 0, good, None) == 1
    assert L.w4a8_debug_stream_read(good, 4096, 2, good, None) == 1
    assert L.w4a8_debug_stream_read(P(4097), 4096, 0, good, None) == 2


def test_new_entry_points_reject_bad_arguments(L):
    """Shape and pointer checks of the gated pair, the RMS norm, the linear on
    codes and decode attention return before any device work (no GPU here)."""
    P = ctypes.c_void_p
    good = P(4096)
    fz = ctypes.c_size_t(0)
    # gated pair
    assert L.w4a8_linear_gated(good, good, good, 0, 8, 64, good, 1, None, fz, None) == 1
    assert L.w4a8_linear_gated(good, good, good, 1, 8, 40, good, 1, None, fz, None) == 1
    assert L.w4a8_linear_gated(good, P(4097), good, 1, 8, 64, good, 1, None, fz, None) == 2
    # RMS norm emitting codes
    f = ctypes.c_float
    assert L.w4a8_rmsnorm_quant(good, None, good, f(1e-6), 1, 40, None, None, good, good, None) == 1
    assert L.w4a8_rmsnorm_quant(good, None, good, f(-1.0), 1, 64, None, None, good, good, None) == 1
    assert L.w4a8_rmsnorm_quant(good, None, good, f(float("nan")), 1, 64, None, None, good, good, None) == 1
    assert L.w4a8_rmsnorm_quant(good, P(4098), good, f(1e-6), 1, 64, None, None, good, good, None) == 2
    assert L.w4a8_rmsnorm_quant(good, None, good, f(1e-6), 1, 64, None, P(8), good, good, None) == 2
    # linear on codes
    assert L.w4a8_linear_q8(good, good, good, good, 1, 0, 64, good, None, fz, None) == 1
    assert L.w4a8_linear_q8(P(4100), good, good, good, 1, 8, 64, good, None, fz, None) == 2
    # decode attention: D, group size and head divisibility
    assert L.w4a8_decode_attention(good, good, good, good, 1, 8, 1, 96, 64, good, None, fz, None) == 1
    assert L.w4a8_decode_attention(good, good, good, good, 1, 6, 4, 64, 64, good, None, fz, None) == 1
    assert L.w4a8_decode_attention(good, good, good, good, 1, 32, 1, 64, 64, good, None, fz, None) == 1
    assert L.w4a8_decode_attention(good, good, good, good, 1, 8, 1, 64, 0, good, None, fz, None) == 1
    assert L.w4a8_decode_attention(good, P(12), good, good, 1, 8, 1, 64, 64, good, None, fz, None) == 2


def test_new_workspace_sizes(L):
    """Workspace queries are pure host arithmetic: the fused decode routes
    need none; the unfused gated route holds the 2N-row intermediate; the
    attention combine needs space only beyond one chunk (64 tokens for head
    dimensions 128 and 256, 128 tokens for 64)."""
    L.w4a8_gated_workspace_bytes.restype = ctypes.c_size_t
    L.w4a8_linear_q8_workspace_bytes.restype = ctypes.c_size_t
    L.w4a8_decode_attention_workspace_bytes.restype = ctypes.c_size_t
    assert L.w4a8_gated_workspace_bytes(1, 8192, 2048) == 0
    assert L.w4a8_gated_workspace_bytes(64, 128, 256) >= 64 * 256 * 2
    assert L.w4a8_linear_q8_workspace_bytes(1, 8192, 2048) == 0
    assert L.w4a8_linear_q8_workspace_bytes(64, 128, 256) == L.w4a8_workspace_bytes(64, 128, 256, 2)
    assert L.w4a8_decode_attention_workspace_bytes(4, 8, 1, 256, 64) == 0
    nb = L.w4a8_decode_attention_workspace_bytes(4, 8, 1, 256, 65)
    assert nb >= 4 * 8 * 2 * 256 * 4 + 4 * 8 * 2 * 2 * 4
    assert L.w4a8_decode_attention_workspace_bytes(4, 8, 1, 256, 640) >= 4 * 8 * 10 * 256 * 4 + 4 * 8 * 10 * 2 * 4
    assert L.w4a8_decode_attention_workspace_bytes(4, 8, 1, 64, 128) == 0
    assert L.w4a8_decode_attention_workspace_bytes(4, 8, 1, 64, 129) >= 4 * 8 * 2 * 64 * 4
    assert L.w4a8_decode_attention_workspace_bytes(4, 8, 3, 256, 129) == 0      # invalid: 8 % 3
    assert L.w4a8_decode_attention_workspace_bytes(1, 8, 1, 256, 131072) > 0
    assert L.w4a8_decode_attention_workspace_bytes(1, 8, 1, 256, 131073) == 0   # past the longest cache
    assert L.w4a8_prefill_splits(512, 8192, 2048) == 1
    assert L.w4a8_prefill_splits(16, 128, 1056) == 8      # K % 256 != 0: the 128 x 128-tile kernel
    assert L.w4a8_prefill_splits(100, 256, 4096) == 8     # 128-token tiles of the streaming kernel
    assert L.w4a8_prefill_splits(0, 128, 1024) == 0


def _plan(M, N, K, gated=False):
    import int4_weight_quantized_gb300 as w4
    return w4.debug_decode_plan(M, N, K, gated)


def test_decode_plan_invariants(L):
    """The streaming decode kernel's launch plan (host arithmetic only) stays
    inside the hardware's limits and covers every row and K block, over a
    grid of shapes and both the plain and the gated kernel."""
    Ms = (1, 2, 3, 4, 5, 8, 9, 16)
    Ns = (1, 7, 64, 256, 300, 2048, 4096, 8192, 14336, 28672)
    Ks = (32, 96, 256, 1024, 2048, 3072, 4096, 6176, 8192, 10240, 14336, 16384, 28672)
    checked = 0
    for gated in (False, True):
        nv = 2 if gated else 1
        for M in Ms:
            for N in Ns:
                for K in Ks:
                    p = _plan(M, N, K, gated)
                    if p is None:
                        continue
                    checked += 1
                    nb = K // 32
                    MT = min(M, 8)
                    assert p["tokens"] == MT
                    assert 1 <= p["ring_slots"] <= 8
                    assert 1 <= p["rows_per_chunk"] <= p["rows_per_cta"]
                    assert p["slot_bytes"] % 16 == 0
                    assert p["slot_bytes"] >= p["rows_per_chunk"] * nv * K // 2
                    assert p["smem_bytes"] <= 224 * 1024
                    assert p["smem_bytes"] >= p["ring_slots"] * p["slot_bytes"] + MT * nb * 32
                    assert 1 <= p["ctas"] <= 152
                    assert p["ctas"] * p["rows_per_cta"] >= N > (p["ctas"] - 1) * p["rows_per_cta"]
                    chunks = -(-p["rows_per_cta"] // p["rows_per_chunk"])
                    assert p["ring_slots"] <= chunks
                    if p["ring_slots"] < chunks:
                        assert p["ring_slots"] >= 2            # a refilled ring never has one slot
                    assert p["code_slices"] in (0, 1, 2, 4, 8)
                    assert p["k_groups"] in (1, 2, 4)
                    if p["code_slices"]:
                        assert p["code_slices"] * 32 * p["k_groups"] >= nb
                        assert MT * p["code_slices"] <= 8
                    if p["k_groups"] > 1:
                        assert MT == 1 and p["code_slices"] == 4
                        assert 8 % p["k_groups"] == 0
                    assert p["rows_per_pass"] == min(8 // MT, 4)
    assert checked > 1000


def test_decode_plans_of_the_workloads(L):
    # headline FFN up: one 54-row chunk, small enough for three CTAs per SM
    p = _plan(1, 8192, 2048)
    assert (p["code_slices"], p["k_groups"], p["rows_per_chunk"], p["ring_slots"]) == (2, 1, 54, 1)
    assert 3 * (p["smem_bytes"] + 1024) <= 228 * 1024
    # 14336 x 4096: all 95 rows of a CTA in flight in three chunks
    p = _plan(1, 14336, 4096)
    assert p["ring_slots"] == 3 and p["ring_slots"] * p["rows_per_chunk"] >= p["rows_per_cta"]
    # long rows for one token: 4 slices of codes in 2 or 4 K groups
    p = _plan(1, 2048, 8192)
    assert (p["code_slices"], p["k_groups"], p["ring_slots"]) == (4, 2, 1)
    p = _plan(1, 4096, 14336)
    assert (p["code_slices"], p["k_groups"], p["ring_slots"]) == (4, 4, 3)
    # several tokens keep one group: codes in registers while tokens x slices <= 8
    assert _plan(2, 8192, 2048)["k_groups"] == 1
    assert _plan(8, 129, 2048)["code_slices"] == 0
    assert _plan(0, 8192, 2048) is None and _plan(1, 8192, 48) is None
