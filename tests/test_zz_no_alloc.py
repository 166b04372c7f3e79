"""The allocation-free prefill entry point (w4a8_linear_prefill_noalloc).

It serves callers that cannot allocate device memory (graph-node or host
callbacks, engines that own every allocation, real-time loops).  It must give
the same results as the ordinary prefill entry point, call after call, even
though every call reuses one scratch array inside the library.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from int4_weight_quantized_gb300 import workloads as wl

from .parity import assert_fp16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    from int4_weight_quantized_gb300.build import build
    build()
    import int4_weight_quantized_gb300 as w4
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return w4


def _call_noalloc(w4, x, packed, scales, out):
    """Straight through the C ABI."""
    M, K = x.shape
    N = scales.shape[0]
    st = w4.lib().w4a8_linear_prefill_noalloc(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
        M, N, K, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _case(w4, M, N, K, seed):
    x = wl.make_x(M, K, seed, outlier_frac=0.01).cuda()
    codes, scales = wl.make_weights(N, K, seed + 1, 0.002, 0.01)
    packed = w4.pack(codes.cuda())
    return x, packed, scales.cuda()


def test_noalloc_matches_prefill_entry_point_twice(w4):
    # two different shapes back to back: the second call must not see the
    # first call's scratch contents (the smaller M leaves stale rows behind)
    for (M, N, K, seed) in ((300, 1024, 2048, 11), (64, 520, 512, 12), (512, 8192, 2048, 13)):
        x, packed, scales = _case(w4, M, N, K, seed)
        ref = w4.linear(x, packed, scales, path=w4.PATH_PREFILL)
        for _ in range(2):
            out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
            assert _call_noalloc(w4, x, packed, scales, out) == 0
            torch.cuda.synchronize()
            assert_fp16_close(out.cpu().numpy(), ref.cpu().numpy(), f"noalloc {M}x{N}x{K}")
    assert w4.get_device_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(w4):
    M, N, K = 1024, 64, 16384        # needs 32 MiB of scratch > 16 MiB
    assert w4.workspace_bytes(M, N, K, w4.PATH_PREFILL) > 16 << 20
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    packed = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((N, K // 32), dtype=torch.float16, device="cuda")
    out = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert _call_noalloc(w4, x, packed, scales, out) == 7      # W4A8_ERR_WORKSPACE
    assert np.all(out.cpu().numpy() == 0)
