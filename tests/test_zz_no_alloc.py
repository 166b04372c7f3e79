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

import oracle
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


def _codes_of(w4, packed, N, K):
    """The weight codes back from the packed buffer (the oracle's own reader)."""
    return oracle.unpack_weights(packed.cpu().numpy(), N, K)


def _case(w4, M, N, K, seed):
    x = wl.make_x(M, K, seed, outlier_frac=0.01).cuda()
    codes, scales = wl.make_weights(N, K, seed + 1, 0.002, 0.01)
    packed = w4.pack(codes.cuda())
    return x, packed, scales.cuda()


def test_noalloc_matches_prefill_entry_point_twice(w4):
    # Both entry points run the same quantisation pass and the same GEMM, so
    # their outputs must be identical bit for bit, on each of two calls in a
    # row.  The shapes alternate between large and small scratch footprints,
    # and the last one (M=512 at K=14336, 15.6 MB) is the largest the 16 MiB
    # array is documented to hold.
    for (M, N, K, seed) in ((300, 1024, 2048, 11), (64, 520, 512, 12), (512, 8192, 2048, 13),
                            (512, 256, 14336, 14)):
        assert w4.workspace_bytes(M, N, K, w4.PATH_PREFILL) <= 16 << 20
        x, packed, scales = _case(w4, M, N, K, seed)
        ref = w4.linear(x, packed, scales, path=w4.PATH_PREFILL)
        for _ in range(2):
            out = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
            assert _call_noalloc(w4, x, packed, scales, out) == 0
            torch.cuda.synchronize()
            assert torch.equal(out, ref), f"noalloc {M}x{N}x{K} differs from the prefill entry point"
        # and both meet the fp16 tolerance against the oracle on a sample of rows
        rows = np.unique(np.array([0, M // 2, M - 1]))
        yo = oracle.linear(x.cpu().numpy()[rows], _codes_of(w4, packed, N, K), scales.cpu().numpy())
        assert_fp16_close(out.cpu().numpy()[rows], yo, f"noalloc {M}x{N}x{K} vs oracle")
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
