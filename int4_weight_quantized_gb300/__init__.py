"""Python binding of the GB300 W4A8 block-32 linear (libw4a8.so, C ABI in include/w4a8.h).

Argument marshalling only: every step of the operator runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors; each call is issued on the
current torch CUDA stream.  The binding never falls back to another
implementation: if the library is missing or the GPU is not sm_103, calls
raise.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libw4a8.so")

ACT_SILU = 1
ACT_GELU_TANH = 2

PATH_AUTO = 0
PATH_DECODE = 1
PATH_PREFILL = 2
PATH_MID = 3

STATUS = {0: "W4A8_OK", 1: "W4A8_ERR_INVALID_VALUE", 2: "W4A8_ERR_MISALIGNED", 3: "W4A8_ERR_CODE_RANGE",
          4: "W4A8_ERR_CUDA", 5: "W4A8_ERR_TIMEOUT", 6: "W4A8_ERR_UNSUPPORTED", 7: "W4A8_ERR_WORKSPACE"}

_lib = None


class W4A8Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        name = STATUS.get(status, str(status))
        msg = lib().w4a8_status_string(status).decode() if _lib is not None else name
        super().__init__(f"{what}: {name} ({msg})")


def lib():
    """The loaded C library (loaded on first use; raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run int4_weight_quantized_gb300.build.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.w4a8_status_string.argtypes = [i]
        L.w4a8_status_string.restype = ctypes.c_char_p
        L.w4a8_packed_bytes.argtypes = [i, i]
        L.w4a8_packed_bytes.restype = sz
        L.w4a8_pack.argtypes = [P, i, i, P, P]
        L.w4a8_select_path.argtypes = [i, i, i]
        L.w4a8_select_path.restype = i
        L.w4a8_prefill_splits.argtypes = [i, i, i]
        L.w4a8_prefill_splits.restype = i
        L.w4a8_mid_splits.argtypes = [i, i, i]
        L.w4a8_mid_splits.restype = i
        L.w4a8_gated_workspace_bytes.argtypes = [i, i, i]
        L.w4a8_gated_workspace_bytes.restype = sz
        L.w4a8_linear_gated.argtypes = [P, P, P, i, i, i, P, i, P, sz, P]
        L.w4a8_rmsnorm_quant.argtypes = [P, P, P, ctypes.c_float, i, i, P, P, P, P, P]
        L.w4a8_linear_q8_workspace_bytes.argtypes = [i, i, i]
        L.w4a8_linear_q8_workspace_bytes.restype = sz
        L.w4a8_linear_q8.argtypes = [P, P, P, P, i, i, i, P, P, sz, P]
        L.w4a8_decode_attention_workspace_bytes.argtypes = [i, i, i, i, i]
        L.w4a8_decode_attention_workspace_bytes.restype = sz
        L.w4a8_decode_attention.argtypes = [P, P, P, P, i, i, i, i, i, P, P, sz, P]
        L.w4a8_workspace_bytes.argtypes = [i, i, i, i]
        L.w4a8_workspace_bytes.restype = sz
        L.w4a8_linear.argtypes = [P, P, P, i, i, i, P, P]
        L.w4a8_linear_ex.argtypes = [P, P, P, i, i, i, P, i, P, sz, P]
        L.w4a8_debug_quantize_act.argtypes = [P, i, i, P, P, P]
        L.w4a8_debug_block_dots.argtypes = [P, P, P, i, i, i, P, P, i, P, sz, P]
        L.w4a8_linear_prefill_noalloc.argtypes = [P, P, P, i, i, i, P, P]
        L.w4a8_debug_stream_read.argtypes = [P, sz, i, P, P]
        L.w4a8_get_device_status.argtypes = [P]
        L.w4a8_set_wait_budget.argtypes = [ctypes.c_longlong]
        L.w4a8_debug_wait_timeout.argtypes = [P]
        L.w4a8_debug_decode_plan.argtypes = [i, i, i, i, P]
        L.w4a8_debug_decode_plan.restype = i
        for f in ("w4a8_pack", "w4a8_linear", "w4a8_linear_ex", "w4a8_linear_gated", "w4a8_rmsnorm_quant",
                  "w4a8_linear_q8", "w4a8_decode_attention", "w4a8_linear_prefill_noalloc", "w4a8_debug_quantize_act",
                  "w4a8_debug_block_dots", "w4a8_debug_stream_read", "w4a8_get_device_status", "w4a8_set_wait_budget",
                  "w4a8_debug_wait_timeout"):
            getattr(L, f).restype = i
        _lib = L
    return _lib


def _check(status, what):
    if status != 0:
        raise W4A8Error(status, what)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def packed_bytes(N, K):
    return lib().w4a8_packed_bytes(N, K)


def select_path(M, N, K):
    return lib().w4a8_select_path(M, N, K)


def prefill_splits(M, N, K):
    """CTAs along K per output tile that the prefill path uses (1, 2, 4 or 8)."""
    return lib().w4a8_prefill_splits(M, N, K)


DECODE_PLAN_FIELDS = ("tokens", "code_slices", "k_groups", "rows_per_cta", "rows_per_chunk", "ring_slots",
                      "slot_bytes", "smem_bytes", "ctas", "rows_per_pass")


def debug_decode_plan(M, N, K, gated=False):
    """The streaming decode kernel's launch plan (host only): a dict of
    DECODE_PLAN_FIELDS, or None when the kernel does not take the shape."""
    buf = (ctypes.c_int * len(DECODE_PLAN_FIELDS))()
    if not lib().w4a8_debug_decode_plan(M, N, K, 1 if gated else 0, ctypes.cast(buf, ctypes.c_void_p)):
        return None
    return dict(zip(DECODE_PLAN_FIELDS, list(buf)))


def mid_splits(M, N, K):
    """CTAs along K per 128-row tile that the mid path uses (0 if it does not take the shape)."""
    return lib().w4a8_mid_splits(M, N, K)


def workspace_bytes(M, N, K, path=PATH_AUTO):
    return lib().w4a8_workspace_bytes(M, N, K, path)


def pack(codes):
    """int8 weight codes [N][K] in [-8, 7] (CUDA) -> packed uint8 [N, K//2] (synchronises)."""
    N, K = codes.shape
    _need(codes, torch.int8, (N, K), "codes")
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=codes.device)
    _check(lib().w4a8_pack(_p(codes), N, K, _p(packed), _stream()), "w4a8_pack")
    return packed


def _linear_shapes(x, packed, scales):
    M, K = x.shape
    N = scales.shape[0]
    _need(x, torch.float16, (M, K), "x")
    _need(packed, torch.uint8, (N, K // 2), "packed")
    _need(scales, torch.float16, (N, K // 32), "scales")
    return M, N, K


def make_workspace(M, N, K, path=PATH_AUTO, device="cuda"):
    """A device workspace of the size the chosen path needs (None when it needs none)."""
    n = workspace_bytes(M, N, K, path)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def linear(x, packed, scales, out=None, path=PATH_AUTO, workspace=None):
    """y = W4A8 linear of x: x fp16 [M][K], packed [N][K/2], scales fp16 [N][K/32] -> fp16 [M][N].

    Runs w4a8_linear_ex on the current stream with a caller-side workspace
    (allocated here from torch's caching allocator when not given)."""
    M, N, K = _linear_shapes(x, packed, scales)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, (M, N), "out")
    need = workspace_bytes(M, N, K, path)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().w4a8_linear_ex(_p(x), _p(packed), _p(scales), M, N, K, _p(out), path,
                                _p(workspace), wsb, _stream()), "w4a8_linear_ex")
    return out


def gated_workspace_bytes(M, N, K):
    return lib().w4a8_gated_workspace_bytes(M, N, K)


def linear_gated(x, packed_gu, scales_gu, act=ACT_SILU, out=None, workspace=None):
    """act(x . gate) * (x . up): packed_gu [2N, K/2] and scales_gu fp16 [2N, K/32]
    stack the gate rows over the up rows; returns fp16 [M][N] (w4a8_linear_gated)."""
    M, K = x.shape
    N2 = scales_gu.shape[0]
    if N2 % 2:
        raise ValueError("scales_gu must have an even number of rows (gate rows over up rows)")
    N = N2 // 2
    _need(x, torch.float16, (M, K), "x")
    _need(packed_gu, torch.uint8, (N2, K // 2), "packed_gu")
    _need(scales_gu, torch.float16, (N2, K // 32), "scales_gu")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _need(out, torch.float16, (M, N), "out")
    need = gated_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().w4a8_linear_gated(_p(x), _p(packed_gu), _p(scales_gu), M, N, K, _p(out), int(act),
                                   _p(workspace), wsb, _stream()), "w4a8_linear_gated")
    return out


def rmsnorm_quant(x, gamma, eps=1e-6, residual=None, residual_out=None, y_out=None, codes=None, sx=None):
    """RMS norm (+ residual add) of x fp16 [M][K] with gamma fp16 [K], quantised for
    the next linear: returns (codes int8 [M][K], sx fp32 [M][K/32]); residual_out and
    y_out (fp16 [M][K]) are filled when given."""
    M, K = x.shape
    _need(x, torch.float16, (M, K), "x")
    _need(gamma, torch.float16, (K,), "gamma")
    for t, nm in ((residual, "residual"), (residual_out, "residual_out"), (y_out, "y_out")):
        if t is not None:
            _need(t, torch.float16, (M, K), nm)
    if codes is None:
        codes = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if sx is None:
        sx = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    _need(codes, torch.int8, (M, K), "codes")
    _need(sx, torch.float32, (M, K // 32), "sx")
    _check(lib().w4a8_rmsnorm_quant(_p(x), _p(residual), _p(gamma), float(eps), M, K, _p(residual_out), _p(y_out),
                                    _p(codes), _p(sx), _stream()), "w4a8_rmsnorm_quant")
    return codes, sx


def linear_q8(codes, sx, packed, scales, out=None, workspace=None):
    """The linear on producer-quantised activations (codes int8 [M][K], sx fp32 [M][K/32])."""
    M, K = codes.shape
    N = scales.shape[0]
    _need(codes, torch.int8, (M, K), "codes")
    _need(sx, torch.float32, (M, K // 32), "sx")
    _need(packed, torch.uint8, (N, K // 2), "packed")
    _need(scales, torch.float16, (N, K // 32), "scales")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=codes.device)
    _need(out, torch.float16, (M, N), "out")
    need = lib().w4a8_linear_q8_workspace_bytes(M, N, K)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=codes.device)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().w4a8_linear_q8(_p(codes), _p(sx), _p(packed), _p(scales), M, N, K, _p(out), _p(workspace), wsb,
                                _stream()), "w4a8_linear_q8")
    return out


def decode_attention(q, k_cache, v_cache, lens, out=None, workspace=None):
    """Decode attention: q fp16 [B][Hq][D], caches fp16 [B][Hkv][Lmax][D], lens int32 [B]
    (device) -> fp16 [B][Hq][D] (w4a8_decode_attention)."""
    B, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    _need(q, torch.float16, (B, Hq, D), "q")
    _need(k_cache, torch.float16, (B, Hkv, Lmax, D), "k_cache")
    _need(v_cache, torch.float16, (B, Hkv, Lmax, D), "v_cache")
    _need(lens, torch.int32, (B,), "lens")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=q.device)
    _need(out, torch.float16, (B, Hq, D), "out")
    need = lib().w4a8_decode_attention_workspace_bytes(B, Hq, Hkv, D, Lmax)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().w4a8_decode_attention(_p(q), _p(k_cache), _p(v_cache), _p(lens), B, Hq, Hkv, D, Lmax, _p(out),
                                       _p(workspace), wsb, _stream()), "w4a8_decode_attention")
    return out


def linear_c(x, packed, scales, out):
    """The plain C entry point w4a8_linear (automatic path, library-managed workspace)."""
    M, N, K = _linear_shapes(x, packed, scales)
    _need(out, torch.float16, (M, N), "out")
    _check(lib().w4a8_linear(_p(x), _p(packed), _p(scales), M, N, K, _p(out), _stream()), "w4a8_linear")
    return out


def linear_prefill_noalloc(x, packed, scales, out):
    """Prefill linear through w4a8_linear_prefill_noalloc: no device allocation
    anywhere (the library's fixed scratch array holds the quantised
    activations).  For callers that cannot allocate; calls must not overlap."""
    M, N, K = _linear_shapes(x, packed, scales)
    _need(out, torch.float16, (M, N), "out")
    _check(lib().w4a8_linear_prefill_noalloc(_p(x), _p(packed), _p(scales), M, N, K, _p(out), _stream()),
           "w4a8_linear_prefill_noalloc")
    return out


def debug_quantize_act(x):
    """Activation codes int8 [M][K] and scales fp32 [M][K/32] from the library's quantiser."""
    M, K = x.shape
    _need(x, torch.float16, (M, K), "x")
    codes = torch.empty((M, K), dtype=torch.int8, device=x.device)
    sx = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    _check(lib().w4a8_debug_quantize_act(_p(x), M, K, _p(codes), _p(sx), _stream()),
           "w4a8_debug_quantize_act")
    return codes, sx


def debug_block_dots(x, packed, scales, path=PATH_AUTO, workspace=None):
    """(block dots int32 [M][N][K/32], y fp16 [M][N]) from the chosen path's debug kernel."""
    M, N, K = _linear_shapes(x, packed, scales)
    dots = torch.empty((M, N, K // 32), dtype=torch.int32, device=x.device)
    out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    need = workspace_bytes(M, N, K, path)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().w4a8_debug_block_dots(_p(x), _p(packed), _p(scales), M, N, K, _p(dots), _p(out), path,
                                       _p(workspace), wsb, _stream()), "w4a8_debug_block_dots")
    return dots, out


def debug_stream_read(buf, mode=0, sink=None):
    """Read the bytes of the CUDA tensor `buf` once (measurement aid: mode 0 bulk
    copies, mode 1 128-bit loads); returns the sink tensor (int32[152])."""
    if sink is None:
        sink = torch.zeros(152, dtype=torch.int32, device=buf.device)
    _check(lib().w4a8_debug_stream_read(_p(buf), buf.numel() * buf.element_size(), int(mode), _p(sink), _stream()),
           "w4a8_debug_stream_read")
    return sink


def get_device_status():
    """Synchronise the current stream and return (and clear) the library's device status code."""
    return lib().w4a8_get_device_status(_stream())


def set_wait_budget(cycles):
    _check(lib().w4a8_set_wait_budget(int(cycles)), "w4a8_set_wait_budget")


def debug_wait_timeout():
    _check(lib().w4a8_debug_wait_timeout(_stream()), "w4a8_debug_wait_timeout")
