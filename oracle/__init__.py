"""ctypes front end of the C oracle (test infrastructure only).

The oracle is the plain CPU statement of the W4A8 block-32 linear that the
CUDA library is checked against.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this package; the product path never
does.  fp16 arrays are numpy float16; their bit patterns go to C as uint16.
"""
import ctypes

import numpy as np

from .build import build_oracle


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test-built variant)."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P, i = ctypes.c_void_p, ctypes.c_int
        L.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_half_to_float.restype = ctypes.c_float
        L.oracle_float_to_half.argtypes = [ctypes.c_float]
        L.oracle_float_to_half.restype = ctypes.c_uint16
        L.oracle_quantize_act.argtypes = [P, i, i, P, P]
        L.oracle_block_dots.argtypes = [P, P, i, i, i, P]
        L.oracle_linear.argtypes = [P, P, P, i, i, i, P, P]
        L.oracle_linear_f64.argtypes = [P, P, P, i, i, i, P]
        L.oracle_linear_gated.argtypes = [P, P, P, i, i, i, i, P]
        L.oracle_rmsnorm_quant.argtypes = [P, P, P, ctypes.c_float, i, i, P, P, P, P]
        L.oracle_decode_attention.argtypes = [P, P, P, P, i, i, i, i, i, P]
        L.oracle_unpack_weights.argtypes = [P, i, i, P]
        for f in ("oracle_quantize_act", "oracle_block_dots", "oracle_linear",
                  "oracle_linear_f64", "oracle_linear_gated", "oracle_rmsnorm_quant", "oracle_decode_attention",
                  "oracle_unpack_weights"):
            getattr(L, f).restype = ctypes.c_int
        self.L = L
        self.path = path

    def half_to_float(self, bits: int) -> float:
        return self.L.oracle_half_to_float(int(bits))

    def float_to_half(self, f: float) -> int:
        return self.L.oracle_float_to_half(float(f))

    def quantize_act(self, x):
        """x fp16 [M][K] -> (codes int8 [M][K], scales fp32 [M][K/32])."""
        x = np.ascontiguousarray(x, np.float16)
        M, K = x.shape
        q = np.empty((M, K), np.int8)
        sx = np.empty((M, K // 32), np.float32)
        _check(self.L.oracle_quantize_act(_ptr(x), M, K, _ptr(q), _ptr(sx)), "quantize_act")
        return q, sx

    def block_dots(self, q, w):
        """q int8 [M][K], w int8 [N][K] -> int32 [M][N][K/32]."""
        q = np.ascontiguousarray(q, np.int8)
        w = np.ascontiguousarray(w, np.int8)
        M, K = q.shape
        N = w.shape[0]
        d = np.empty((M, N, K // 32), np.int32)
        _check(self.L.oracle_block_dots(_ptr(q), _ptr(w), M, N, K, _ptr(d)), "block_dots")
        return d

    def linear(self, x, w, sw, return_acc=False):
        """x fp16 [M][K], w int8 [N][K], sw fp16 [N][K/32] -> y fp16 [M][N] (and fp32 sums)."""
        x = np.ascontiguousarray(x, np.float16)
        w = np.ascontiguousarray(w, np.int8)
        sw = np.ascontiguousarray(sw, np.float16)
        M, K = x.shape
        N = w.shape[0]
        y = np.empty((M, N), np.float16)
        acc = np.empty((M, N), np.float32)
        _check(self.L.oracle_linear(_ptr(x), _ptr(w), _ptr(sw), M, N, K, _ptr(y), _ptr(acc)), "linear")
        return (y, acc) if return_acc else y

    def linear_gated(self, x, w, sw, act):
        """Gated pair: w int8 [2N][K] and sw fp16 [2N][K/32] stack gate over up rows;
        act 1 = SiLU, 2 = GELU (tanh form) -> y fp16 [M][N] = act(gate) * up."""
        x = np.ascontiguousarray(x, np.float16)
        w = np.ascontiguousarray(w, np.int8)
        sw = np.ascontiguousarray(sw, np.float16)
        M, K = x.shape
        N = w.shape[0] // 2
        y = np.empty((M, N), np.float16)
        _check(self.L.oracle_linear_gated(_ptr(x), _ptr(w), _ptr(sw), M, N, K, int(act), _ptr(y)), "linear_gated")
        return y

    def rmsnorm_quant(self, x, res, gamma, eps):
        """x, res (or None) fp16 [M][K], gamma fp16 [K] -> (residual out fp16 [M][K],
        normalised y fp16 [M][K], codes int8 [M][K], scales fp32 [M][K/32])."""
        x = np.ascontiguousarray(x, np.float16)
        M, K = x.shape
        rp = None
        if res is not None:
            res = np.ascontiguousarray(res, np.float16)
            rp = _ptr(res)
        gamma = np.ascontiguousarray(gamma, np.float16)
        ro = np.empty((M, K), np.float16)
        y = np.empty((M, K), np.float16)
        q = np.empty((M, K), np.int8)
        sx = np.empty((M, K // 32), np.float32)
        _check(self.L.oracle_rmsnorm_quant(_ptr(x), rp, _ptr(gamma), float(eps), M, K, _ptr(ro), _ptr(y), _ptr(q),
                                           _ptr(sx)), "rmsnorm_quant")
        return ro, y, q, sx

    def decode_attention(self, q, k, v, lens):
        """q fp16 [B][Hq][D], k/v fp16 [B][Hkv][Lmax][D], lens int [B] -> out fp16 [B][Hq][D]."""
        q = np.ascontiguousarray(q, np.float16)
        k = np.ascontiguousarray(k, np.float16)
        v = np.ascontiguousarray(v, np.float16)
        lens = np.ascontiguousarray(lens, np.int32)
        B, Hq, D = q.shape
        Hkv, Lmax = k.shape[1], k.shape[2]
        out = np.empty((B, Hq, D), np.float16)
        _check(self.L.oracle_decode_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(lens), B, Hq, Hkv, D, Lmax, _ptr(out)),
               "decode_attention")
        return out

    def linear_f64(self, x, w, sw):
        """fp64 dequantise-then-multiply of the same codes and scales -> float64 [M][N]."""
        x = np.ascontiguousarray(x, np.float16)
        w = np.ascontiguousarray(w, np.int8)
        sw = np.ascontiguousarray(sw, np.float16)
        M, K = x.shape
        N = w.shape[0]
        ref = np.empty((M, N), np.float64)
        _check(self.L.oracle_linear_f64(_ptr(x), _ptr(w), _ptr(sw), M, N, K, _ptr(ref)), "linear_f64")
        return ref

    def unpack_weights(self, packed, N, K):
        """Packed bytes (the library's layout) -> int8 codes [N][K]."""
        packed = np.ascontiguousarray(packed, np.uint8).reshape(-1)
        if packed.size != N * K // 2:
            raise ValueError("packed buffer has the wrong size")
        w = np.empty((N, K), np.int8)
        _check(self.L.oracle_unpack_weights(_ptr(packed), N, K, _ptr(w)), "unpack_weights")
        return w


_default = None


def get() -> Oracle:
    """The oracle built from oracle/w4a8_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build_oracle())
    return _default


def quantize_act(x):
    return get().quantize_act(x)


def block_dots(q, w):
    return get().block_dots(q, w)


def linear(x, w, sw, return_acc=False):
    return get().linear(x, w, sw, return_acc)


def linear_f64(x, w, sw):
    return get().linear_f64(x, w, sw)


def linear_gated(x, w, sw, act):
    return get().linear_gated(x, w, sw, act)


def rmsnorm_quant(x, res, gamma, eps):
    return get().rmsnorm_quant(x, res, gamma, eps)


def decode_attention(q, k, v, lens):
    return get().decode_attention(q, k, v, lens)


def unpack_weights(packed, N, K):
    return get().unpack_weights(packed, N, K)


def half_to_float(bits):
    return get().half_to_float(bits)


def float_to_half(f):
    return get().float_to_half(f)
