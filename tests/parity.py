"""Shared comparison rules for the GPU parity tests.

Codes, scales and block dots must match the oracle bit for bit.  fp16
outputs must satisfy |y_gpu - y_oracle| <= 2e-3 * max|y_oracle| + ulp(y_oracle)
elementwise, max taken over the whole compared output, ulp being the fp16
spacing at y_oracle (2^(e-10) for a normal value in [2^e, 2^(e+1)), 2^-24 for
subnormals).  The kernels sum the per-block fp32 terms in another order than
the oracle's sequential sum (and may fuse multiply-adds), which is why the
fp16 outputs get a tolerance while the integer work does not.
"""
import numpy as np

REL_TOL = 2e-3


def ulp_fp16(y):
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def fp16_close(y_gpu, y_ref):
    """Returns (ok, worst_ratio, bound) for the tolerance above."""
    g = np.asarray(y_gpu, np.float16).astype(np.float64)
    r = np.asarray(y_ref, np.float16).astype(np.float64)
    if g.shape != r.shape:
        return False, np.inf, None
    if r.size == 0:
        return True, 0.0, 0.0
    bound = REL_TOL * np.max(np.abs(r)) + ulp_fp16(r)
    err = np.abs(g - r)
    ratio = float(np.max(err / bound))
    return bool(np.all(err <= bound)), ratio, bound


def assert_fp16_close(y_gpu, y_ref, what=""):
    ok, ratio, _ = fp16_close(y_gpu, y_ref)
    assert ok, f"{what}: fp16 output outside tolerance (worst err/bound = {ratio:.3g})"
