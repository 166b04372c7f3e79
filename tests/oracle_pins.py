"""Pins of the CPU oracle against facts fixed outside it.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with a closed form, a hand-derived vector, a brute
force count, a library routine on a special case, or an exact invariant.
None of them compares the oracle with a copy of its own formulas.
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with a planted mistake and checks that at
least one pin fails for every such copy.

Passages: 4-bit weights in blocks of 32 and in-kernel activation
quantisation ("Що змінює ML Drift для on-device AI-інференсу на вашому
телефоні?", tech.dede.sh, section "Stage-aware оптимізація для великих
мовних моделей").  The quantiser reading (fp32 amax/127 scale, one fp32
division, ties to even, clamp +-127) is the plainest one those pages support.
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _f32_bits(v):
    return int(np.array([v], np.float32).view(np.uint32)[0])


def load_quant_blocks():
    """Parse tests/golden/quant_blocks.txt -> list of (name, x fp16[32], q int8[32], s_bits)."""
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "quant_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("block "):
                cur = {"name": line.split()[1]}
                blocks.append(cur)
            elif line.startswith("x:"):
                v = [int(t, 16) for t in line[2:].split()]
                cur["x"] = np.array(v + [0] * (32 - len(v)), np.uint16).view(np.float16)
            elif line.startswith("q:"):
                v = [int(t) for t in line[2:].split()]
                cur["q"] = np.array(v + [0] * (32 - len(v)), np.int8)
            elif line.startswith("s:"):
                cur["s"] = int(line[2:].strip(), 16)
    return [(b["name"], b["x"], b["q"], b["s"]) for b in blocks]


# ---------------------------------------------------------------- fp16 format

def pin_half_to_float_exhaustive(orc):
    """All 65536 binary16 patterns against numpy's float16 -> float32 conversion."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.half_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_float_to_half_sample(orc):
    """Random fp32 bit patterns and the rounding edge cases against numpy's float32 -> float16."""
    r = _rng(1)
    pats = r.integers(0, 2**32, 60000, dtype=np.uint64).astype(np.uint32)
    # concentrate on the fp16 range: exponents 2^-26 .. 2^17
    e = r.integers(127 - 26, 127 + 17, 60000).astype(np.uint32)
    pats2 = (pats & np.uint32(0x807FFFFF)) | (e << np.uint32(23))
    edge = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, -65520.0, 1e30, 2.0**-24, 2.0**-25,
                     1.5 * 2.0**-25, 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11,
                     1.0 + 3 * 2.0**-11, 2049.0, 2051.0, np.inf, -np.inf], np.float32)
    vals = np.concatenate([pats.view(np.float32), pats2.view(np.float32), edge])
    vals = vals[~np.isnan(vals)]
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.float_to_half(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref), vals[got != ref][:5]


# ---------------------------------------------------- activation quantisation

def pin_golden_blocks(orc):
    """Hand-derived blocks of tests/golden/quant_blocks.txt: codes and scale bits."""
    for name, x, q, s in load_quant_blocks():
        gq, gs = orc.quantize_act(x.reshape(1, 32))
        assert np.array_equal(gq[0], q), (name, gq[0], q)
        assert _f32_bits(gs[0, 0]) == s, (name, hex(_f32_bits(gs[0, 0])), hex(s))


def pin_golden_blocks_in_rows(orc):
    """The golden blocks placed side by side in one row and in several rows
    keep their codes and scales: blocks are the aligned 32-column groups of
    each token, independent of one another."""
    blocks = load_quant_blocks()
    x = np.concatenate([b[1] for b in blocks]).reshape(1, -1)
    q, s = orc.quantize_act(x)
    for i, (name, _, qb, sb) in enumerate(blocks):
        assert np.array_equal(q[0, 32 * i:32 * i + 32], qb), name
        assert _f32_bits(s[0, i]) == sb, name
    x2 = np.stack([np.concatenate([blocks[i][1], blocks[(i + 1) % len(blocks)][1]])
                   for i in range(len(blocks))])
    q2, s2 = orc.quantize_act(x2)
    for i in range(len(blocks)):
        assert np.array_equal(q2[i, :32], blocks[i][2])
        assert np.array_equal(q2[i, 32:], blocks[(i + 1) % len(blocks)][2])


def pin_pow2_invariance(orc):
    """x * 2^j (no overflow or underflow) gives the same codes and s * 2^j."""
    r = _rng(2)
    # multiples of 2^-8 (or 0): every scaling below stays exact in fp16
    x = (r.integers(-4000, 4000, (8, 128)) / 256.0).astype(np.float16)
    q0, s0 = orc.quantize_act(x)
    for j in (-6, -3, -1, 1, 2, 5):
        xj = (x.astype(np.float32) * np.float32(2.0 ** j)).astype(np.float16)
        assert np.array_equal(xj.astype(np.float32), x.astype(np.float32) * np.float32(2.0 ** j))
        qj, sj = orc.quantize_act(xj)
        assert np.array_equal(qj, q0)
        assert np.array_equal(sj, s0 * np.float32(2.0 ** j))


def pin_subnormal_inputs(orc):
    """Subnormal fp16 inputs m*2^-24 quantise like the normal values m*2^-10
    (an exact 2^-14 scaling), with the scale divided by 2^14."""
    r = _rng(3)
    m = r.integers(-1023, 1024, (4, 64))
    sub = np.where(m < 0, 0x8000 | (-m), m).astype(np.uint16).view(np.float16)
    nrm = (m.astype(np.float64) * 2.0 ** -10).astype(np.float16)
    assert np.array_equal(nrm.astype(np.float64), m * 2.0 ** -10)
    qs, ss = orc.quantize_act(sub)
    qn, sn = orc.quantize_act(nrm)
    assert np.array_equal(qs, qn)
    assert np.array_equal(ss, sn * np.float32(2.0 ** -14))


def pin_code_range_and_extremes(orc):
    """Codes stay in [-127,127]; each block's largest |x| gets code +-127; the
    sign of every code follows the sign of x; |q*s - x| <= s/2 up to fp32 rounding."""
    r = _rng(4)
    x = (r.standard_normal((16, 256)) * r.choice([0.01, 1, 300], (16, 1))).astype(np.float16)
    q, s = orc.quantize_act(x)
    assert q.min() >= -127 and q.max() <= 127
    xf = x.astype(np.float64).reshape(16, 8, 32)
    qb = q.astype(np.int32).reshape(16, 8, 32)
    idx = np.abs(xf).argmax(axis=2)
    top = np.take_along_axis(qb, idx[..., None], 2)[..., 0]
    assert np.all(np.abs(top) == 127)
    assert np.all((qb == 0) | (np.sign(qb) == np.sign(xf)))
    err = np.abs(qb * s.astype(np.float64)[..., None] - xf)
    assert np.all(err <= s.astype(np.float64)[..., None] * (0.5 + 1e-5))


# ------------------------------------------------------------ integer dots

def pin_block_dots_bruteforce(orc):
    """Block dots against numpy's integer einsum on small random shapes."""
    r = _rng(5)
    for (M, N, K) in ((1, 1, 32), (3, 5, 64), (2, 7, 160)):
        q = r.integers(-127, 128, (M, K)).astype(np.int8)
        w = r.integers(-8, 8, (N, K)).astype(np.int8)
        ref = np.einsum("mbk,nbk->mnb", q.reshape(M, K // 32, 32).astype(np.int64),
                        w.reshape(N, K // 32, 32).astype(np.int64))
        assert np.array_equal(orc.block_dots(q, w), ref)


def pin_block_dots_extremes(orc):
    """All -8 weights against all -127 codes give 32*8*127 = 32512 per block;
    against all +127 codes, -32512."""
    q = np.full((2, 64), -127, np.int8)
    q[1] = 127
    w = np.full((1, 64), -8, np.int8)
    d = orc.block_dots(q, w)
    assert np.all(d[0] == 32512) and np.all(d[1] == -32512)


def pin_block_dots_symmetries(orc):
    """Negating W negates every dot; permuting the 32-blocks of q and W together permutes the dots."""
    r = _rng(6)
    q = r.integers(-127, 128, (3, 128)).astype(np.int8)
    w = r.integers(-7, 8, (4, 128)).astype(np.int8)
    d = orc.block_dots(q, w)
    assert np.array_equal(orc.block_dots(q, -w), -d)
    perm = np.array([2, 0, 3, 1])
    qp = q.reshape(3, 4, 32)[:, perm].reshape(3, 128)
    wp = w.reshape(4, 4, 32)[:, perm].reshape(4, 128)
    assert np.array_equal(orc.block_dots(qp, wp), d[:, :, perm])


# ------------------------------------------------------------- whole linear

def pin_linear_closed_form(orc):
    """Rows built from the golden blocks with weights 1 and unit scales give
    the sum of their codes times their scales, exactly:
    amax_127 codes sum to 128 (s = 1), amax_63_5 codes sum to 135 (s = 0.5),
    so y = 128 + 67.5 = 195.5; with weights 2 and scales 0.25 the result halves."""
    blocks = {b[0]: b for b in load_quant_blocks()}
    x = np.concatenate([blocks["amax_127"][1], blocks["amax_63_5"][1]]).reshape(1, 64)
    w = np.ones((3, 64), np.int8)
    sw = np.ones((3, 2), np.float16)
    y, acc = orc.linear(x, w, sw, return_acc=True)
    assert np.all(acc == 195.5) and np.all(y == np.float16(195.5))
    y2 = orc.linear(x, 2 * w, np.full((3, 2), 0.25, np.float16))
    assert np.all(y2 == np.float16(97.75))


def pin_linear_all_ones(orc):
    """Weights 1 and unit scales: every output column equals the same row sum
    sum_b s_x[b] * sum_k q[k], which lies within sum_b 16*s_x[b] (half a step
    per element) of sum_k x[k]."""
    r = _rng(7)
    M, N, K = 4, 6, 256
    x = (r.standard_normal((M, K)) * 2).astype(np.float16)
    w = np.ones((N, K), np.int8)
    sw = np.ones((N, K // 32), np.float16)
    _, acc = orc.linear(x, w, sw, return_acc=True)
    assert np.all(acc == acc[:, :1])
    _, s = orc.quantize_act(x)
    bound = 16.0 * s.astype(np.float64).sum(1) * (1 + 1e-5) + 1e-6
    dev = np.abs(acc[:, 0].astype(np.float64) - x.astype(np.float64).sum(1))
    assert np.all(dev <= bound), (dev, bound)


def pin_linear_vs_f64(orc):
    """fp32 accumulation against an fp64 dequantise-then-matmul done with numpy
    (codes and scales from the quantiser): within the fp32 rounding bound
    (nb + 3) * 2^-24 * sum_b |d_b * s_w * s_x|.  Also pins the oracle's own
    fp64 checker to the numpy product."""
    r = _rng(8)
    for (M, N, K) in ((1, 8, 64), (3, 5, 256), (2, 4, 1024)):
        x = (r.standard_normal((M, K)) * 1.5).astype(np.float16)
        w = r.integers(-8, 8, (N, K)).astype(np.int8)
        sw = r.uniform(0.002, 0.02, (N, K // 32)).astype(np.float16)
        q, s = orc.quantize_act(x)
        nb = K // 32
        deq_x = (q.astype(np.float64).reshape(M, nb, 32) * s.astype(np.float64)[..., None]).reshape(M, K)
        deq_w = (w.astype(np.float64).reshape(N, nb, 32) * sw.astype(np.float64)[..., None]).reshape(N, K)
        ref = deq_x @ deq_w.T
        assert np.allclose(orc.linear_f64(x, w, sw), ref, rtol=1e-12, atol=1e-12)
        _, acc = orc.linear(x, w, sw, return_acc=True)
        d = np.einsum("mbk,nbk->mnb", q.reshape(M, nb, 32).astype(np.int64),
                      w.reshape(N, nb, 32).astype(np.int64)).astype(np.float64)
        mag = np.abs(d * sw.astype(np.float64)[None] * s.astype(np.float64)[:, None]).sum(2)
        bound = (nb + 3) * 2.0 ** -24 * mag
        assert np.all(np.abs(acc - ref) <= bound)


def pin_linear_invariants(orc):
    """Zero x rows give zero y rows; zero W gives zero y; scaling s_w or x by
    2^j scales the fp32 sums by 2^j exactly; permuting W rows permutes y columns."""
    r = _rng(9)
    M, N, K = 3, 6, 128
    x = (r.integers(-4000, 4000, (M, K)) / 256.0).astype(np.float16)
    x[1] = 0
    w = r.integers(-8, 8, (N, K)).astype(np.int8)
    sw = r.uniform(0.002, 0.01, (N, K // 32)).astype(np.float16)
    y, acc = orc.linear(x, w, sw, return_acc=True)
    assert np.all(y[1] == 0)
    assert np.all(orc.linear(x, np.zeros_like(w), sw) == 0)
    _, acc4 = orc.linear(x, w, (sw.astype(np.float32) * 4).astype(np.float16), return_acc=True)
    assert np.array_equal(acc4, acc * np.float32(4))
    _, accx = orc.linear((x.astype(np.float32) * 0.25).astype(np.float16), w, sw, return_acc=True)
    assert np.array_equal(accx, acc * np.float32(0.25))
    perm = r.permutation(N)
    assert np.array_equal(orc.linear(x, w[perm], sw[perm]), y[:, perm])


# ------------------------------------------------------------ packed layout

def pin_unpack_layout(orc):
    """The packed layout's written definition: byte j of a row holds k = 2j in
    its low nibble and k = 2j+1 in its high nibble, each as w + 8."""
    N, K = 2, 32
    packed = np.zeros((N, K // 2), np.uint8)
    packed[0, 0] = 0x0F   # k0 = 15-8 = 7, k1 = 0-8 = -8
    packed[0, 1] = 0x80   # k2 = -8, k3 = 0
    packed[0, 15] = 0x98  # k30 = 0, k31 = 1
    packed[1, :] = 0x88   # all zero
    w = orc.unpack_weights(packed, N, K)
    assert list(w[0, :4]) == [7, -8, -8, 0]
    assert list(w[0, 30:]) == [0, 1]
    assert np.all(w[0, 4:30] == -8)
    assert np.all(w[1] == 0)


def _gated_closed_form_case(act):
    """x of 127*(m+1) everywhere (s_x = m+1 exactly, every code 127); gate row
    n all codes cg[n] with block scales 2^-(10+n), up row n all codes cu[n]
    with 2^-(8+n).  Every block dot is 32*127*code and every product is exact
    in fp32, so g and u are known in closed form; act(g)*u follows from the
    activation's definition with Python's math library."""
    import math
    M, N, K = 2, 3, 64
    nb = K // 32
    cg, cu = [-3, 2, 5], [7, -8, 1]
    x = np.array([[127.0 * (m + 1)] * K for m in range(M)], np.float16)
    w = np.zeros((2 * N, K), np.int8)
    sw = np.zeros((2 * N, nb), np.float16)
    for n in range(N):
        w[n, :] = cg[n]
        w[N + n, :] = cu[n]
        sw[n, :] = 2.0 ** -(10 + n)
        sw[N + n, :] = 2.0 ** -(8 + n)
    y = np.zeros((M, N), np.float16)
    for m in range(M):
        for n in range(N):
            g = nb * 32 * 127 * cg[n] * 2.0 ** -(10 + n) * (m + 1)
            u = nb * 32 * 127 * cu[n] * 2.0 ** -(8 + n) * (m + 1)
            if act == 1:
                a = g / (1.0 + math.exp(-g))
            else:
                a = 0.5 * g * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))
            y[m, n] = np.float16(np.float32(a * u))
    return x, w, sw, y


def pin_gated_silu_closed_form(orc):
    x, w, sw, y = _gated_closed_form_case(1)
    assert np.array_equal(orc.linear_gated(x, w, sw, 1).view(np.uint16), y.view(np.uint16))


def pin_gated_gelu_closed_form(orc):
    x, w, sw, y = _gated_closed_form_case(2)
    assert np.array_equal(orc.linear_gated(x, w, sw, 2).view(np.uint16), y.view(np.uint16))


def pin_gated_special_values(orc):
    """act(0) = 0 for both activations: zero gate rows give exact zeros; a
    zero up row gives zeros; SiLU of a large gate is the gate itself, so with
    unit up values y = g to fp16 precision."""
    rng = _rng(31)
    M, N, K = 3, 4, 96
    x = rng.standard_normal((M, K)).astype(np.float16)
    w = rng.integers(-8, 8, (2 * N, K)).astype(np.int8)
    sw = rng.uniform(0.001, 0.01, (2 * N, K // 32)).astype(np.float16)
    for act in (1, 2):
        wz = w.copy()
        wz[:N] = 0
        assert not np.any(orc.linear_gated(x, wz, sw, act).astype(np.float32))
        wz = w.copy()
        wz[N:] = 0
        assert not np.any(orc.linear_gated(x, wz, sw, act).astype(np.float32))
    # x = 127 (s_x = 1, codes 127); gate codes 7 with scale 1/2 over 3 blocks:
    # g = 3*32*127*7/2 = 42672, and silu(g) = g in double precision; up codes 1
    # with scale 2^-14 over 3 blocks: u = 3*4064*2^-14 = 0.744140625
    xs = np.full((1, K), 127.0, np.float16)
    wg = np.zeros((2, K), np.int8)
    wg[0, :] = 7
    wg[1, :] = 1
    sg = np.array([[0.5] * 3, [2.0 ** -14] * 3], np.float16)
    got = orc.linear_gated(xs, wg, sg, 1)
    assert got[0, 0] == np.float16(np.float32(42672.0 * 0.744140625))


def pin_rmsnorm_closed_form(orc):
    """K=32, eps=0, unit gamma, no residual: a row of 16 threes and 16 fours has
    mean square 12.5, so y = 3/sqrt(12.5) and 4/sqrt(12.5); a constant row c
    gives y = sign(c) exactly, hence codes +-127 and scale 1/127."""
    import math
    K = 32
    x = np.array([[3.0] * 16 + [4.0] * 16, [-5.0] * 32, [0.25] * 32], np.float16)
    gamma = np.ones(K, np.float16)
    ro, y, q, sx = orc.rmsnorm_quant(x, None, gamma, 0.0)
    want0 = [np.float16(np.float32(3.0 / math.sqrt(12.5)))] * 16 + [np.float16(np.float32(4.0 / math.sqrt(12.5)))] * 16
    assert np.array_equal(y[0].view(np.uint16), np.array(want0, np.float16).view(np.uint16))
    assert np.all(y[1] == -1.0) and np.all(y[2] == 1.0)
    assert np.all(q[1] == -127) and np.all(q[2] == 127)
    assert sx[1, 0] == np.float32(1.0) / np.float32(127.0) and sx[2, 0] == sx[1, 0]
    assert np.array_equal(ro.view(np.uint16), x.view(np.uint16))


def pin_rmsnorm_residual_and_eps(orc):
    """The residual stream is the fp16 sum x + res (IEEE addition in fp32, one
    rounding); eps enters under the root: a zero row gives y = 0 with eps > 0,
    and for a constant row c, y = c / sqrt(c^2 + eps)."""
    import math
    rng = _rng(41)
    M, K = 3, 64
    x = rng.standard_normal((M, K)).astype(np.float16)
    res = rng.standard_normal((M, K)).astype(np.float16)
    gamma = np.ones(K, np.float16)
    ro, _, _, _ = orc.rmsnorm_quant(x, res, gamma, 1e-6)
    assert np.array_equal(ro.view(np.uint16), (x.astype(np.float32) + res.astype(np.float32)).astype(np.float16).view(np.uint16))
    z = np.zeros((1, K), np.float16)
    _, y, q, sx = orc.rmsnorm_quant(z, None, gamma, 1e-5)
    assert not np.any(y.astype(np.float32)) and not np.any(q) and np.all(sx == 1.0)
    c = np.full((1, K), 0.5, np.float16)
    _, y, _, _ = orc.rmsnorm_quant(c, None, gamma, 0.25)
    assert y[0, 0] == np.float16(np.float32(0.5 / math.sqrt(0.25 + 0.25)))


def pin_rmsnorm_invariants(orc):
    """With eps = 0 the norm is invariant to scaling the row by 2^j (codes and
    scales identical); gamma * 2 doubles y exactly (same codes, scales * 2);
    the codes are those of the activation quantiser applied to y."""
    rng = _rng(43)
    M, K = 4, 96
    x = (rng.standard_normal((M, K)) * 3).astype(np.float16)
    gamma = rng.uniform(0.5, 1.5, K).astype(np.float16)
    _, y, q, sx = orc.rmsnorm_quant(x, None, gamma, 0.0)
    _, y2, q2, sx2 = orc.rmsnorm_quant((x.astype(np.float32) * 4).astype(np.float16), None, gamma, 0.0)
    assert np.array_equal(y.view(np.uint16), y2.view(np.uint16)) and np.array_equal(q, q2)
    _, y3, q3, sx3 = orc.rmsnorm_quant(x, None, (gamma.astype(np.float32) * 2).astype(np.float16), 0.0)
    assert np.array_equal(y3.astype(np.float32), y.astype(np.float32) * 2) and np.array_equal(q3, q)
    assert np.array_equal(sx3, sx * 2)
    qa, sa = orc.quantize_act(y)
    assert np.array_equal(qa, q) and np.array_equal(sa, sx)


def pin_attention_single_and_uniform(orc):
    """One cached token: softmax weight 1, so out = v_0 exactly.  All keys
    equal: uniform weights, so out = the mean of the value rows."""
    rng = _rng(51)
    B, Hq, Hkv, D, Lmax = 2, 4, 2, 64, 9
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    v = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    out = orc.decode_attention(q, k, v, np.array([1, 1], np.int32))
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(out[b, h].view(np.uint16), v[b, h // 2, 0].view(np.uint16))
    ke = np.repeat(k[:, :, :1, :], Lmax, axis=2)
    out = orc.decode_attention(q, ke, v, np.array([Lmax, 5], np.int32))
    for b, L in ((0, Lmax), (1, 5)):
        for h in range(Hq):
            mean = v[b, h // 2, :L].astype(np.float64).mean(axis=0)
            assert np.array_equal(out[b, h].view(np.uint16), mean.astype(np.float32).astype(np.float16).view(np.uint16))


def pin_attention_group_mapping_and_lengths(orc):
    """Query head h reads KV head h / (Hq/Hkv): with constant value rows 1,2,3
    per KV head the outputs are those constants; rows past lens[b] never
    matter (filled with huge values here)."""
    B, Hq, Hkv, D, Lmax = 1, 6, 3, 32, 7
    rng = _rng(53)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    k = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    v = np.zeros((B, Hkv, Lmax, D), np.float16)
    for g in range(Hkv):
        v[0, g] = g + 1
    L = 4
    k[0, :, L:] = 30000.0
    v[0, :, L:] = -30000.0
    out = orc.decode_attention(q, k, v, np.array([L], np.int32))
    for h in range(Hq):
        assert np.all(out[0, h] == (h // 2) + 1)


def pin_attention_two_keys_closed_form(orc):
    """Two cached tokens, q = e_0 * a, k_0 = e_0, k_1 = 0: scores a/sqrt(D) and
    0, so with v_0 = 1 and v_1 = 0 the output is the logistic 1/(1+e^-s);
    and a dominant key (score gap > 40) returns its value row exactly, even
    where exp of the raw score would overflow (the max is subtracted first)."""
    import math
    D = 64
    for a in (1.0, 4.0, -6.0, 20.0):
        q = np.zeros((1, 1, D), np.float16)
        q[0, 0, 0] = a
        k = np.zeros((1, 1, 2, D), np.float16)
        k[0, 0, 0, 0] = 1.0
        v = np.zeros((1, 1, 2, D), np.float16)
        v[0, 0, 0] = 1.0
        out = orc.decode_attention(q, k, v, np.array([2], np.int32)).astype(np.float64)
        s = a / math.sqrt(D)
        want = 1.0 / (1.0 + math.exp(-s))
        assert np.all(np.abs(out[0, 0] - want) <= 2.0 ** -11 * max(want, 2.0 ** -14))
    rng = _rng(57)
    q = np.zeros((1, 1, D), np.float16)
    q[0, 0, :] = 1.0
    k = (rng.standard_normal((1, 1, 5, D)) * 0.1).astype(np.float16)
    k[0, 0, 3, :] = 120.0     # score 120*64/8 = 960: far above the rest (|s| < 8), and past exp's fp64 range
    v = rng.standard_normal((1, 1, 5, D)).astype(np.float16)
    out = orc.decode_attention(q, k, v, np.array([5], np.int32))
    assert np.array_equal(out[0, 0].view(np.uint16), v[0, 0, 3].view(np.uint16))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
