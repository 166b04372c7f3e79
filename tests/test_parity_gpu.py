"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer work (packing, activation codes and scales, per-block dots) must be
bit-exact; fp16 outputs must meet the tolerance of parity.py.  Inputs come
from the seeded generators of int4_weight_quantized_gb300.workloads.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from int4_weight_quantized_gb300 import workloads as wl

from .oracle_pins import load_quant_blocks
from .parity import assert_fp16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    from int4_weight_quantized_gb300.build import build
    build()
    import int4_weight_quantized_gb300 as w4
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return w4


def _dev(t):
    return t.cuda()


def _setup(w4, x, codes, scales):
    xd, cd, sd = _dev(x), _dev(codes), _dev(scales)
    packed = w4.pack(cd)
    return xd, packed, sd


def _np(t):
    return t.detach().cpu().numpy()


# ---------------------------------------------------------------- packing

@pytest.mark.parametrize("N,K", [(1, 32), (7, 96), (512, 256), (300, 2048), (8192, 2048)])
def test_pack_layout(w4, N, K):
    codes, _ = wl.make_weights(N, K, seed=11 + N, s_lo=0.01, s_hi=0.02)
    packed = w4.pack(_dev(codes))
    assert packed.numel() == w4.packed_bytes(N, K)
    back = oracle.unpack_weights(_np(packed), N, K)
    assert np.array_equal(back, codes.numpy())


def test_pack_rejects_out_of_range_codes(w4):
    codes = torch.zeros((4, 64), dtype=torch.int8)
    codes[2, 17] = 9
    with pytest.raises(w4.W4A8Error) as e:
        w4.pack(_dev(codes))
    assert e.value.status == 3
    codes[2, 17] = -9
    with pytest.raises(w4.W4A8Error):
        w4.pack(_dev(codes))


# --------------------------------------------------- activation quantiser

def test_quantizer_golden_blocks(w4):
    blocks = load_quant_blocks()
    x = np.stack([b[1] for b in blocks])                     # one block per token
    q, s = w4.debug_quantize_act(_dev(torch.from_numpy(x)))
    torch.cuda.synchronize()
    for i, (name, _, qb, sb) in enumerate(blocks):
        assert np.array_equal(_np(q)[i], qb), name
        assert int(_np(s)[i].view(np.uint32)[0]) == sb, name


@pytest.mark.parametrize("M,K,scale,outliers", [(1, 32, 1.0, 0.0), (3, 256, 1.0, 0.01), (8, 2048, 0.01, 0.01),
                                                (64, 4096, 300.0, 0.0), (512, 2048, 1.0, 0.01)])
def test_quantizer_bit_exact(w4, M, K, scale, outliers):
    x = wl.make_x(M, K, seed=M * 7 + K, outlier_frac=outliers)
    x = (x.float() * scale).half()
    if M > 2:
        x[1] = 0                                            # an all-zero token
        x[2, 5:37] = torch.tensor(np.arange(1, 33), dtype=torch.int16).view(torch.float16)  # subnormals
    q, s = w4.debug_quantize_act(_dev(x))
    qo, so = oracle.quantize_act(x.numpy())
    assert np.array_equal(_np(q), qo)
    assert np.array_equal(_np(s).view(np.uint32), so.view(np.uint32))


# ---------------------------------------------------------- block dots

# decode kernels by shape: codes in registers (K/32 in 1, 2, 4 or 8 slices of
# 32 blocks and tokens x slices <= 8), one token with rows of 5-16 slices in 2
# or 4 K groups of 4 slices (ragged last groups: 193 and 448 blocks), codes
# read from shared memory (two tokens with long rows; long rows make small
# chunks, and the longest need one CTA per SM), and the cluster split-K kernel
# (3 to 8 tokens with long rows)
DOT_SHAPES = [(1, 1, 32), (1, 37, 96), (2, 100, 1024), (3, 64, 1056), (8, 129, 2048), (5, 257, 4096),
              (1, 300, 3072), (2, 77, 14336), (1, 40, 14336), (1, 700, 14336), (1, 1500, 4096),
              (1, 130, 6176), (1, 2048, 8192)]


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("M,N,K", DOT_SHAPES + [(9, 130, 512), (64, 96, 256), (130, 70, 320)])
def test_block_dots_bit_exact(w4, path, M, N, K):
    x = wl.make_x(M, K, seed=100 + M, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=200 + N, s_lo=0.002, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    dots, y = w4.debug_block_dots(xd, packed, sd, path=path)
    q, _ = oracle.quantize_act(x.numpy())
    ref = oracle.block_dots(q, codes.numpy())
    assert np.array_equal(_np(dots), ref)
    assert_fp16_close(_np(y), oracle.linear(x.numpy(), codes.numpy(), scales.numpy()), f"y {M}x{N}x{K}")


# shapes whose prefill tiles run as 1, 2, 4 and 8 CTAs along K (cluster
# split-K with a fixed-order reduction in distributed shared memory): with
# K % 256 != 0 they take the 128 x 128-tile kernel, otherwise the kernel with
# the weights as the 128-row operand and 128-token tiles
SPLIT_SHAPES = [((200, 10240, 288), 1), ((65, 8192, 544), 2), ((33, 2560, 1056), 4), ((16, 128, 1056), 8),
                ((130, 70, 320), 4), ((65, 8192, 512), 1), ((129, 300, 1024), 2), ((200, 1024, 2048), 4),
                ((100, 256, 4096), 8), ((512, 256, 14336), 4)]


@pytest.mark.parametrize("shape,splits", SPLIT_SHAPES)
def test_prefill_split_k_bit_exact(w4, shape, splits):
    M, N, K = shape
    assert w4.prefill_splits(M, N, K) == splits
    x = wl.make_x(M, K, seed=500 + M, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=600 + N, s_lo=-0.01, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    dots, y = w4.debug_block_dots(xd, packed, sd, path=2)
    q, _ = oracle.quantize_act(x.numpy())
    assert np.array_equal(_np(dots), oracle.block_dots(q, codes.numpy()))
    ref = oracle.linear(x.numpy(), codes.numpy(), scales.numpy())
    assert_fp16_close(_np(y), ref, f"debug {M}x{N}x{K}")
    assert_fp16_close(_np(w4.linear(xd, packed, sd, path=2)), ref, f"linear {M}x{N}x{K}")


# the short-sequence tensor-core path (weights as the 128-row operand, tokens
# padded to 16, 32 or 64): token counts on both sides of each padding step,
# ragged N (partial last 128-row tile), and K split over 1, 2, 4 and 8 CTAs
MID_SHAPES = [(1, 130, 256), (3, 300, 1024), (8, 1000, 2048), (9, 129, 512), (16, 64, 4096), (17, 257, 768),
              (33, 200, 2048), (64, 520, 1024), (40, 4096, 14336), (5, 128, 8192), (64, 77, 256)]


@pytest.mark.parametrize("M,N,K", MID_SHAPES)
def test_mid_path_bit_exact(w4, M, N, K):
    x = wl.make_x(M, K, seed=1500 + M, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=1600 + N, s_lo=-0.01, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    dots, y = w4.debug_block_dots(xd, packed, sd, path=w4.PATH_MID)
    q, _ = oracle.quantize_act(x.numpy())
    assert np.array_equal(_np(dots), oracle.block_dots(q, codes.numpy()))
    ref = oracle.linear(x.numpy(), codes.numpy(), scales.numpy())
    assert_fp16_close(_np(y), ref, f"mid debug {M}x{N}x{K}")
    y2 = w4.linear(xd, packed, sd, path=w4.PATH_MID)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert w4.get_device_status() == 0


def test_mid_path_split_counts(w4):
    """The shapes above reach every split count of the mid path."""
    seen = {w4.mid_splits(M, N, K) for (M, N, K) in MID_SHAPES}
    assert {1, 2, 4, 8} <= seen, seen


# --------------------------------------------------------- gated pair

# decode shapes take the fused kernel (codes in registers, or codes from
# shared memory with one or two tokens); the others take the linear over 2N
# rows and the element-wise pass
GATED_SHAPES = [(1, 64, 64, True), (1, 300, 2048, True), (2, 96, 3072, True), (3, 130, 1024, True),
                (8, 200, 256, True), (1, 1000, 4096, True), (1, 96, 8192, True), (1, 64, 14336, True),
                (5, 70, 4096, False),
                (9, 70, 512, False),
                (64, 128, 256, False), (200, 96, 320, False)]


@pytest.mark.parametrize("act", [1, 2])
@pytest.mark.parametrize("M,N,K,fused", GATED_SHAPES)
def test_linear_gated(w4, M, N, K, fused, act):
    assert (w4.gated_workspace_bytes(M, N, K) == 0) == fused
    x = wl.make_x(M, K, seed=700 + M + K, outlier_frac=0.01)
    codes, scales = wl.make_weights(2 * N, K, seed=800 + N + K, s_lo=0.002, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    y = w4.linear_gated(xd, packed, sd, act=act)
    ref = oracle.linear_gated(x.numpy(), codes.numpy(), scales.numpy(), act)
    assert_fp16_close(_np(y), ref, f"gated act={act} {M}x{N}x{K}")


def test_linear_gated_rejects_bad_act_and_missing_workspace(w4):
    M, N, K = 16, 64, 256
    x = wl.make_x(M, K, seed=3)
    codes, scales = wl.make_weights(2 * N, K, seed=4, s_lo=0.002, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    out = torch.empty((M, N), dtype=torch.float16, device="cuda")
    P = ctypes.c_void_p
    st = w4.lib().w4a8_linear_gated(P(xd.data_ptr()), P(packed.data_ptr()), P(sd.data_ptr()), M, N, K,
                                    P(out.data_ptr()), 3, P(0), 0, P(torch.cuda.current_stream().cuda_stream))
    assert st == 1   # W4A8_ERR_INVALID_VALUE
    st = w4.lib().w4a8_linear_gated(P(xd.data_ptr()), P(packed.data_ptr()), P(sd.data_ptr()), M, N, K,
                                    P(out.data_ptr()), 1, P(0), 0, P(torch.cuda.current_stream().cuda_stream))
    assert st == 7   # W4A8_ERR_WORKSPACE


# ------------------------------------------ producer-side quantisation

def _fp16_ulp(v):
    a = np.abs(v.astype(np.float32))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


NORM_SHAPES = [(1, 32), (3, 2048), (8, 4096), (5, 14336), (130, 320)]


@pytest.mark.parametrize("with_res", [False, True])
@pytest.mark.parametrize("M,K", NORM_SHAPES)
def test_rmsnorm_quant(w4, M, K, with_res):
    """Residual stream bit-exact; y (fp32 arithmetic here, fp64 in the oracle)
    within one fp16 ulp; codes and scales bit-exact against the oracle's
    quantiser applied to the kernel's own y (the decision is taken on the
    same fp16 values on both sides)."""
    g = np.random.default_rng(900 + M + K)
    x = (g.standard_normal((M, K)) * 2).astype(np.float16)
    res = g.standard_normal((M, K)).astype(np.float16) if with_res else None
    gamma = g.uniform(0.5, 1.5, K).astype(np.float16)
    eps = 1e-6
    xd = torch.from_numpy(x).cuda()
    rd = torch.from_numpy(res).cuda() if with_res else None
    gd = torch.from_numpy(gamma).cuda()
    ro = torch.empty_like(xd)
    yo = torch.empty_like(xd)
    codes, sx = w4.rmsnorm_quant(xd, gd, eps, residual=rd, residual_out=ro, y_out=yo)
    r_ref, y_ref, q_ref, s_ref = oracle.rmsnorm_quant(x, res, gamma, eps)
    assert np.array_equal(_np(ro).view(np.uint16), r_ref.view(np.uint16))
    yg = _np(yo)
    assert np.all(np.abs(yg.astype(np.float32) - y_ref.astype(np.float32)) <= _fp16_ulp(y_ref))
    assert np.mean(yg == y_ref) > 0.95
    qg, sg = oracle.quantize_act(yg)
    assert np.array_equal(_np(codes), qg) and np.array_equal(_np(sx), sg)
    # end to end against the oracle's own codes: every 32-block whose y equals
    # the oracle's y has identical codes and scale; the few blocks holding a
    # one-ulp difference of y stay within one code step
    same_blk = np.all((yg == y_ref).reshape(M, K // 32, 32), axis=2)
    cg = _np(codes).reshape(M, K // 32, 32)
    cr = q_ref.reshape(M, K // 32, 32)
    assert np.array_equal(cg[same_blk], cr[same_blk])
    assert np.array_equal(_np(sx).view(np.uint32)[same_blk], s_ref.view(np.uint32)[same_blk])
    assert np.mean(same_blk) > 0.5
    assert np.all(np.abs(cg[~same_blk].astype(np.int32) - cr[~same_blk].astype(np.int32)) <= 1)


# (M, N, K, same kernel as the fp16 linear): codes input always decodes with
# the streaming kernel, while the fp16 linear takes the cluster split-K
# kernel for 3-8 tokens with long rows, whose summation order differs
Q8_SHAPES = [(1, 512, 2048, True), (2, 300, 3072, True), (1, 200, 10240, True), (5, 257, 4096, False),
             (8, 129, 2048, False),
             (9, 130, 512, True), (64, 96, 256, True), (200, 70, 320, True)]


@pytest.mark.parametrize("M,N,K,same", Q8_SHAPES)
def test_linear_q8_matches_linear(w4, M, N, K, same):
    """The linear on producer codes matches the oracle within the fp16
    tolerance, and gives exactly what the linear on the fp16 activations
    gives when both run the same kernel after the quantisation step."""
    x = wl.make_x(M, K, seed=1000 + M, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=1100 + N, s_lo=0.002, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    q, s = oracle.quantize_act(x.numpy())
    y8 = w4.linear_q8(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), packed, sd)
    y = w4.linear(xd, packed, sd)
    torch.cuda.synchronize()
    if same:
        assert torch.equal(y8, y)
    assert_fp16_close(_np(y8), oracle.linear(x.numpy(), codes.numpy(), scales.numpy()), f"q8 {M}x{N}x{K}")


def test_rmsnorm_then_linear_q8(w4):
    M, N, K = 1, 2048, 2048
    g = np.random.default_rng(77)
    x = g.standard_normal((M, K)).astype(np.float16)
    gamma = g.uniform(0.5, 1.5, K).astype(np.float16)
    codes_w, scales_w = wl.make_weights(N, K, seed=78, s_lo=0.002, s_hi=0.01)
    packed = w4.pack(codes_w.cuda())
    yo = torch.empty((M, K), dtype=torch.float16, device="cuda")
    q, s = w4.rmsnorm_quant(torch.from_numpy(x).cuda(), torch.from_numpy(gamma).cuda(), 1e-6, y_out=yo)
    out = w4.linear_q8(q, s, packed, scales_w.cuda())
    assert_fp16_close(_np(out), oracle.linear(_np(yo), codes_w.numpy(), scales_w.numpy()), "norm+q8")


# ---------------------------------------------------------- decode attention

# (B, Hq, Hkv, D, Lmax, lens): the decoder layer's 8 query heads over one KV
# head of 256 (10 chunks of 64 on the tensor cores, merged in one cluster),
# ragged lengths incl. 1 and a chunk edge (clusters with empty chunks), 16
# chunks (the largest cluster), one chunk (direct write), 16 heads per group
# with D=64 (128-token chunks on CUDA cores, combine kernel), 3 KV heads,
# group sizes 3 and 5 (not powers of two)
ATTN_CASES = [(1, 8, 1, 256, 640, [640]), (3, 8, 1, 256, 200, [1, 129, 200]), (2, 4, 2, 128, 128, [128, 64]),
              (4, 16, 1, 64, 300, [300, 1, 257, 128]), (2, 6, 3, 128, 1000, [999, 500]),
              (2, 6, 2, 256, 130, [130, 3]), (1, 5, 1, 64, 64, [64]),
              # tensor-core kernel: more than 16 chunks (workspace and combine
              # kernel instead of the cluster merge), and one chunk
              (2, 8, 2, 128, 1500, [1500, 700]), (2, 8, 1, 256, 64, [64, 10])]


@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax,lens", ATTN_CASES)
def test_decode_attention(w4, B, Hq, Hkv, D, Lmax, lens):
    g = np.random.default_rng(1300 + B * Lmax + D)
    q = g.standard_normal((B, Hq, D)).astype(np.float16)
    k = g.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    v = g.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    ln = np.array(lens, np.int32)
    out = w4.decode_attention(torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                              torch.from_numpy(ln).cuda())
    ref = oracle.decode_attention(q, k, v, ln)
    assert_fp16_close(_np(out).reshape(B * Hq, D), ref.reshape(B * Hq, D), f"attention {B},{Hq},{Hkv},{D},{Lmax}")


def test_decode_attention_edge_lengths(w4):
    """Lengths are clamped to [0, Lmax]: 0 gives zeros, more than Lmax reads Lmax rows."""
    B, Hq, Hkv, D, Lmax = 3, 4, 1, 64, 300
    g = np.random.default_rng(1400)
    q = g.standard_normal((B, Hq, D)).astype(np.float16)
    k = g.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    v = g.standard_normal((B, Hkv, Lmax, D)).astype(np.float16)
    ln = np.array([0, 100000, 7], np.int32)
    out = _np(w4.decode_attention(torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                                  torch.from_numpy(ln).cuda()))
    assert not np.any(out[0].astype(np.float32))
    ref = oracle.decode_attention(q[1:], k[1:], v[1:], np.array([Lmax, 7], np.int32))
    assert_fp16_close(out[1:].reshape(-1, D), ref.reshape(-1, D), "clamped lengths")


# ---------------------------------------------------------------- linear

EDGE_SHAPES = ([(M, 67, 160) for M in range(1, 10)] + [(15, 33, 64), (16, 256, 512), (17, 50, 96),
               (63, 40, 128), (64, 128, 256), (65, 129, 288), (129, 200, 64), (1, 1, 32), (3, 1, 32),
               (200, 1, 64), (1, 5000, 32), (2, 3, 8192)])


@pytest.mark.parametrize("M,N,K", EDGE_SHAPES)
def test_linear_edge_shapes(w4, M, N, K):
    x = wl.make_x(M, K, seed=300 + M + K, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=400 + N + K, s_lo=-0.01, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    y = w4.linear(xd, packed, sd)
    assert_fp16_close(_np(y), oracle.linear(x.numpy(), codes.numpy(), scales.numpy()), f"{M}x{N}x{K}")


@pytest.mark.parametrize("path", [1, 2, 3])
def test_linear_zero_inputs(w4, path):
    M, N, K = 12, 96, 256
    x = wl.make_x(M, K, seed=5)
    x[3] = 0
    x[7, :64] = 0
    codes, scales = wl.make_weights(N, K, seed=6, s_lo=0.002, s_hi=0.01)
    codes[10] = 0
    xd, packed, sd = _setup(w4, x, codes, scales)
    y = _np(w4.linear(xd, packed, sd, path=path))
    assert np.all(y[3] == 0) and np.all(y[:, 10] == 0)
    assert_fp16_close(y, oracle.linear(x.numpy(), codes.numpy(), scales.numpy()))
    y0 = _np(w4.linear(torch.zeros_like(xd), packed, sd, path=path))
    assert np.all(y0 == 0)


@pytest.mark.parametrize("M", [1, 4, 8, 16, 64])
def test_paths_agree_on_integer_work(w4, M):
    """Both kernels compute the same codes and dots; their fp16 outputs differ
    only by fp32 summation order."""
    N, K = 300, 1024
    x = wl.make_x(M, K, seed=M, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=M + 1, s_lo=0.002, s_hi=0.01)
    xd, packed, sd = _setup(w4, x, codes, scales)
    d1, y1 = w4.debug_block_dots(xd, packed, sd, path=1)
    d2, y2 = w4.debug_block_dots(xd, packed, sd, path=2)
    d3, y3 = w4.debug_block_dots(xd, packed, sd, path=3)
    assert torch.equal(d1, d2) and torch.equal(d1, d3)
    assert_fp16_close(_np(y1), _np(y2))
    assert_fp16_close(_np(y3), _np(y2))


def test_c_entry_point_matches_ex(w4):
    for (M, N, K) in ((1, 512, 256), (300, 256, 512)):
        x = wl.make_x(M, K, seed=9)
        codes, scales = wl.make_weights(N, K, seed=10, s_lo=0.002, s_hi=0.01)
        xd, packed, sd = _setup(w4, x, codes, scales)
        a = w4.linear(xd, packed, sd)
        b = torch.empty_like(a)
        w4.linear_c(xd, packed, sd, b)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


# ---------------------------------------------- the five workloads at full size

def _sampled_check(w4, lin, seed, weight_set=0, n_cols=96, n_rows=48):
    """Full-size call on the GPU; the oracle recomputes a sample of output
    columns (whole W rows, so each sampled output is exact) for a sample of
    tokens, including the first and last of each."""
    x, codes, scales = wl.make_linear_inputs(lin, seed, weight_set)
    xd, packed, sd = _setup(w4, x, codes, scales)
    y = _np(w4.linear(xd, packed, sd))
    g = np.random.default_rng(seed + weight_set)
    cols = np.unique(np.concatenate([[0, lin.N - 1], g.choice(lin.N, min(n_cols, lin.N), replace=False)]))
    rows = np.unique(np.concatenate([[0, lin.M - 1], g.choice(lin.M, min(n_rows, lin.M), replace=False)]))
    ref = oracle.linear(x.numpy()[rows], codes.numpy()[cols], scales.numpy()[cols])
    assert_fp16_close(y[np.ix_(rows, cols)], ref, lin.name)
    return y


def _sampled_check_gated(w4, lin, seed, n_cols=96):
    """Full-size gated pair on the GPU; the oracle recomputes a sample of
    output columns from their gate and up rows."""
    x, codes, scales = wl.make_linear_inputs(lin, seed)
    xd, packed, sd = _setup(w4, x, codes, scales)
    y = _np(w4.linear_gated(xd, packed, sd, act=lin.gated))
    g = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([[0, lin.N - 1], g.choice(lin.N, min(n_cols, lin.N), replace=False)]))
    rows = np.concatenate([cols, lin.N + cols])
    ref = oracle.linear_gated(x.numpy(), codes.numpy()[rows], scales.numpy()[rows], lin.gated)
    assert_fp16_close(y[:, cols], ref, lin.name)


@pytest.mark.parametrize("wi", range(len(wl.workloads())))
def test_workloads_full_size(w4, wi):
    W = wl.workloads()[wi]
    for li, lin in enumerate(W.linears):
        if lin.gated:
            _sampled_check_gated(w4, lin, W.seed + li * 100)
        else:
            _sampled_check(w4, lin, W.seed + li * 100)


def test_tiny_workload_exhaustive(w4):
    W = wl.workloads()[0]
    lin = W.linears[0]
    x, codes, scales = wl.make_linear_inputs(lin, W.seed)
    xd, packed, sd = _setup(w4, x, codes, scales)
    dots, y = w4.debug_block_dots(xd, packed, sd)
    q, _ = oracle.quantize_act(x.numpy())
    assert np.array_equal(_np(dots), oracle.block_dots(q, codes.numpy()))
    assert_fp16_close(_np(y), oracle.linear(x.numpy(), codes.numpy(), scales.numpy()))


# --------------------------------------------------------- failure reporting

def test_bounded_wait_reports_timeout(w4):
    assert w4.get_device_status() == 0
    w4.set_wait_budget(200000)
    try:
        w4.debug_wait_timeout()
        assert w4.get_device_status() == 5
        assert w4.get_device_status() == 0       # cleared by the read
    finally:
        w4.set_wait_budget(0)
    # the context is still usable
    x = wl.make_x(1, 256, seed=1)
    codes, scales = wl.make_weights(64, 256, seed=2, s_lo=0.01, s_hi=0.02)
    xd, packed, sd = _setup(w4, x, codes, scales)
    assert_fp16_close(_np(w4.linear(xd, packed, sd)), oracle.linear(x.numpy(), codes.numpy(), scales.numpy()))


def test_workspace_too_small_is_rejected(w4):
    M, N, K = 64, 128, 256
    need = w4.workspace_bytes(M, N, K, 2)
    if need == 0:
        pytest.skip("prefill path needs no workspace")
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    codes, scales = wl.make_weights(N, K, seed=3, s_lo=0.01, s_hi=0.02)
    packed = w4.pack(_dev(codes))
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4A8Error) as e:
        w4.linear(x, packed, _dev(scales), path=2, workspace=ws)
    assert e.value.status == 7
