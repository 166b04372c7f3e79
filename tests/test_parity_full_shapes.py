"""Integer parity at the workloads' full shapes, through the dispatcher's path.

The small-shape tests in test_parity_gpu.py compare every block dot, but
they never reach the pipelines that the benchmark's shapes take: the prefill
GEMM with one split and 32 to 224 stages (its operand and scale rings wrap
many times), the decode kernels' plans for 2048 to 14336-wide rows, and the
mid-M shapes.  Here every linear of every workload is run at its real size
on the kernel that the automatic (stage-aware) dispatch picks, and

  - the activation codes and block scales of the whole input are compared
    bit for bit with the oracle's quantiser;
  - the int32 block dots d[m, n, b] are compared bit for bit on a sample of
    at least 64 token rows (all of them when M <= 64; the first and last
    always) times at least 256 weight rows (one in every 128-row tile, the
    first and last, the rest drawn at random), over every block b.  Each dot
    depends only on its own token row and weight row, so a sampled dot is
    exactly the dot of the full problem;
  - the fp16 outputs of the debug instantiation equal the production
    kernel's outputs exactly (the debug kernel adds stores, nothing else),
    which ties the production path to the dots checked here, and meet the
    fp16 tolerance against the oracle on the sample.

The block structure being checked is the pages' 4-bit weights in blocks of
32 ("Що змінює ML Drift для on-device AI-інференсу на вашому телефоні?",
tech.dede.sh, section "Stage-aware оптимізація для великих мовних моделей").
"""
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


def _full_shape_cases():
    """(id, linear, seed) for every plain linear of every workload except the
    tiny one (compared exhaustively elsewhere); shapes repeated within a
    workload are taken once."""
    cases = []
    for W in wl.workloads()[1:]:
        seen = set()
        for li, lin in enumerate(W.linears):
            if lin.gated:
                continue                       # gated pairs have no debug dots entry point
            key = (lin.M, lin.N, lin.K)
            if key in seen:
                continue
            seen.add(key)
            cases.append((f"{W.name}:{lin.name}:m{lin.M}_n{lin.N}_k{lin.K}", lin, W.seed + li * 100))
    return cases


CASES = _full_shape_cases()


def _sample_rows(M, g):
    if M <= 64:
        return np.arange(M)
    return np.unique(np.concatenate([[0, M - 1], g.choice(np.arange(1, M - 1), 62, replace=False)]))


def _sample_cols(N, g):
    if N <= 256:
        return np.arange(N)
    per_tile = [t * 128 + g.integers(0, min(128, N - t * 128)) for t in range((N + 127) // 128)]
    cols = set([0, N - 1] + [int(c) for c in per_tile])
    rest = g.permutation(N)
    i = 0
    while len(cols) < 256:
        cols.add(int(rest[i]))
        i += 1
    return np.array(sorted(cols))


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_full_shape_codes_and_dots_bit_exact(w4, case):
    _, lin, seed = case
    M, N, K = lin.M, lin.N, lin.K
    x, codes, scales = wl.make_linear_inputs(lin, seed)
    xd, sd = x.cuda(), scales.cuda()
    packed = w4.pack(codes.cuda())

    # activation codes and block scales of the whole input
    qg, sg = w4.debug_quantize_act(xd)
    q, s = oracle.quantize_act(x.numpy())
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(sg.cpu().numpy().view(np.uint32), s.view(np.uint32))

    # block dots of the dispatcher's kernel, on a sample
    dots, y_dbg = w4.debug_block_dots(xd, packed, sd, path=w4.PATH_AUTO)
    y = w4.linear(xd, packed, sd)
    torch.cuda.synchronize()
    g = np.random.default_rng(seed)
    rows, cols = _sample_rows(M, g), _sample_cols(N, g)
    ri, ci = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    got = dots.index_select(0, ri).index_select(1, ci).cpu().numpy()
    del dots
    ref = oracle.block_dots(q[rows], codes.numpy()[cols])
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (f"{bad.shape[0]} block dots differ, first at (row {rows[bad[0][0]]}, "
                           f"col {cols[bad[0][1]]}, block {bad[0][2]}): {got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}")

    # production outputs equal the debug instantiation's, and meet the tolerance
    assert torch.equal(y, y_dbg)
    yo = oracle.linear(x.numpy()[rows], codes.numpy()[cols], scales.numpy()[cols])
    assert_fp16_close(y.cpu().numpy()[np.ix_(rows, cols)], yo, case[0])
    assert w4.get_device_status() == 0


# The sweep's two shapes at further token counts on the tensor-core path for
# short sequences (the sweep itself runs M = 4, 8 and 64 through the dispatch
# above): both token tiles (16 and 32 tokens with the weights in tensor
# memory, 64 tokens in shared memory), with and without split-K.
SWEEP_MID = [(M, N, K) for M in (3, 9, 16, 33) for (N, K) in ((14336, 4096), (4096, 14336))]


@pytest.mark.parametrize("M,N,K", SWEEP_MID, ids=[f"m{M}_n{N}_k{K}" for (M, N, K) in SWEEP_MID])
def test_sweep_shapes_mid_path_dots_bit_exact(w4, M, N, K):
    x = wl.make_x(M, K, seed=2700 + M, outlier_frac=0.01)
    codes, scales = wl.make_weights(N, K, seed=2800 + K, s_lo=0.001, s_hi=0.008)
    xd, sd = x.cuda(), scales.cuda()
    packed = w4.pack(codes.cuda())
    dots, y_dbg = w4.debug_block_dots(xd, packed, sd, path=w4.PATH_MID)
    y = w4.linear(xd, packed, sd, path=w4.PATH_MID)
    torch.cuda.synchronize()
    g = np.random.default_rng(M * 7 + K)
    cols = _sample_cols(N, g)
    got = dots.index_select(1, torch.from_numpy(cols).cuda()).cpu().numpy()
    del dots
    q, _ = oracle.quantize_act(x.numpy())
    ref = oracle.block_dots(q, codes.numpy()[cols])
    assert np.array_equal(got, ref)
    assert torch.equal(y, y_dbg)
    yo = oracle.linear(x.numpy(), codes.numpy()[cols], scales.numpy()[cols])
    assert_fp16_close(y.cpu().numpy()[:, cols], yo, f"mid {M}x{N}x{K}")
    assert w4.get_device_status() == 0
