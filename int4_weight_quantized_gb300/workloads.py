"""Seeded synthetic inputs for the W4A8 linear (weights, block scales, activations).

This module only draws random numbers: it holds none of the operator's
arithmetic, and both the CUDA path and the CPU oracle take their inputs from
it.  Draws use a CPU ``torch.Generator`` so that the same seed gives the same
tensors on any host; only make_weights_on (for the 876 MB decoder-layer
benchmark, never compared with the oracle) draws on the GPU.

Shapes follow the pages' LLM workload: prefill length 512 and one-token decode
with 4-bit weights in blocks of 32 ("Що змінює ML Drift для on-device
AI-інференсу на вашому телефоні?", tech.dede.sh, section "Stage-aware
оптимізація для великих мовних моделей"), on the linears of a 2048-wide
decoder layer (8 query heads of 256, one KV head, FFN 8192).  No trained
weights are available, so uniform random int4 codes and uniform fp16 block
scales stand in for them, and activations are standard normal with 1% of
channels scaled by 20 to mimic the outlier channels of LLM activations.
"""
from dataclasses import dataclass, field

import torch

BLOCK = 32


def make_weights(N: int, K: int, seed: int, s_lo: float, s_hi: float):
    """Weight codes int8 [N][K] uniform in [-8, 7] and fp16 scales [N][K/32] U[s_lo, s_hi]."""
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    g = torch.Generator().manual_seed(seed)
    codes = torch.randint(-8, 8, (N, K), generator=g, dtype=torch.int8)
    scales = (torch.rand((N, K // BLOCK), generator=g, dtype=torch.float32)
              * (s_hi - s_lo) + s_lo).to(torch.float16)
    return codes, scales


def make_weights_on(device, N: int, K: int, seed: int, s_lo: float, s_hi: float):
    """As make_weights, drawn by a seeded generator on `device` (for workloads
    too large to draw on the host; the values differ from make_weights')."""
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    g = torch.Generator(device=device).manual_seed(seed)
    codes = torch.randint(-8, 8, (N, K), generator=g, dtype=torch.int8, device=device)
    scales = (torch.rand((N, K // BLOCK), generator=g, dtype=torch.float32, device=device)
              * (s_hi - s_lo) + s_lo).to(torch.float16)
    return codes, scales


def make_x(M: int, K: int, seed: int, outlier_frac: float = 0.0, outlier_gain: float = 20.0):
    """Activations fp16 [M][K]: N(0,1), with round(outlier_frac*K) channels (shared by all tokens) times outlier_gain."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, K), generator=g, dtype=torch.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        ch = torch.randperm(K, generator=g)[:n_out]
        x[:, ch] *= outlier_gain
    return x.to(torch.float16)


@dataclass
class Linear:
    """One linear layer's shape and input distribution."""
    M: int
    N: int
    K: int
    s_lo: float
    s_hi: float
    outlier_frac: float
    name: str = ""
    gated: int = 0    # 0: plain linear; 1 SiLU / 2 GELU-tanh: gated pair with 2N weight rows

    @property
    def rows(self) -> int:
        """Weight rows: N, or 2N (gate rows over up rows) for a gated pair."""
        return 2 * self.N if self.gated else self.N

    @property
    def weight_bytes(self) -> int:
        """Algorithmic bytes of packed int4 weights plus fp16 block scales."""
        return self.rows * self.K // 2 + self.rows * (self.K // BLOCK) * 2

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes of one call: weights + scales + x + y."""
        return self.weight_bytes + 2 * self.M * self.K + 2 * self.M * self.N

    @property
    def ops(self) -> int:
        """Integer multiply-add operations of one call, counted as 2*M*rows*K."""
        return 2 * self.M * self.rows * self.K


@dataclass
class Workload:
    name: str
    seed: int
    linears: list
    weight_sets: int = 1
    description: str = ""
    extra: dict = field(default_factory=dict)


# Decoder layer at hidden 2048: q, k, v, o, gate, up, down as (N, K).
DECODER_LAYER = [("q", 2048, 2048), ("k", 256, 2048), ("v", 256, 2048), ("o", 2048, 2048),
                 ("gate", 8192, 2048), ("up", 8192, 2048), ("down", 2048, 8192)]

# The same layer with the fusions of the pages' Figure 4 left ("Scaling
# On-Device GPU Inference for Large Generative Models"): q, k and v as one
# N=2560 projection of the shared input, and gate and up as one gated pair
# (GELU, tanh form) whose element-wise product is the down projection's input.
DECODER_LAYER_FUSED = [("qkv", 2560, 2048, 0), ("o", 2048, 2048, 0), ("gate_up", 8192, 2048, 2),
                       ("down", 2048, 8192, 0)]


def workloads():
    """The workloads, in order: tiny, decode FFN up, prefill FFN up, decoder layers, shape sweep,
    fused decoder layers."""
    w = []
    w.append(Workload("tiny_m1_k256_n512", 0,
                      [Linear(1, 512, 256, 0.005, 0.02, 0.0, "tiny")],
                      description="single linear M=1 K=256 N=512, scales U[0.005,0.02], x N(0,1)"))
    w.append(Workload("decode_ffn_up_m1_k2048_n8192", 1000,
                      [Linear(1, 8192, 2048, 0.002, 0.01, 0.01, "ffn_up")], weight_sets=16,
                      description="decode FFN up-projection M=1 K=2048 N=8192, 16 rotating weight sets"))
    w.append(Workload("prefill_ffn_up_m512_k2048_n8192", 2000,
                      [Linear(512, 8192, 2048, 0.002, 0.01, 0.01, "ffn_up")],
                      description="prefill FFN up-projection M=512 K=2048 N=8192"))
    w.append(Workload("decoder_layers_m1_26x7", 3000,
                      [Linear(1, n, k, 0.002, 0.01, 0.01, nm) for nm, n, k in DECODER_LAYER],
                      weight_sets=26,
                      description="decode step over 26 decoder layers x 7 linears, M=1",
                      extra={"layers": 26, "decode_steps": 128}))
    sweep = []
    for K, N in ((4096, 14336), (14336, 4096)):
        for M in (1, 4, 8, 64, 512):
            sweep.append(Linear(M, N, K, 0.001, 0.008, 0.01, f"sweep_m{M}_k{K}_n{N}"))
    w.append(Workload("shape_sweep", 4000, sweep,
                      description="K,N in {(4096,14336),(14336,4096)}, M in {1,4,8,64,512}"))
    w.append(Workload("decoder_layers_m1_26x4_fused", 5000,
                      [Linear(1, n, k, 0.002, 0.01, 0.01, nm, gated=act) for nm, n, k, act in DECODER_LAYER_FUSED],
                      weight_sets=26,
                      description="decode step over 26 decoder layers: qkv (N=2560), o, gated gate/up (GELU), down",
                      extra={"layers": 26, "decode_steps": 128}))
    return w


def make_linear_inputs(lin: Linear, seed: int, weight_set: int = 0):
    """(x fp16 [M][K], codes int8 [rows][K], scales fp16 [rows][K/32]) for one linear of a workload
    (rows = N, or 2N with the gate rows over the up rows for a gated pair)."""
    codes, scales = make_weights(lin.rows, lin.K, seed + 1 + weight_set, lin.s_lo, lin.s_hi)
    x = make_x(lin.M, lin.K, seed, lin.outlier_frac)
    return x, codes, scales
