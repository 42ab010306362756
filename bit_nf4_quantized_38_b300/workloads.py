"""Seeded synthetic inputs shaped like the LLaMA layers the method is run on.

This module only draws random numbers and describes shapes; it holds none of
the method's arithmetic, so both the CUDA path's tests/benchmarks and the CPU
oracle's tests can take their inputs from it.

Shapes are the linear layers of LLaMA 7B / 13B / 33B / 65B (the model family
the QLoRA pages finetune: 7/13/33/65B Guanaco).  Values are drawn in fp32
with torch's CPU generator (or a seeded CUDA generator for the 33B stack,
which is too large to draw on the host) and rounded to bf16 (RNE).  Every draw
is seeded with `seed0 + index` in a fixed order.
"""
import math
from dataclasses import dataclass, field

import numpy as np
import torch


# ----------------------------------------------------------------------------
# shapes

LLAMA7B_LINEARS = [  # (name, out N, in K)
    ("q_proj", 4096, 4096), ("k_proj", 4096, 4096), ("v_proj", 4096, 4096),
    ("o_proj", 4096, 4096), ("gate_proj", 11008, 4096), ("up_proj", 11008, 4096),
    ("down_proj", 4096, 11008),
]
LLAMA13B_DECODE_SHAPES = [("attn_5120x5120", 5120, 5120), ("up_13824x5120", 13824, 5120),
                          ("down_5120x13824", 5120, 13824)]
LLAMA33B_LINEARS = [
    ("q_proj", 6656, 6656), ("k_proj", 6656, 6656), ("v_proj", 6656, 6656),
    ("o_proj", 6656, 6656), ("gate_proj", 17920, 6656), ("up_proj", 17920, 6656),
    ("down_proj", 6656, 17920),
]
LLAMA65B_LINEARS = [
    ("q_proj", 8192, 8192), ("k_proj", 8192, 8192), ("v_proj", 8192, 8192),
    ("o_proj", 8192, 8192), ("gate_proj", 22016, 8192), ("up_proj", 22016, 8192),
    ("down_proj", 8192, 22016),
]


@dataclass
class LinearCase:
    """One QLoRA linear: weight N x K, tokens M, LoRA rank r, scale alpha / r."""
    name: str
    N: int
    K: int
    M: int
    r: int
    alpha: float
    w_std: float
    seed0: int
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    w_dist: str = "normal"  # or "student_t4"

    @property
    def scale(self):
        return self.alpha / self.r


@dataclass
class Workload:
    name: str
    cases: list = field(default_factory=list)
    layers: int = 1


def single_linear_1024():
    """1024 x 1024 weight N(0, 0.02^2), 16 tokens, r=8, alpha=16 (s=2), seed 0."""
    return Workload("single_linear_1024x1024_M16_r8",
                    [LinearCase("linear", 1024, 1024, 16, 8, 16.0, 0.02, 0)])


def llama7b_linears(M=4096, r=64, alpha=16.0):
    """The 7 LLaMA-7B linears, weights N(0, 0.02^2) with 0.1% of entries x20, M tokens."""
    return Workload(f"llama7b_7linears_M{M}_r{r}",
                    [LinearCase(n, N, K, M, r, alpha, 0.02, 100 + 10 * i, 0.001, 20.0)
                     for i, (n, N, K) in enumerate(LLAMA7B_LINEARS)])


def llama13b_decode(M=1, r=64, alpha=16.0):
    """LLaMA-13B linear shapes at decode batch M (1, 4 or 16)."""
    return Workload(f"llama13b_decode_M{M}_r{r}",
                    [LinearCase(n, N, K, M, r, alpha, 0.02, 200 + 10 * i)
                     for i, (n, N, K) in enumerate(LLAMA13B_DECODE_SHAPES)])


def llama65b_layer_quant():
    """The 7 linear weights of one LLaMA-65B layer, Student-t(4) values with std 0.015."""
    return Workload("llama65b_layer_quantize",
                    [LinearCase(n, N, K, 0, 0, 0.0, 0.015, 300 + 10 * i, w_dist="student_t4")
                     for i, (n, N, K) in enumerate(LLAMA65B_LINEARS)])


def llama33b_stack(M=2048, r=64, alpha=16.0, layers=60):
    """60 layers x 7 LLaMA-33B linears, weights N(0, 0.015^2), M tokens."""
    cases = []
    for L in range(layers):
        for i, (n, N, K) in enumerate(LLAMA33B_LINEARS):
            cases.append(LinearCase(f"layer{L}.{n}", N, K, M, r, alpha, 0.015,
                                    10_000 + 100 * L + 10 * i))
    return Workload(f"llama33b_stack_{layers}x7_M{M}_r{r}", cases, layers=layers)


# ----------------------------------------------------------------------------
# draws

def _gen(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std, seed, device="cpu"):
    """N(0, std^2) drawn in fp32, rounded to bf16."""
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def normal_with_outliers_bf16(shape, std, p, factor, seed, device="cpu"):
    """N(0, std^2) in fp32; an independent Bernoulli(p) mask scales entries by `factor`; bf16."""
    g = _gen(seed, device)
    w = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    if p > 0:
        mask = torch.rand(shape, generator=g, device=device) < p
        w = torch.where(mask, w * factor, w)
    return w.to(torch.bfloat16)


def student_t4_bf16(shape, std, seed, device="cpu", rows_per_chunk=1024):
    """Student-t with 4 degrees of freedom scaled to standard deviation `std`; bf16.

    t = z0 / sqrt((z1^2 + z2^2 + z3^2 + z4^2) / 4) has variance 4 / (4 - 2) = 2,
    so it is multiplied by std / sqrt(2).  Rows are drawn in chunks of
    `rows_per_chunk` (five normal planes per chunk, in order) to bound memory.
    """
    g = _gen(seed, device)
    rows, cols = shape
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, rows_per_chunk):
        r1 = min(rows, r0 + rows_per_chunk)
        z = torch.randn((5, r1 - r0, cols), generator=g, device=device, dtype=torch.float32)
        chi = (z[1:] ** 2).sum(0) / 4.0
        out[r0:r1] = (z[0] / torch.sqrt(chi) * (std / math.sqrt(2.0))).to(torch.bfloat16)
    return out


def case_weight(case, device="cpu"):
    if case.w_dist == "student_t4":
        return student_t4_bf16((case.N, case.K), case.w_std, case.seed0, device)
    return normal_with_outliers_bf16((case.N, case.K), case.w_std, case.outlier_p,
                                     case.outlier_scale, case.seed0, device)


def case_inputs(case, device="cpu", M=None):
    """X (M x K), A (K x r), B (r x N), dY (M x N): bf16, seeds seed0+1..4."""
    M = case.M if M is None else M
    X = normal_bf16((M, case.K), 1.0, case.seed0 + 1, device)
    A = normal_bf16((case.K, case.r), 1.0 / math.sqrt(case.r), case.seed0 + 2, device)
    B = normal_bf16((case.r, case.N), 0.01, case.seed0 + 3, device)
    dY = normal_bf16((M, case.N), 1.0, case.seed0 + 4, device)
    return X, A, B, dY


def bf16_bits(t):
    """A bf16 torch tensor's bit patterns as a numpy uint16 array (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
