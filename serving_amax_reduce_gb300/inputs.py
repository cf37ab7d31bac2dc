"""Seeded synthetic inputs for the quantized-linear workloads.

This module holds random-number generation and shapes only: none of the
quantization or GEMM arithmetic.  Both the CUDA path and the CPU oracle read
the bytes it produces.

The pages' own workloads (Qwen-Image-2512 at 1024x1024, Wan2.2 video DiTs,
FLUX.1-dev; "vLLM-Omni 量化推理实践" section "实验设置与样例输出", and
"vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다" section "모델 적용 범위")
need trained checkpoints that are not available, so these tensors stand in for
their linear layers: the same GEMM shapes and the value distributions stated
for each workload below.

Seeds: ``1000 + 10 * workload + variant``; every tensor of a workload draws
from its own generator so that the weights do not depend on the activations.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in float32, then rounded to bf16."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def outlier_channel_bf16(M: int, K: int, seed: int, frac: float = 0.01, mult: float = 20.0,
                         df: int = 3, device="cpu", return_cols: bool = False):
    """DiT-like activations: N(0,1) except ceil(frac*K) seeded channels (columns)
    whose entries are replaced by mult * t_df (Student-t with df degrees of
    freedom, drawn as Z / sqrt(chi2_df / df))."""
    g = _gen(seed, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    n_out = int(math.ceil(frac * K))
    cols = torch.randperm(K, generator=g, device=device)[:n_out]
    z = torch.randn(M, n_out, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.randn(M, n_out, df, generator=g, device=device, dtype=torch.float32).pow(2).sum(-1)
    t = z / torch.sqrt(chi2 / df)
    x[:, cols] = mult * t
    x = x.to(torch.bfloat16)
    return (x, cols) if return_cols else x


@dataclass
class Linear:
    """One linear layer's inputs: X [M,K] and W [N,K] (nn.Linear layout)."""
    name: str
    M: int
    K: int
    N: int
    x_fmt: str
    w_fmt: str
    x_seed: int
    w_seed: int
    x_kind: str          # "normal" or "outlier"
    x_std: float = 1.0
    w_std: float = 0.02
    extra: dict = field(default_factory=dict)

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def make_x(self, device="cpu") -> torch.Tensor:
        if self.x_kind == "outlier":
            return outlier_channel_bf16(self.M, self.K, self.x_seed, device=device)
        return normal_bf16((self.M, self.K), self.x_std, self.x_seed, device=device)

    def make_w(self, device="cpu") -> torch.Tensor:
        return normal_bf16((self.N, self.K), self.w_std, self.w_seed, device=device)


def _seed(workload: int, variant: int) -> int:
    return 1000 + 10 * workload + variant


def fp8_tensor_linear(M=128, K=1024, N=1024) -> Linear:
    """FP8 E4M3 per-tensor W8A8: X and W both N(0, 0.02^2)."""
    return Linear("fp8_tensor", M, K, N, "fp8_tensor", "fp8_tensor",
                  _seed(1, 0), _seed(1, 1), "normal", x_std=0.02, w_std=0.02)


def fp8_tensor_fused_linear(M=128, K=1024, N=1024) -> Linear:
    """The per-tensor FP8 linear with its activation quantization fused into the
    GEMM: the same X and W as fp8_tensor_linear, X handed over in bf16."""
    return Linear("fp8_tensor_fused_x", M, K, N, "bf16", "fp8_tensor",
                  _seed(1, 0), _seed(1, 1), "normal", x_std=0.02, w_std=0.02)


W4A16_SHAPES = [(4096, 4096), (4096, 12288), (12288, 4096)]   # (K, N)
W4A16_M = [1, 16, 64]


def w4a16_linear(M: int, K: int, N: int) -> Linear:
    """int4 g128 weight-only decode GEMM: W N(0, 0.02^2), X N(0, 1) bf16."""
    v = W4A16_SHAPES.index((K, N)) if (K, N) in W4A16_SHAPES else 9
    return Linear(f"w4a16_M{M}_K{K}_N{N}", M, K, N, "bf16", "int4_g128",
                  _seed(2, 2 * v), _seed(2, 2 * v + 1), "normal", x_std=1.0, w_std=0.02)


def w4a16_sym_linear(M: int, K: int, N: int) -> Linear:
    """The W4A16 decode shapes and distributions with symmetric int4 weights
    (zero point 8), seeds of workload 9."""
    v = W4A16_SHAPES.index((K, N)) if (K, N) in W4A16_SHAPES else 4
    return Linear(f"w4a16_sym_M{M}_K{K}_N{N}", M, K, N, "bf16", "int4_g128_sym",
                  _seed(9, 2 * v), _seed(9, 2 * v + 1), "normal", x_std=1.0, w_std=0.02)


FP8_MLP_SHAPES = [(3072, 12288), (12288, 3072)]                # (K, N)
FP8_MLP_B = [1, 4, 8]


def fp8_block_linear(B: int, K: int, N: int, M: int | None = None) -> Linear:
    """DiT MLP: per-token E4M3 activations with 1% outlier channels (x20 Student-t
    df=3) over N(0,1); 128x128-block E4M3 weights N(0, 0.02^2)."""
    v = FP8_MLP_SHAPES.index((K, N)) if (K, N) in FP8_MLP_SHAPES else 5
    M = 4096 * B if M is None else M
    return Linear(f"fp8_block_B{B}_K{K}_N{N}", M, K, N, "fp8_token", "fp8_block128",
                  _seed(3, 2 * v), _seed(3, 2 * v + 1), "outlier", w_std=0.02)


MXFP8_SHAPES = [(5120, 13824), (13824, 5120), (5120, 5120)]   # (K, N)
MXFP8_M = 20280


def mxfp8_linear(K: int, N: int, M: int = MXFP8_M) -> Linear:
    """Video-DiT MXFP8: X N(0,1), W N(0, 0.015^2), M = 20280 tokens."""
    v = MXFP8_SHAPES.index((K, N)) if (K, N) in MXFP8_SHAPES else 7
    return Linear(f"mxfp8_K{K}_N{N}", M, K, N, "mxfp8", "mxfp8",
                  _seed(4, 2 * v), _seed(4, 2 * v + 1), "normal", x_std=1.0, w_std=0.015)


def mxfp4_dual_linear(K: int, N: int, M: int = MXFP8_M) -> Linear:
    """MXFP4 dual-scale W4A4 on the video-DiT shapes and distributions of the
    MXFP8 workload, the same X and W as the single-scale MXFP4 row (seeds of
    workload 6)."""
    v = MXFP8_SHAPES.index((K, N)) if (K, N) in MXFP8_SHAPES else 7
    return Linear(f"mxfp4_dual_K{K}_N{N}", M, K, N, "mxfp4_dual", "mxfp4_dual",
                  _seed(6, 2 * v), _seed(6, 2 * v + 1), "normal", x_std=1.0, w_std=0.015)


def fp8_group_linear(K: int, N: int, M: int = 4096) -> Linear:
    """FP8 1 x 128 dynamic activation groups x 128x128-block weights on the DiT MLP
    shapes and distributions of the FP8 block workload (1% outlier channels)."""
    v = FP8_MLP_SHAPES.index((K, N)) if (K, N) in FP8_MLP_SHAPES else 5
    return Linear(f"fp8_group_K{K}_N{N}", M, K, N, "fp8_group128", "fp8_block128",
                  _seed(7, 2 * v), _seed(7, 2 * v + 1), "outlier", x_std=1.0, w_std=0.02)


def int8_linear(K: int, N: int, M: int = 4096) -> Linear:
    """INT8 W8A8 (per-token X, per-channel W) on the DiT MLP shapes and
    distributions of the FP8 block workload (1% outlier channels in X)."""
    v = FP8_MLP_SHAPES.index((K, N)) if (K, N) in FP8_MLP_SHAPES else 5
    return Linear(f"int8_K{K}_N{N}", M, K, N, "int8_row", "int8_row",
                  _seed(8, 2 * v), _seed(8, 2 * v + 1), "outlier", x_std=1.0, w_std=0.02)


def mxfp4_linear(K: int, N: int, M: int = MXFP8_M) -> Linear:
    """MXFP4 W4A4 (the next format of the online MXFP4 path) on the video-DiT
    shapes and distributions of the MXFP8 workload: X N(0,1), W N(0, 0.015^2)."""
    v = MXFP8_SHAPES.index((K, N)) if (K, N) in MXFP8_SHAPES else 7
    return Linear(f"mxfp4_K{K}_N{N}", M, K, N, "mxfp4", "mxfp4",
                  _seed(6, 2 * v), _seed(6, 2 * v + 1), "normal", x_std=1.0, w_std=0.015)


def mixed_stack(M: int = 32768, d: int = 3072, ff: int = 12288) -> list[Linear]:
    """Eight linears: NVFP4 W4A4 q/k/v/out projections (d x d) and FP8 block-128
    MLP linears (two d->ff, two ff->d); activations as the DiT MLP workload."""
    layers = []
    for i, nm in enumerate(["q", "k", "v", "out"]):
        layers.append(Linear(f"nvfp4_{nm}", M, d, d, "nvfp4", "nvfp4",
                             _seed(5, 2 * i), _seed(5, 2 * i + 1), "outlier", w_std=0.02))
    for i, (nm, K, N) in enumerate([("up0", d, ff), ("down0", ff, d), ("up1", d, ff), ("down1", ff, d)]):
        j = 4 + i
        layers.append(Linear(f"fp8_block_{nm}", M, K, N, "fp8_token", "fp8_block128",
                             _seed(5, 2 * j), _seed(5, 2 * j + 1), "outlier", w_std=0.02))
    return layers
