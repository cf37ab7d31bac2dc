"""Shared helpers for the GPU parity tests (marshalling only)."""
import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from serving_amax_reduce_gb300 import build
    build.build()
    from serving_amax_reduce_gb300 import qlin
    return qlin


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy()


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.float32).numpy()


def edge_bf16(rows: int, K: int, seed: int = 0) -> torch.Tensor:
    """Edge-case values: zeros of both signs, bf16 subnormals, values far
    beyond the formats' ranges, exact powers of two, whole zero rows and
    granules, on top of N(0,1)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g)
    u = torch.rand(rows, K, generator=g)
    x[u < 0.05] = 0.0
    x[(u >= 0.05) & (u < 0.10)] = -0.0
    x[(u >= 0.10) & (u < 0.13)] *= 1e-39                        # bf16 subnormals
    x[(u >= 0.13) & (u < 0.15)] *= 1e30
    x[(u >= 0.15) & (u < 0.18)] = torch.exp2(torch.randint(-20, 20, (int(((u >= 0.15) & (u < 0.18)).sum()),),
                                                           generator=g).float())
    if rows > 2:
        x[1] = 0.0
    x[:, :32] = 0.0                                                # a zero granule in every row
    return x.to(torch.bfloat16)
