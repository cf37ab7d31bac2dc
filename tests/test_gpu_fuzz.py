"""Randomized shapes: every quantizer bit for bit and every GEMM pair within
the GEMM pass rule against the oracle, on shapes drawn from a seeded
generator rather than chosen by hand, so that row, column, K-block and tile
tails fall at arbitrary positions.

Each shape obeys the format's documented divisibility rules (K % 32 for MX,
whole scale chunks for the tensor-core tiling, 128-row blocks for the block
formats, N % 8 for int4 and for Y's 16-byte rows) and is small enough for the
oracle to finish in a second or two.  The checks themselves are the ones of
test_gpu_quant.py and test_gpu_gemm.py, called with these shapes.
"""
import numpy as np
import pytest
import torch

import test_gpu_gemm as G
import test_gpu_quant as Qt
from gpu_util import np_f32, np_u8, require_gpu
from serving_amax_reduce_gb300 import inputs

pytestmark = pytest.mark.gpu

N_SHAPES = 6


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def draw(kind: str, seed: int):
    """(M, N, K) for a GEMM kind, or (rows, K) for a quantizer kind."""
    rng = np.random.default_rng(seed)
    r = lambda lo, hi: int(rng.integers(lo, hi + 1))     # noqa: E731
    M = r(1, 600)
    if kind == "fp8_tensor":
        return M, 8 * r(1, 128), 16 * r(1, 128)
    if kind in ("fp8_block_token", "fp8_block_group128"):
        return M, 128 * r(1, 8), 128 * r(1, 16)
    if kind == "mxfp8":
        return M, 8 * r(1, 128), 128 * r(1, 16)
    if kind in ("mxfp4", "nvfp4"):
        return M, 8 * r(1, 128), 256 * r(1, 8)
    if kind == "mxfp4_dual":
        return M, 8 * r(1, 128), 512 * r(1, 4)
    if kind == "int8":
        return M, 8 * r(1, 128), 16 * r(1, 128)
    if kind == "fp8_tensor_fused_x":
        return r(1, 128), 8 * r(1, 128), 16 * r(1, 128)
    if kind == "w4a16":     # half of the draws on the warp-level kernel (M <= 16), half on the tcgen05 one
        return (r(1, 16) if rng.random() < 0.5 else r(17, 80)), 8 * r(1, 128), 128 * r(1, 24)
    # quantizers: (rows, K)
    if kind == "q_row":
        return r(1, 600), 8 * r(1, 2048)
    if kind == "q_block128":
        return 128 * r(1, 6), 128 * r(1, 24)
    if kind == "q_group128":
        return r(1, 600), 128 * r(1, 24)
    if kind == "q_mx":
        return r(1, 600), 32 * r(1, 96)
    if kind == "q_nvfp4":
        return r(1, 600), 16 * r(1, 192)
    if kind == "q_dual":
        return r(1, 600), 512 * r(1, 6)
    if kind == "q_int4":
        return 8 * r(1, 100), 128 * r(1, 24)
    raise ValueError(kind)


def fp8_tensor_case(q, orc, M, N, K):
    lin = inputs.fp8_tensor_linear(M, K, N)
    x, w = lin.make_x(), lin.make_w()
    F = q.Fmt
    bx = q.quantize_act(F.FP8_TENSOR, x.cuda())
    bw = q.quantize_weight(F.FP8_TENSOR, w.cuda())
    y = q.gemm(F.FP8_TENSOR, F.FP8_TENSOR, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"])
    torch.cuda.synchronize()
    xh = orc.dequant_fp8_tensor(np_u8(bx["codes"]).reshape(M, K), np_f32(bx["scales"])[0])
    wh = orc.dequant_fp8_tensor(np_u8(bw["codes"]).reshape(N, K), np_f32(bw["scales"])[0])
    G.check(orc, G.y_np(y), orc.gemm_ref(xh, wh), x, w)


GEMMS = {
    "fp8_tensor": fp8_tensor_case,
    "fp8_block_token": G.fp8_block_case,
    "fp8_block_group128": G.fp8_group_case,
    "mxfp8": G.mxfp8_case,
    "mxfp4": G.mxfp4_case,
    "mxfp4_dual": G.mxfp4_dual_case,
    "nvfp4": G.nvfp4_case,
    "int8": G.int8_case,
    "fp8_tensor_fused_x": G.fused_x_case,
    "w4a16": lambda q, orc, M, N, K: G.w4a16_case(q, orc, M, K, N),
}


@pytest.mark.parametrize("i", range(N_SHAPES))
@pytest.mark.parametrize("kind", list(GEMMS))
def test_gemm_random_shapes(q, orc, kind, i):
    M, N, K = draw(kind, 7919 * i + sum(map(ord, kind)))
    GEMMS[kind](q, orc, M, N, K)


# Pairs whose kernels take any N (the W scales of the tensor-core tiling are padded to 128 rows,
# Y is stored by TMA with its columns clipped at N): N is drawn freely, Y then needs a padded
# leading dimension for its 16-byte rows, as a caller with such N would pass it.
RAGGED_N = ["fp8_tensor", "mxfp8", "mxfp4", "mxfp4_dual", "nvfp4", "int8", "fp8_tensor_fused_x"]


@pytest.mark.parametrize("i", range(3))
@pytest.mark.parametrize("kind", RAGGED_N)
def test_gemm_random_shapes_any_n(q, orc, kind, i, monkeypatch):
    M, _, K = draw(kind, 3571 * i + sum(map(ord, kind)))
    N = int(np.random.default_rng(9001 * i + len(kind)).integers(1, 1031))
    orig = q.gemm

    def gemm_padded_y(*args, **kw):
        if kw.get("y") is None:
            m, n = args[2], args[3]
            ld = (n + 7) // 8 * 8 + 8
            kw["y"] = torch.full((m, ld), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :n]
        return orig(*args, **kw)

    monkeypatch.setattr(q, "gemm", gemm_padded_y)
    GEMMS[kind](q, orc, M, N, K)


QUANTS = {
    "q_row": lambda q, orc, rows, K, i: (Qt.test_fp8_token(q, orc, rows, K, "outlier"),
                                         Qt.test_int8_row(q, orc, rows, K, "outlier", i % 2 == 1)),
    "q_block128": lambda q, orc, rows, K, i: Qt.test_fp8_block128(q, orc, rows, K, "normal"),
    "q_group128": lambda q, orc, rows, K, i: Qt.test_fp8_group128(q, orc, rows, K, "outlier"),
    "q_mx": lambda q, orc, rows, K, i: (Qt.test_mxfp8(q, orc, rows, K, "normal", i % 2 == 1),
                                        Qt.test_mxfp4(q, orc, rows, K, "normal", i % 2 == 0)),
    "q_nvfp4": lambda q, orc, rows, K, i: Qt.test_nvfp4(q, orc, rows, K, "outlier", i % 2 == 1),
    "q_dual": lambda q, orc, rows, K, i: Qt.test_mxfp4_dual(q, orc, rows, K, "normal", i % 2 == 1),
    "q_int4": lambda q, orc, rows, K, i: (Qt.test_int4_g128(q, orc, rows, K, "normal"),
                                          Qt.test_int4_g128_sym(q, orc, rows, K, "normal")),
}


@pytest.mark.parametrize("i", range(N_SHAPES))
@pytest.mark.parametrize("kind", list(QUANTS))
def test_quantizer_random_shapes(q, orc, kind, i):
    rows, K = draw(kind, 104729 * i + sum(map(ord, kind)))
    QUANTS[kind](q, orc, rows, K, i)
