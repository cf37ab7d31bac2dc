"""GPU quantized GEMMs against the fp64 oracle on identical quantized inputs.

Pass rule: relative Frobenius error <= 2e-3 + the relative error of rounding
the oracle's own result to bf16.  Each case also checks that the output is
not the unquantized bf16 product (the quantized path really ran).
"""
import numpy as np
import pytest
import torch

from gpu_util import bits, np_f32, np_u8, require_gpu
from layouts import mma_to_canonical
from serving_amax_reduce_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def y_np(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def check(orc, y_gpu, y_ref, x=None, w=None, rows=None):
    from serving_amax_reduce_gb300 import qlin
    assert qlin.read_device_status() == 0, "a bounded device wait expired"
    ok, m = orc.gemm_pass(y_gpu, y_ref)
    assert ok, m
    assert np.isfinite(y_gpu).all()
    if x is not None:
        xb = x.float() if rows is None else x[rows].float()
        plain = (xb.double() @ w.double().T).numpy()
        d = np.linalg.norm(y_gpu - plain) / np.linalg.norm(plain)
        assert d > 1e-5, "output equals the unquantized product"
    return m


def sample_rows(M, n, seed=0):
    if M <= n:
        return np.arange(M)
    return np.sort(np.random.default_rng(seed).choice(M, n, replace=False))


# ------------------------------------------------------------------ FP8 per-tensor
@pytest.mark.parametrize("M,N,K", [(128, 1024, 1024), (200, 512, 384), (1, 256, 128), (333, 1040, 1040)])
def test_fp8_tensor_gemm(q, orc, M, N, K):
    lin = inputs.fp8_tensor_linear(M, K, N)
    x, w = lin.make_x(), lin.make_w()
    F = q.Fmt
    bx = q.quantize_act(F.FP8_TENSOR, x.cuda())
    bw = q.quantize_weight(F.FP8_TENSOR, w.cuda())
    y = q.gemm(F.FP8_TENSOR, F.FP8_TENSOR, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"])
    torch.cuda.synchronize()
    xh = orc.dequant_fp8_tensor(np_u8(bx["codes"]).reshape(M, K), np_f32(bx["scales"])[0])
    wh = orc.dequant_fp8_tensor(np_u8(bw["codes"]).reshape(N, K), np_f32(bw["scales"])[0])
    check(orc, y_np(y), orc.gemm_ref(xh, wh), x, w)


def test_fp8_tensor_gemm_bias(q, orc):
    M, N, K = 200, 512, 256
    lin = inputs.fp8_tensor_linear(M, K, N)
    x, w = lin.make_x(), lin.make_w()
    bias = inputs.normal_bf16((1, N), 0.05, 99)[0]
    F = q.Fmt
    bx = q.quantize_act(F.FP8_TENSOR, x.cuda())
    bw = q.quantize_weight(F.FP8_TENSOR, w.cuda())
    y = q.gemm(F.FP8_TENSOR, F.FP8_TENSOR, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"],
               bias=bias.cuda())
    torch.cuda.synchronize()
    xh = orc.dequant_fp8_tensor(np_u8(bx["codes"]).reshape(M, K), np_f32(bx["scales"])[0])
    wh = orc.dequant_fp8_tensor(np_u8(bw["codes"]).reshape(N, K), np_f32(bw["scales"])[0])
    check(orc, y_np(y), orc.gemm_ref(xh, wh, bias=orc.bf16_values(bits(bias)[None, :])[0]))


# ------------------------------------------------------------------ FP8 token x block-128
def fp8_block_case(q, orc, M, N, K, nrows=None, with_bias=False):
    lin = inputs.fp8_block_linear(1, K, N, M=M)
    x, w = lin.make_x(), lin.make_w()
    F = q.Fmt
    bx = q.quantize_act(F.FP8_TOKEN, x.cuda())
    bw = q.quantize_weight(F.FP8_BLOCK128, w.cuda())
    bias = inputs.normal_bf16((1, N), 0.05, 78)[0] if with_bias else None
    y = q.gemm(F.FP8_BLOCK128, F.FP8_TOKEN, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"],
               bias=bias.cuda() if with_bias else None)
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    xc = np_u8(bx["codes"]).reshape(M, K)[rows]
    xs = np_f32(bx["scales"])[:M][rows]
    xh = orc.dequant_fp8_token(xc, xs)
    wh = orc.dequant_fp8_block128(np_u8(bw["codes"]).reshape(N, K), np_f32(bw["scales"]).reshape(N // 128, K // 128))
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh, bias=b), x, w, rows=torch.from_numpy(rows))


@pytest.mark.parametrize("M,N,K", [(200, 512, 384), (128, 256, 128), (1, 384, 256), (513, 1280, 1152)])
def test_fp8_block_gemm(q, orc, M, N, K):
    fp8_block_case(q, orc, M, N, K)


def test_fp8_block_gemm_bias_ragged(q, orc):
    # N = 640 is not a multiple of the 192-column tile: the last tile is partial
    fp8_block_case(q, orc, 130, 640, 256, with_bias=True)


@pytest.mark.slow
@pytest.mark.parametrize("B", [1, 4, 8])
@pytest.mark.parametrize("K,N", [(3072, 12288), (12288, 3072)])
def test_fp8_block_gemm_full_size(q, orc, B, K, N):
    fp8_block_case(q, orc, 4096 * B, N, K, nrows=256)


# ------------------------------------------------------------------ FP8 per-tensor, X quantized inside the GEMM
def fused_x_case(q, orc, M, N, K, with_bias=False, zero_x=False):
    lin = inputs.fp8_tensor_linear(M, K, N)
    x, w = lin.make_x(), lin.make_w()
    if zero_x:
        x = torch.zeros_like(x)
    F = q.Fmt
    xd = x.cuda()
    bw = q.quantize_weight(F.FP8_TENSOR, w.cuda())
    bias = inputs.normal_bf16((1, N), 0.05, 82)[0] if with_bias else None
    bd = bias.cuda() if with_bias else None
    y = q.gemm(F.FP8_TENSOR, F.BF16, M, N, K, xd, None, bw["codes"], bw["scales"], bias=bd)
    # the same linear in two steps: quantize X, then the per-tensor GEMM
    bx = q.quantize_act(F.FP8_TENSOR, xd)
    y2 = q.gemm(F.FP8_TENSOR, F.FP8_TENSOR, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"], bias=bd)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "fused and two-step results differ"
    # and against the oracle's own quantization of X
    cx, sx = orc.quant_fp8_tensor(bits(x))
    wh = orc.dequant_fp8_tensor(np_u8(bw["codes"]).reshape(N, K), np_f32(bw["scales"])[0])
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    ref = orc.gemm_ref(orc.dequant_fp8_tensor(cx, sx), wh, bias=b)
    if zero_x:
        assert np.array_equal(y_np(y), np.broadcast_to(orc.bf16_values(bits(bias)[None, :]) if with_bias else 0.0,
                                                       (M, N)))
        return None
    return check(orc, y_np(y), ref, x, w)


# one row tile at single-request row counts; ragged N and K; K of one block
@pytest.mark.parametrize("M,N,K", [(128, 1024, 1024), (1, 256, 128), (77, 640, 1040), (128, 12288, 3072),
                                   (5, 320, 2048)])
def test_fp8_tensor_fused_x_gemm(q, orc, M, N, K):
    fused_x_case(q, orc, M, N, K)


def test_fp8_tensor_fused_x_gemm_bias_and_zero(q, orc):
    fused_x_case(q, orc, 100, 512, 384, with_bias=True)
    fused_x_case(q, orc, 16, 256, 256, with_bias=True, zero_x=True)


# ------------------------------------------------------------------ FP8 128x128 block W x 1x128 group X
def fp8_group_case(q, orc, M, N, K, nrows=None, with_bias=False):
    lin = inputs.fp8_block_linear(1, K, N, M=M)
    x, w = lin.make_x(), lin.make_w()
    F = q.Fmt
    bx = q.quantize_act(F.FP8_GROUP128, x.cuda())
    bw = q.quantize_weight(F.FP8_BLOCK128, w.cuda())
    bias = inputs.normal_bf16((1, N), 0.05, 80)[0] if with_bias else None
    y = q.gemm(F.FP8_BLOCK128, F.FP8_GROUP128, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"],
               bias=bias.cuda() if with_bias else None)
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    xh = orc.dequant_fp8_group128(np_u8(bx["codes"]).reshape(M, K)[rows],
                                  np_f32(bx["scales"]).reshape(M, K // 128)[rows])
    wh = orc.dequant_fp8_block128(np_u8(bw["codes"]).reshape(N, K), np_f32(bw["scales"]).reshape(N // 128, K // 128))
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh, bias=b), x, w, rows=torch.from_numpy(rows))


@pytest.mark.parametrize("M,N,K", [(200, 512, 384), (128, 256, 128), (1, 384, 256), (513, 1280, 1152)])
def test_fp8_group128_gemm(q, orc, M, N, K):
    fp8_group_case(q, orc, M, N, K)


def test_fp8_group128_gemm_bias(q, orc):
    fp8_group_case(q, orc, 130, 640, 256, with_bias=True)


@pytest.mark.slow
def test_fp8_group128_gemm_full_size(q, orc):
    fp8_group_case(q, orc, 4096, 12288, 3072, nrows=256)


# ------------------------------------------------------------------ INT8 W8A8
def int8_case(q, orc, M, N, K, nrows=None, with_bias=False):
    lin = inputs.int8_linear(K, N, M=M)
    x, w = lin.make_x(), lin.make_w()
    F = q.Fmt
    bx = q.quantize_act(F.INT8_ROW, x.cuda())
    bw = q.quantize_weight(F.INT8_ROW, w.cuda())
    bias = inputs.normal_bf16((1, N), 0.05, 81)[0] if with_bias else None
    y = q.gemm(F.INT8_ROW, F.INT8_ROW, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"],
               bias=bias.cuda() if with_bias else None)
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    cx = np_u8(bx["codes"]).reshape(M, K).view(np.int8)
    cw = np_u8(bw["codes"]).reshape(N, K).view(np.int8)
    xh = orc.dequant_int8_row(cx[rows], np_f32(bx["scales"])[:M][rows])
    wh = orc.dequant_int8_row(cw, np_f32(bw["scales"])[:N])
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh, bias=b), x, w, rows=torch.from_numpy(rows))


# ragged M and N tiles, K not a multiple of the 64-wide stage, one row, one stage
@pytest.mark.parametrize("M,N,K", [(200, 512, 384), (128, 256, 64), (1, 384, 256), (300, 640, 1040),
                                   (513, 1280, 1152)])
def test_int8_gemm(q, orc, M, N, K):
    int8_case(q, orc, M, N, K)


def test_int8_gemm_bias(q, orc):
    int8_case(q, orc, 130, 640, 272, with_bias=True)


@pytest.mark.slow
@pytest.mark.parametrize("K,N", [(3072, 12288), (12288, 3072)])
def test_int8_gemm_full_size(q, orc, K, N):
    int8_case(q, orc, 4096, N, K, nrows=256)


# ------------------------------------------------------------------ MXFP8
def mxfp8_case(q, orc, M, N, K, nrows=None):
    lin = inputs.mxfp8_linear(K, N, M=M)
    x, w = lin.make_x(), lin.make_w()
    F, L = q.Fmt, q.Layout
    bx = q.quantize_act(F.MXFP8, x.cuda(), L.MMA)
    bw = q.quantize_weight(F.MXFP8, w.cuda(), L.MMA)
    y = q.gemm(F.MXFP8, F.MXFP8, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"], layout=L.MMA)
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    xs = mma_to_canonical(np_u8(bx["scales"]), M, K // 32)[rows]
    xh = orc.dequant_mxfp8(np_u8(bx["codes"]).reshape(M, K)[rows], xs)
    wh = orc.dequant_mxfp8(np_u8(bw["codes"]).reshape(N, K), mma_to_canonical(np_u8(bw["scales"]), N, K // 32))
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh), x, w, rows=torch.from_numpy(rows))


@pytest.mark.parametrize("M,N,K", [(200, 512, 512), (128, 256, 128), (1, 256, 256), (300, 640, 1152)])
def test_mxfp8_gemm(q, orc, M, N, K):
    mxfp8_case(q, orc, M, N, K)


@pytest.mark.slow
@pytest.mark.parametrize("K,N", [(5120, 13824), (13824, 5120), (5120, 5120)])
def test_mxfp8_gemm_full_size(q, orc, K, N):
    mxfp8_case(q, orc, 20280, N, K, nrows=256)


# ------------------------------------------------------------------ NVFP4
def nvfp4_case(q, orc, M, N, K, nrows=None):
    lin = inputs.mixed_stack(M=M, d=K)[0]
    x = lin.make_x()
    w = inputs.normal_bf16((N, K), 0.02, lin.w_seed)
    F, L = q.Fmt, q.Layout
    bx = q.quantize_act(F.NVFP4, x.cuda(), L.MMA)
    bw = q.quantize_weight(F.NVFP4, w.cuda(), L.MMA)
    y = q.gemm(F.NVFP4, F.NVFP4, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"], layout=L.MMA,
               x_global=bx["global"], w_global=bw["global"])
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    xs = mma_to_canonical(np_u8(bx["scales"]), M, K // 16)[rows]
    xh = orc.dequant_nvfp4(np_u8(bx["codes"]).reshape(M, K // 2)[rows], xs, np_f32(bx["global"])[0])
    wh = orc.dequant_nvfp4(np_u8(bw["codes"]).reshape(N, K // 2), mma_to_canonical(np_u8(bw["scales"]), N, K // 16),
                           np_f32(bw["global"])[0])
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh), x, w, rows=torch.from_numpy(rows))


@pytest.mark.parametrize("M,N,K", [(200, 512, 512), (128, 256, 256), (1, 256, 256), (300, 640, 1280)])
def test_nvfp4_gemm(q, orc, M, N, K):
    nvfp4_case(q, orc, M, N, K)


@pytest.mark.slow
def test_nvfp4_gemm_full_size(q, orc):
    nvfp4_case(q, orc, 32768, 3072, 3072, nrows=256)


# ------------------------------------------------------------------ MXFP4 (W4A4)
def mxfp4_case(q, orc, M, N, K, nrows=None, with_bias=False):
    lin = inputs.mxfp8_linear(K, N, M=M)          # the MXFP8 workload's distributions, W4A4 formats
    x, w = lin.make_x(), lin.make_w()
    F, L = q.Fmt, q.Layout
    bx = q.quantize_act(F.MXFP4, x.cuda(), L.MMA)
    bw = q.quantize_weight(F.MXFP4, w.cuda(), L.MMA)
    bias = inputs.normal_bf16((1, N), 0.05, 79)[0] if with_bias else None
    y = q.gemm(F.MXFP4, F.MXFP4, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"], layout=L.MMA,
               bias=bias.cuda() if with_bias else None)
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    xs = mma_to_canonical(np_u8(bx["scales"]), M, K // 32)[rows]
    xh = orc.dequant_mxfp4(np_u8(bx["codes"]).reshape(M, K // 2)[rows], xs)
    wh = orc.dequant_mxfp4(np_u8(bw["codes"]).reshape(N, K // 2), mma_to_canonical(np_u8(bw["scales"]), N, K // 32))
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh, bias=b), x, w, rows=torch.from_numpy(rows))


@pytest.mark.parametrize("M,N,K", [(200, 512, 512), (128, 256, 256), (1, 256, 768), (300, 640, 1280)])
def test_mxfp4_gemm(q, orc, M, N, K):
    mxfp4_case(q, orc, M, N, K)


def test_mxfp4_gemm_bias(q, orc):
    mxfp4_case(q, orc, 130, 384, 512, with_bias=True)


@pytest.mark.slow
def test_mxfp4_gemm_full_size(q, orc):
    mxfp4_case(q, orc, 20280, 5120, 5120, nrows=256)


# ------------------------------------------------------------------ MXFP4 dual-scale
def mxfp4_dual_case(q, orc, M, N, K, nrows=None, with_bias=False):
    lin = inputs.mxfp8_linear(K, N, M=M)          # the MXFP8 workload's distributions
    x, w = lin.make_x(), lin.make_w()
    F, L = q.Fmt, q.Layout
    bx = q.quantize_act(F.MXFP4_DUAL, x.cuda(), L.MMA)
    bw = q.quantize_weight(F.MXFP4_DUAL, w.cuda(), L.MMA)
    bias = inputs.normal_bf16((1, N), 0.05, 83)[0] if with_bias else None
    y = q.gemm(F.MXFP4_DUAL, F.MXFP4_DUAL, M, N, K, bx["codes"], bx["scales"], bw["codes"], bw["scales"],
               layout=L.MMA, x_global=bx["global"], w_global=bw["global"], bias=bias.cuda() if with_bias else None)
    torch.cuda.synchronize()
    rows = sample_rows(M, nrows or M)
    xs = mma_to_canonical(np_u8(bx["scales"]), M, K // 32)[rows]
    xc = np_f32(bx["global"])[: M * K // 512].reshape(M, K // 512)[rows]
    xh = orc.dequant_mxfp4_dual(np_u8(bx["codes"]).reshape(M, K // 2)[rows], xs, xc)
    wh = orc.dequant_mxfp4_dual(np_u8(bw["codes"]).reshape(N, K // 2), mma_to_canonical(np_u8(bw["scales"]), N, K // 32),
                                np_f32(bw["global"])[: N * K // 512].reshape(N, K // 512))
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    return check(orc, y_np(y)[rows], orc.gemm_ref(xh, wh, bias=b), x, w, rows=torch.from_numpy(rows))


# ragged M and N tiles, one 512-K block, several blocks, K with an odd number of 512 blocks
@pytest.mark.parametrize("M,N,K", [(200, 512, 512), (128, 256, 1024), (1, 256, 1536), (300, 640, 2560),
                                   (513, 1280, 5120)])
def test_mxfp4_dual_gemm(q, orc, M, N, K):
    mxfp4_dual_case(q, orc, M, N, K)


def test_mxfp4_dual_gemm_bias(q, orc):
    mxfp4_dual_case(q, orc, 130, 384, 1024, with_bias=True)


@pytest.mark.slow
def test_mxfp4_dual_gemm_full_size(q, orc):
    mxfp4_dual_case(q, orc, 20280, 5120, 5120, nrows=256)


# ------------------------------------------------------------------ W4A16 decode
def w4a16_case(q, orc, M, K, N, with_bias=False, sym=False):
    lin = inputs.w4a16_linear(M, K, N)
    x, w = lin.make_x(), lin.make_w()
    F = q.Fmt
    wf = F.INT4_G128_SYM if sym else F.INT4_G128_ASYM
    bw = q.quantize_weight(wf, w.cuda())
    xd = x.cuda()
    bias = inputs.normal_bf16((1, N), 0.05, 77)[0] if with_bias else None
    y = q.gemm(wf, F.BF16, M, N, K, xd, None, bw["codes"], bw["scales"], w_zeros=bw["zeros"],
               bias=bias.cuda() if with_bias else None)
    torch.cuda.synchronize()
    wh = orc.dequant_int4_g128(bw["codes"].cpu().numpy().view(np.int32).reshape(K // 8, N),
                               bw["scales"].cpu().numpy().view(np.uint16).reshape(K // 128, N),
                               bw["zeros"].cpu().numpy().view(np.int32).reshape(K // 128, N // 8))
    b = orc.bf16_values(bits(bias)[None, :])[0] if with_bias else None
    return check(orc, y_np(y), orc.gemm_ref(orc.bf16_values(bits(x)), wh, bias=b), x, w)


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (16, 4096, 12288), (64, 12288, 4096), (5, 256, 72),
                                   (100, 512, 256), (200, 1024, 384), (33, 128, 136), (24, 512, 136),
                                   # split-K over clusters of 2, 4, 5, 6 and 7 CTAs (warp-level kernels),
                                   # and the tcgen05 kernel at its 4-way cap
                                   (1, 512, 128), (3, 1024, 256), (7, 1280, 128), (16, 1536, 136), (2, 1792, 72),
                                   (64, 2048, 1024),
                                   # M <= 8 (tokens as the B operand) with clusters of 3 and 6 CTAs, and
                                   # 8 < M <= 16 with 1, 2, 4, 5, 7 and 8
                                   (2, 768, 128), (4, 1536, 256), (9, 256, 72), (12, 512, 136), (10, 1024, 256),
                                   (13, 1280, 128), (11, 1792, 72), (14, 2048, 512)])
def test_w4a16_gemm(q, orc, M, K, N):
    w4a16_case(q, orc, M, K, N)


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (3, 256, 72), (70, 1024, 256)])
def test_w4a16_gemm_bias(q, orc, M, K, N):
    # (1, 4096, 4096) takes the split-K cluster path, (3, 256, 72) a single CTA
    w4a16_case(q, orc, M, K, N, with_bias=True)


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 16, 64])
@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 12288), (12288, 4096)])
def test_w4a16_gemm_all_decode_shapes(q, orc, M, K, N):
    w4a16_case(q, orc, M, K, N)


# the symmetric int4 weights (zero point 8) through the same kernels
@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (16, 4096, 12288), (64, 12288, 4096), (5, 256, 72)])
def test_w4a16_sym_gemm(q, orc, M, K, N):
    w4a16_case(q, orc, M, K, N, sym=True, with_bias=(M == 5))


# ------------------------------------------------------------------ device timeout path
def test_bounded_wait_expires_with_status(q):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = q.qlin_debug_expire_wait(st.data_ptr(), 1000, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == int(q.Status.DEVICE_TIMEOUT)
    # the context is still usable afterwards
    assert float(torch.ones(4, device="cuda").sum()) == 4.0
