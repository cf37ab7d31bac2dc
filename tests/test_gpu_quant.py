"""GPU quantizers against the CPU oracle: codes and scales bit for bit."""
import numpy as np
import pytest
import torch

from gpu_util import bits, edge_bf16, np_f32, np_u8, require_gpu
from layouts import mma_padding_rows, mma_to_canonical
from serving_amax_reduce_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def run(q, fmt, x, layout=None, weight=False):
    L = q.Layout.CANONICAL if layout is None else layout
    xd = x.cuda()
    b = (q.quantize_weight if weight else q.quantize_act)(fmt, xd, L)
    torch.cuda.synchronize()
    return b


def refused_before_launch(q, fmt, x):
    """The tensor-core scale tiling needs whole 4-scale chunks along K; other K
    are refused with INVALID_ARG before any launch (no output is written)."""
    with pytest.raises(q.QlinError) as e:
        run(q, fmt, x, q.Layout.MMA)
    assert e.value.status == q.Status.INVALID_ARG
    assert q.read_device_status() == 0


def make(kind, rows, K, seed):
    if kind == "outlier":
        return inputs.outlier_channel_bf16(rows, K, seed)
    if kind == "edge":
        return edge_bf16(rows, K, seed)
    return inputs.normal_bf16((rows, K), 0.02, seed)


SHAPES_ROW = [(1, 1024), (200, 3072), (64, 12288), (3, 24576), (129, 1040), (37, 8),
              # with the above, every register-resident (threads, vectors per thread) variant the
              # per-row kernels dispatch to, and the first K past them
              (9, 4096), (9, 5120), (9, 6144), (9, 7168), (9, 8192), (9, 9216), (9, 13312), (9, 16384),
              (9, 16392)]


@pytest.mark.parametrize("rows,K", SHAPES_ROW)
@pytest.mark.parametrize("kind", ["outlier", "edge"])
def test_fp8_token(q, orc, rows, K, kind):
    x = make(kind, rows, K, rows + K)
    b = run(q, q.Fmt.FP8_TOKEN, x)
    codes, scales = orc.quant_fp8_token(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K), codes)
    assert np.array_equal(np_f32(b["scales"])[:rows].view(np.uint32), scales.view(np.uint32))


def int8_ties(rows, K, seed):
    """Rows whose amax is 127 * 2^k, so that 127/amax = 2^-k exactly and
    every x * 127/amax is a half-integer: each odd one is a rounding tie."""
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(-8, 9, (rows, 1), generator=g).float()
    n = torch.randint(-254, 255, (rows, K), generator=g).float()
    n[:, 0] = 254
    return ((n / 2) * torch.pow(2.0, k)).to(torch.bfloat16)


@pytest.mark.parametrize("rows,K", SHAPES_ROW)
@pytest.mark.parametrize("kind", ["outlier", "edge", "ties"])
@pytest.mark.parametrize("weight", [False, True])
def test_int8_row(q, orc, rows, K, kind, weight):
    x = int8_ties(rows, K, rows + 3 * K) if kind == "ties" else make(kind, rows, K, 5 * rows + K)
    b = run(q, q.Fmt.INT8_ROW, x, weight=weight)
    codes, scales = orc.quant_int8_row(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K).view(np.int8), codes)
    assert np.array_equal(np_f32(b["scales"])[:rows].view(np.uint32), scales.view(np.uint32))


@pytest.mark.parametrize("rows,K", [(128, 1024), (1024, 1024), (333, 520), (4096, 4096), (1, 8)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
def test_fp8_tensor(q, orc, rows, K, kind):
    x = make(kind, rows, K, 7 * rows + K)
    b = run(q, q.Fmt.FP8_TENSOR, x)
    codes, s = orc.quant_fp8_tensor(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K), codes)
    assert np_f32(b["scales"])[0].view(np.uint32) == np.float32(s).view(np.uint32)


@pytest.mark.parametrize("rows,K", [(128, 128), (256, 384), (1024, 3072), (12288, 3072)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
def test_fp8_block128(q, orc, rows, K, kind):
    x = make(kind, rows, K, 3 * rows + K)
    b = run(q, q.Fmt.FP8_BLOCK128, x, weight=True)
    codes, s = orc.quant_fp8_block128(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K), codes)
    assert np.array_equal(np_f32(b["scales"]).reshape(s.shape).view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("rows,K", [(1, 128), (200, 5120), (128, 13824), (77, 96)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
@pytest.mark.parametrize("mma", [False, True])
def test_mxfp8(q, orc, rows, K, kind, mma):
    x = make(kind, rows, K, 5 * rows + K) if kind == "edge" else inputs.normal_bf16((rows, K), 1.0, rows + K)
    if mma and K % 128:
        refused_before_launch(q, q.Fmt.MXFP8, x)     # the tiling packs 4 scales (128 K) per chunk
        return
    b = run(q, q.Fmt.MXFP8, x, q.Layout.MMA if mma else None)
    codes, sc = orc.quant_mxfp8(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K), codes)
    got = np_u8(b["scales"])
    if mma:
        assert np.array_equal(mma_to_canonical(got, rows, K // 32), sc)
        assert not mma_padding_rows(got, rows, K // 32).any()
    else:
        assert np.array_equal(got[: rows * K // 32].reshape(rows, K // 32), sc)


@pytest.mark.parametrize("rows,K", [(1, 64), (200, 3072), (300, 12288), (5, 80)])
@pytest.mark.parametrize("kind", ["outlier", "edge"])
@pytest.mark.parametrize("mma", [False, True])
def test_nvfp4(q, orc, rows, K, kind, mma):
    x = make(kind, rows, K, 11 * rows + K)
    if mma and K % 64:
        refused_before_launch(q, q.Fmt.NVFP4, x)     # the tiling packs 4 scales (64 K) per chunk
        return
    b = run(q, q.Fmt.NVFP4, x, q.Layout.MMA if mma else None)
    packed, sc, g = orc.quant_nvfp4(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K // 2), packed)
    assert np_f32(b["global"])[0].view(np.uint32) == np.float32(g).view(np.uint32)
    got = np_u8(b["scales"])
    if mma:
        assert np.array_equal(mma_to_canonical(got, rows, K // 16), sc)
        assert not mma_padding_rows(got, rows, K // 16).any()
    else:
        assert np.array_equal(got[: rows * K // 16].reshape(rows, K // 16), sc)


@pytest.mark.parametrize("rows,K", [(1, 128), (200, 3072), (300, 12288), (7, 384)])
@pytest.mark.parametrize("kind", ["outlier", "edge"])
def test_fp8_group128(q, orc, rows, K, kind):
    x = make(kind, rows, K, 17 * rows + K)
    b = run(q, q.Fmt.FP8_GROUP128, x)
    codes, s = orc.quant_fp8_group128(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K), codes)
    assert np.array_equal(np_f32(b["scales"]).reshape(rows, K // 128).view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("rows,K", [(1, 128), (200, 5120), (128, 13824), (77, 96)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
@pytest.mark.parametrize("mma", [False, True])
def test_mxfp4(q, orc, rows, K, kind, mma):
    x = make(kind, rows, K, 7 * rows + K) if kind == "edge" else inputs.normal_bf16((rows, K), 1.0, rows + 2 * K)
    if mma and K % 128:
        refused_before_launch(q, q.Fmt.MXFP4, x)
        return
    b = run(q, q.Fmt.MXFP4, x, q.Layout.MMA if mma else None)
    packed, sc = orc.quant_mxfp4(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K // 2), packed)
    got = np_u8(b["scales"])
    if mma:
        assert np.array_equal(mma_to_canonical(got, rows, K // 32), sc)
        assert not mma_padding_rows(got, rows, K // 32).any()
    else:
        assert np.array_equal(got[: rows * K // 32].reshape(rows, K // 32), sc)


@pytest.mark.parametrize("rows,K", [(1, 512), (200, 5120), (130, 13824), (77, 1536), (3, 1024)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
@pytest.mark.parametrize("mma", [False, True])
def test_mxfp4_dual(q, orc, rows, K, kind, mma):
    x = make(kind, rows, K, 9 * rows + K) if kind == "edge" else inputs.normal_bf16((rows, K), 1.0, rows + 3 * K)
    b = run(q, q.Fmt.MXFP4_DUAL, x, q.Layout.MMA if mma else None)
    packed, sc, coarse = orc.quant_mxfp4_dual(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(rows, K // 2), packed)
    assert np.array_equal(np_f32(b["global"])[: rows * K // 512].reshape(rows, K // 512).view(np.uint32),
                          coarse.view(np.uint32))
    got = np_u8(b["scales"])
    if mma:
        assert np.array_equal(mma_to_canonical(got, rows, K // 32), sc)
        assert not mma_padding_rows(got, rows, K // 32).any()
    else:
        assert np.array_equal(got[: rows * K // 32].reshape(rows, K // 32), sc)


@pytest.mark.parametrize("N,K", [(72, 256), (4096, 4096), (12288, 4096), (64, 12288)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
def test_int4_g128(q, orc, N, K, kind):
    w = make(kind, N, K, 13 * N + K)
    b = run(q, q.Fmt.INT4_G128_ASYM, w, weight=True)
    qw, sc, qz = orc.quant_int4_g128(bits(w))
    assert np.array_equal(b["codes"].cpu().numpy().view(np.int32).reshape(K // 8, N), qw)
    assert np.array_equal(b["scales"].cpu().numpy().view(np.uint16).reshape(K // 128, N), sc)
    assert np.array_equal(b["zeros"].cpu().numpy().view(np.int32).reshape(K // 128, N // 8), qz)


@pytest.mark.parametrize("N,K", [(72, 256), (4096, 4096), (12288, 4096), (64, 12288)])
@pytest.mark.parametrize("kind", ["normal", "edge"])
def test_int4_g128_sym(q, orc, N, K, kind):
    w = make(kind, N, K, 19 * N + K)
    b = run(q, q.Fmt.INT4_G128_SYM, w, weight=True)
    qw, sc, qz = orc.quant_int4_g128_sym(bits(w))
    assert np.array_equal(b["codes"].cpu().numpy().view(np.int32).reshape(K // 8, N), qw)
    assert np.array_equal(b["scales"].cpu().numpy().view(np.uint16).reshape(K // 128, N), sc)
    assert np.array_equal(b["zeros"].cpu().numpy().view(np.int32).reshape(K // 128, N // 8), qz)


def test_int4_sym_half_step_groups(q, orc):
    """Symmetric groups whose x * fl(1/s) sits next to rounding ties: the
    kernel's codes, scales and zero points equal the oracle's."""
    from hard_cases import int4_sym_half_step_weight
    w = int4_sym_half_step_weight()
    N, K = w.shape
    b = run(q, q.Fmt.INT4_G128_SYM, torch.from_numpy(w.view(np.int16)).view(torch.bfloat16), weight=True)
    qw, sc, qz = orc.quant_int4_g128_sym(w)
    assert np.array_equal(b["codes"].cpu().numpy().view(np.int32).reshape(K // 8, N), qw)
    assert np.array_equal(b["scales"].cpu().numpy().view(np.uint16).reshape(K // 128, N), sc)
    assert np.array_equal(b["zeros"].cpu().numpy().view(np.int32).reshape(K // 128, N // 8), qz)


def test_row_amax_sweep(q, orc):
    """Rows led by their amax with every bf16 value below it: the per-row
    encoders' products x * fl(c / amax) meet values next to rounding ties; the
    INT8 and per-token FP8 kernels equal the oracle on every row."""
    from hard_cases import row_amax_sweep
    rows = row_amax_sweep()
    x = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16)
    for fmt, ref in [(q.Fmt.INT8_ROW, orc.quant_int8_row), (q.Fmt.FP8_TOKEN, orc.quant_fp8_token)]:
        b = run(q, fmt, x)
        codes, s = ref(rows)
        assert np.array_equal(np_u8(b["codes"]).reshape(rows.shape), codes.view(np.uint8)), fmt
        assert np.array_equal(np_f32(b["scales"]).view(np.uint32), np.asarray(s, np.float32).view(np.uint32)), fmt


def test_int4_half_step_groups(q, orc):
    """Groups whose values x * fl(1/s) and -min * fl(1/s) sit next to rounding
    ties: the kernel's codes, scales and zero points equal the oracle's."""
    from hard_cases import int4_half_step_weight
    w = int4_half_step_weight()
    N, K = w.shape
    b = run(q, q.Fmt.INT4_G128_ASYM, torch.from_numpy(w.view(np.int16)).view(torch.bfloat16), weight=True)
    qw, sc, qz = orc.quant_int4_g128(w)
    assert np.array_equal(b["codes"].cpu().numpy().view(np.int32).reshape(K // 8, N), qw)
    assert np.array_equal(b["scales"].cpu().numpy().view(np.uint16).reshape(K // 128, N), sc)
    assert np.array_equal(b["zeros"].cpu().numpy().view(np.int32).reshape(K // 128, N // 8), qz)


def test_int4_scale_tie_groups(q, orc):
    """Groups whose (max - min) / 15 lies on a bf16 rounding midpoint or a few
    fp32 ulps off one: the kernel's scales (and codes and zero points) equal
    the oracle's, which rounds the range to nearest with ties to even."""
    from hard_cases import int4_scale_tie_weight
    w = int4_scale_tie_weight()
    N, K = w.shape
    b = run(q, q.Fmt.INT4_G128_ASYM, torch.from_numpy(w.view(np.int16)).view(torch.bfloat16), weight=True)
    qw, sc, qz = orc.quant_int4_g128(w)
    assert np.array_equal(b["scales"].cpu().numpy().view(np.uint16).reshape(K // 128, N), sc)
    assert np.array_equal(b["codes"].cpu().numpy().view(np.int32).reshape(K // 8, N), qw)
    assert np.array_equal(b["zeros"].cpu().numpy().view(np.int32).reshape(K // 128, N // 8), qz)


def test_fp8_reciprocal_form_rows(q, orc):
    """Rows on which x * fl(448 / amax) and x / fl(amax / 448) round to
    different codes: the kernels follow the oracle (the reciprocal form) bit
    for bit, per token, per 1 x 128 group and per tensor."""
    from hard_cases import fp8_reciprocal_candidates, rows_of_pairs
    rows = rows_of_pairs(fp8_reciprocal_candidates([orc.dec_e4m3(c) for c in range(256)]), 128)
    x = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16)
    for fmt, ref in [(q.Fmt.FP8_TOKEN, orc.quant_fp8_token), (q.Fmt.FP8_GROUP128, orc.quant_fp8_group128)]:
        b = run(q, fmt, x)
        codes, s = ref(rows)
        s = np.asarray(s, np.float32)
        assert np.array_equal(np_u8(b["codes"]).reshape(rows.shape), codes)
        assert np.array_equal(np_f32(b["scales"]).reshape(s.shape).view(np.uint32), s.view(np.uint32))
    from hard_cases import tiles_of_pairs
    pairs = fp8_reciprocal_candidates([orc.dec_e4m3(c) for c in range(256)])
    tiles = tiles_of_pairs(pairs[::max(1, len(pairs) // 64)])
    b = run(q, q.Fmt.FP8_BLOCK128, torch.from_numpy(tiles.view(np.int16)).view(torch.bfloat16), weight=True)
    codes, s = orc.quant_fp8_block128(tiles)
    assert np.array_equal(np_u8(b["codes"]).reshape(tiles.shape), codes)
    assert np.array_equal(np_f32(b["scales"]).reshape(s.shape).view(np.uint32), s.view(np.uint32))
    for i in range(0, len(rows), max(1, len(rows) // 16)):
        b = run(q, q.Fmt.FP8_TENSOR, x[i:i + 1])
        codes, s = orc.quant_fp8_tensor(rows[i:i + 1])
        assert np.array_equal(np_u8(b["codes"]).reshape(1, 128), codes)
        assert np_f32(b["scales"])[0].view(np.uint32) == np.float32(s).view(np.uint32)


def test_nvfp4_step_sweeps(q, orc):
    """Sweeps of bf16 blocks under fixed tensor amaxes, which put block and
    element values within an ulp of code midpoints at both NVFP4 steps: the
    kernel's codes, block scales and global scale equal the oracle's."""
    from hard_cases import NVFP4_AMAXES, nvfp4_block_sweep
    for A in NVFP4_AMAXES:
        rows = nvfp4_block_sweep(A)
        R, K = rows.shape
        b = run(q, q.Fmt.NVFP4, torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16))
        packed, sc, g = orc.quant_nvfp4(rows)
        assert np.array_equal(np_u8(b["codes"]).reshape(R, K // 2), packed), A
        assert np.array_equal(np_u8(b["scales"])[: R * K // 16].reshape(R, K // 16), sc), A
        assert np_f32(b["global"])[0].view(np.uint32) == np.float32(g).view(np.uint32), A


def test_leading_dimension_is_honoured(q, orc):
    """A strided view (ld > K) quantizes exactly like its contiguous copy."""
    big = inputs.outlier_channel_bf16(96, 4096, 5)
    x = big[:, 1024:3072]
    xd = big.cuda()[:, 1024:3072]
    for fmt, ref in [(q.Fmt.FP8_TOKEN, orc.quant_fp8_token), (q.Fmt.MXFP8, orc.quant_mxfp8)]:
        b = q.quantize_act(fmt, xd)
        torch.cuda.synchronize()
        codes, sc = ref(bits(x.contiguous()))
        assert np.array_equal(np_u8(b["codes"]).reshape(96, 2048), codes)


STRIDED = [  # format name, weight side, scale layout
    ("FP8_TENSOR", False, "CANONICAL"), ("FP8_TOKEN", False, "CANONICAL"), ("FP8_GROUP128", False, "CANONICAL"),
    ("INT8_ROW", False, "CANONICAL"), ("MXFP8", False, "MMA"), ("MXFP4", False, "MMA"), ("NVFP4", False, "MMA"),
    ("MXFP4_DUAL", False, "MMA"), ("FP8_BLOCK128", True, "CANONICAL"), ("INT4_G128_ASYM", True, "CANONICAL"),
    ("INT4_G128_SYM", True, "CANONICAL"), ("MXFP8", True, "CANONICAL"), ("NVFP4", True, "CANONICAL"),
]


@pytest.mark.parametrize("name,weight,lname", STRIDED, ids=[f"{n}-{'w' if w else 'x'}-{l}" for n, w, l in STRIDED])
def test_every_quantizer_honours_the_leading_dimension(q, name, weight, lname):
    """Every format, on a strided view (ld = 4096 > K = 2048, starting 1024 columns in) of a
    tensor with a large-magnitude band outside the view: codes, scales, zero points and global
    scales equal, bit for bit, those of the contiguous copy."""
    big = inputs.outlier_channel_bf16(128, 4096, 7)
    big[:, :1024] *= 1000                                  # outside the view; must not leak into its amax
    view = big.cuda()[:, 1024:3072]
    assert view.stride(0) == 4096 and not view.is_contiguous()
    fn = q.quantize_weight if weight else q.quantize_act
    fmt, lay = q.Fmt[name], q.Layout[lname]
    a = fn(fmt, view, lay)
    b = fn(fmt, view.contiguous(), lay)
    torch.cuda.synchronize()
    assert set(a) == set(b)
    for key in ("codes", "scales", "zeros", "global"):     # the outputs (the workspace is scratch)
        if a.get(key) is not None:
            assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


@pytest.mark.slow
def test_full_size_activation_quantizers(q, orc):
    """The workloads' largest activations: MXFP8 X [20280, 13824] and NVFP4 X
    [32768, 3072] (per-tensor amax over 100 M elements), compared in full."""
    x = inputs.mxfp8_linear(13824, 5120).make_x()
    b = run(q, q.Fmt.MXFP8, x, q.Layout.MMA)
    codes, sc = orc.quant_mxfp8(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(codes.shape), codes)
    assert np.array_equal(mma_to_canonical(np_u8(b["scales"]), x.shape[0], x.shape[1] // 32), sc)
    del b, codes, sc
    x = inputs.mixed_stack()[0].make_x()
    b = run(q, q.Fmt.NVFP4, x, q.Layout.MMA)
    packed, sc, g = orc.quant_nvfp4(bits(x))
    assert np.array_equal(np_u8(b["codes"]).reshape(packed.shape), packed)
    assert np.array_equal(mma_to_canonical(np_u8(b["scales"]), x.shape[0], x.shape[1] // 16), sc)
    assert np_f32(b["global"])[0] == g
