"""Guard bands: every library call writes its own outputs and nothing else.

Each quantizer output (codes, scales, zero points, global scale) is placed
between two 512-byte guard bands filled with a byte pattern.  Each GEMM
writes Y into a pattern-filled matrix with one guard row above, one below,
and 8 padding columns per row (ldy = N + 8).  After the call the guards and
the padding must still hold the pattern, and the outputs must equal, byte
for byte, those of the same call on exact-size buffers (whose agreement with
the oracle the other GPU tests establish).  The shapes have ragged row and
column tails, so the predicated stores at the edges are exercised.
"""
import pytest
import torch

from serving_amax_reduce_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 512               # bytes; keeps the 16-byte alignment of the buffer between
PATTERN8 = 0xA5
PATTERN16 = 0x5A5A


def sync():
    torch.cuda.synchronize()


@pytest.fixture(scope="module")
def q():
    from gpu_util import require_gpu
    return require_gpu()


def guarded_like(t: torch.Tensor):
    """(raw, inner): inner has t's dtype and size and sits between two guard bands of raw."""
    nbytes = t.numel() * t.element_size()
    raw = torch.full((GUARD + nbytes + GUARD,), PATTERN8, dtype=torch.uint8, device=t.device)
    return raw, raw[GUARD:GUARD + nbytes].view(t.dtype)


def guards_intact(raw: torch.Tensor) -> bool:
    return bool((raw[:GUARD] == PATTERN8).all()) and bool((raw[-GUARD:] == PATTERN8).all())


QUANT_CASES = [
    # format, scale layout, rows, K
    ("FP8_TENSOR", "CANONICAL", 333, 1024),
    ("FP8_TOKEN", "CANONICAL", 333, 1040),
    ("FP8_TOKEN", "CANONICAL", 3, 20480),          # rows longer than the register-resident kernel takes
    ("FP8_BLOCK128", "CANONICAL", 256, 384),
    ("FP8_GROUP128", "CANONICAL", 333, 384),
    ("MXFP8", "CANONICAL", 333, 512),
    ("MXFP8", "MMA", 333, 512),                     # rows padded to 384 in the scale tiling
    ("MXFP4", "MMA", 333, 512),
    ("NVFP4", "CANONICAL", 333, 512),
    ("NVFP4", "MMA", 333, 512),
    ("INT8_ROW", "CANONICAL", 333, 1040),
    ("INT8_ROW", "CANONICAL", 3, 20480),
    ("INT4_G128_ASYM", "CANONICAL", 200, 1024),
    ("INT4_G128_SYM", "CANONICAL", 200, 1024),
    ("MXFP4_DUAL", "CANONICAL", 333, 1536),
    ("MXFP4_DUAL", "MMA", 333, 1536),
]


@pytest.mark.parametrize("fmt,layout,rows,K", QUANT_CASES)
def test_quantizer_writes_only_its_outputs(q, fmt, layout, rows, K):
    f, lay = q.Fmt[fmt], q.Layout[layout]
    quant = q.quantize_weight if f in (q.Fmt.INT4_G128_ASYM, q.Fmt.INT4_G128_SYM) else q.quantize_act
    x = inputs.normal_bf16((rows, K), 1.0, 91).to(DEV)
    ref = quant(f, x, lay)
    bufs, raws = dict(ref), {}
    for key in ("codes", "scales", "zeros", "global"):
        if ref.get(key) is not None:
            raws[key], bufs[key] = guarded_like(ref[key])
    quant(f, x, lay, bufs=bufs)
    sync()
    assert q.read_device_status() == 0
    for key, raw in raws.items():
        assert guards_intact(raw), f"{key}: a write outside the buffer"
        assert torch.equal(bufs[key].view(torch.uint8), ref[key].view(torch.uint8)), f"{key} differs"


def test_noalloc_quantizer_writes_only_its_outputs(q):
    rows, K = 333, 1040
    x = inputs.normal_bf16((rows, K), 1.0, 92).to(DEV)
    ref = q.quantize_act(q.Fmt.FP8_TENSOR, x)
    raw_c, codes = guarded_like(ref["codes"])
    raw_s, scale = guarded_like(ref["scales"])
    rc = q.qlin_quantize_fp8_tensor_noalloc(x.data_ptr(), rows, K, x.stride(0), codes.data_ptr(), scale.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    sync()
    assert guards_intact(raw_c) and guards_intact(raw_s)
    assert torch.equal(codes, ref["codes"]) and torch.equal(scale.view(torch.uint8), ref["scales"].view(torch.uint8))


PAIRS = {
    # name: weight format, activation format, scale layout
    "fp8_tensor": ("FP8_TENSOR", "FP8_TENSOR", "CANONICAL"),
    "fp8_block_token": ("FP8_BLOCK128", "FP8_TOKEN", "CANONICAL"),
    "fp8_block_group128": ("FP8_BLOCK128", "FP8_GROUP128", "CANONICAL"),
    "mxfp8": ("MXFP8", "MXFP8", "MMA"),
    "mxfp4": ("MXFP4", "MXFP4", "MMA"),
    "mxfp4_dual": ("MXFP4_DUAL", "MXFP4_DUAL", "MMA"),
    "nvfp4": ("NVFP4", "NVFP4", "MMA"),
    "int8": ("INT8_ROW", "INT8_ROW", "CANONICAL"),
    "fp8_tensor_fused_x": ("FP8_TENSOR", "BF16", "CANONICAL"),
    "w4a16": ("INT4_G128_ASYM", "BF16", "CANONICAL"),
}

GEMM_CASES = [
    # pair, M, N, K
    ("fp8_tensor", 200, 520, 384),
    ("fp8_block_token", 130, 640, 256),
    ("fp8_block_group128", 130, 640, 256),
    ("mxfp8", 300, 640, 512),
    ("mxfp4", 130, 384, 512),
    ("mxfp4_dual", 130, 384, 1024),
    ("nvfp4", 130, 384, 512),
    ("int8", 130, 640, 272),
    ("fp8_tensor_fused_x", 77, 640, 1040),
    ("w4a16", 1, 4096, 4096),        # warp-level kernel, split-K over a cluster
    ("w4a16", 5, 72, 256),           # warp-level kernel, one CTA, ragged channel tile
    ("w4a16", 70, 256, 1024),        # tcgen05 kernel, ragged token tile
]


def gemm_operands(q, name, M, N, K):
    wname, xname, lname = PAIRS[name]
    wf, xf, lay = q.Fmt[wname], q.Fmt[xname], q.Layout[lname]
    x = inputs.normal_bf16((M, K), 1.0, 93).to(DEV)
    w = inputs.normal_bf16((N, K), 0.02, 94).to(DEV)
    bias = inputs.normal_bf16((1, N), 0.05, 95)[0].to(DEV)
    bw = q.quantize_weight(wf, w, lay)
    kw = {"layout": lay, "bias": bias}
    if xf == q.Fmt.BF16:
        xa, xs = x, None
    else:
        bx = q.quantize_act(xf, x, lay)
        xa, xs = bx["codes"], bx["scales"]
        if xf in (q.Fmt.NVFP4, q.Fmt.MXFP4_DUAL):
            kw["x_global"] = bx["global"]
    if wf in (q.Fmt.NVFP4, q.Fmt.MXFP4_DUAL):
        kw["w_global"] = bw["global"]
    if wf in (q.Fmt.INT4_G128_ASYM, q.Fmt.INT4_G128_SYM):
        kw["w_zeros"] = bw["zeros"]
    return (wf, xf, M, N, K, xa, xs, bw["codes"], bw["scales"]), kw


@pytest.mark.parametrize("name,M,N,K", GEMM_CASES)
def test_gemm_writes_only_y(q, name, M, N, K):
    args, kw = gemm_operands(q, name, M, N, K)
    y_ref = q.gemm(*args, **kw)
    pad = 8                                               # keeps ldy * 2 bytes a multiple of 16
    y_big = torch.full((M + 2, N + pad), PATTERN16, dtype=torch.int16, device=DEV)
    y = y_big.view(torch.bfloat16)[1:M + 1, :N]
    assert y.stride(0) == N + pad
    q.gemm(*args, y=y, **kw)
    sync()
    assert q.read_device_status() == 0
    assert bool((y_big[0] == PATTERN16).all()), "a write above Y"
    assert bool((y_big[M + 1] == PATTERN16).all()), "a write below Y"
    assert bool((y_big[1:M + 1, N:] == PATTERN16).all()), "a write into the row padding"
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), "strided Y differs"
