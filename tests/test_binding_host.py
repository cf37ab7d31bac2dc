"""The Python binding's own checks, on the CPU with the C entry points stubbed.

The torch helpers hand raw pointers to the library, which trusts the sizes it
is given; so the helpers refuse a buffer smaller than the library's size
query, a non-contiguous one, or a Y of the wrong shape, before any pointer is
handed over.  These tests check both directions: every call pattern that the
GPU tests, smoke() and bench.py make passes the checks, and each kind of
mis-sized argument is refused without reaching the library.
"""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from serving_amax_reduce_gb300 import inputs  # noqa: E402


@pytest.fixture()
def q(monkeypatch):
    from serving_amax_reduce_gb300 import build
    build.build()
    from serving_amax_reduce_gb300 import qlin
    calls = []

    def stub(name):
        def f(*args):
            calls.append(name)
            return 0
        return f

    for name in ("qlin_quantize_weight", "qlin_quantize_act", "qlin_gemm"):
        monkeypatch.setattr(qlin, name, stub(name))
    monkeypatch.setattr(qlin, "device_status", lambda device=None: torch.zeros(1, dtype=torch.int32))
    monkeypatch.setattr(qlin, "_stream", lambda stream=None: 0)
    qlin.calls = calls
    return qlin


PAIRS = [
    # w_fmt, x_fmt, layout, (M, N, K) as the GPU tests use them
    ("FP8_TENSOR", "FP8_TENSOR", "CANONICAL", (333, 1040, 1040)),
    ("FP8_BLOCK128", "FP8_TOKEN", "CANONICAL", (513, 1280, 1152)),
    ("FP8_BLOCK128", "FP8_GROUP128", "CANONICAL", (130, 640, 256)),
    ("MXFP8", "MXFP8", "MMA", (300, 640, 1152)),
    ("MXFP4", "MXFP4", "MMA", (300, 640, 1280)),
    ("NVFP4", "NVFP4", "MMA", (300, 640, 1280)),
    ("INT8_ROW", "INT8_ROW", "CANONICAL", (300, 640, 1040)),
    ("FP8_TENSOR", "BF16", "CANONICAL", (77, 640, 1040)),
    ("INT4_G128_ASYM", "BF16", "CANONICAL", (33, 136, 128)),
    ("INT4_G128_SYM", "BF16", "CANONICAL", (16, 4096, 4096)),
    ("MXFP4_DUAL", "MXFP4_DUAL", "MMA", (300, 640, 2560)),
]


def operands(q, wname, xname, lname, M, N, K):
    wf, xf, lay = q.Fmt[wname], q.Fmt[xname], q.Layout[lname]
    x = inputs.normal_bf16((M, K), 1.0, 1)
    w = inputs.normal_bf16((N, K), 0.02, 2)
    bw = q.quantize_weight(wf, w, lay)
    kw = {"layout": lay, "bias": inputs.normal_bf16((1, N), 0.05, 3)[0]}
    if xf == q.Fmt.BF16:
        xa, xs = x, None
    else:
        bx = q.quantize_act(xf, x, lay)
        xa, xs = bx["codes"], bx["scales"]
        kw["x_global"] = bx.get("global")
    kw["w_global"] = bw.get("global")
    kw["w_zeros"] = bw.get("zeros")
    return (wf, xf, M, N, K, xa, xs, bw["codes"], bw["scales"]), kw


@pytest.mark.parametrize("wname,xname,lname,shape", PAIRS)
def test_every_pair_as_called_passes_the_checks(q, wname, xname, lname, shape):
    args, kw = operands(q, wname, xname, lname, *shape)
    M, N = shape[0], shape[1]
    y = q.gemm(*args, **kw)
    assert tuple(y.shape) == (M, N) and q.calls[-1] == "qlin_gemm"
    # and into a strided Y (ldy = N + 8), as the guard-band test does
    big = torch.empty(M + 2, N + 8, dtype=torch.bfloat16)
    q.gemm(*args, y=big[1:M + 1, :N], **kw)
    # and the quantizers into caller buffers of exactly the queried size
    fmt, lay = args[0], kw["layout"]
    w = inputs.normal_bf16((shape[1], shape[2]), 0.02, 4)
    b = q.alloc_quant(fmt, shape[1], shape[2], lay, "cpu")
    q.quantize_weight(fmt, w, lay, bufs=b)


def test_bench_jobs_pass_the_checks(q):
    import bench
    lins = [inputs.fp8_tensor_linear(), inputs.w4a16_linear(16, 4096, 4096), inputs.w4a16_linear(64, 4096, 4096),
            inputs.fp8_block_linear(1, 3072, 12288, M=256), inputs.mxfp8_linear(5120, 5120, M=200),
            inputs.mixed_stack(M=256)[0], inputs.mixed_stack(M=256)[4], inputs.mxfp4_linear(5120, 5120, M=200),
            inputs.fp8_group_linear(3072, 12288, M=256), inputs.int8_linear(3072, 12288, M=256),
            inputs.fp8_tensor_fused_linear()]
    for lin in lins:
        j = bench.Job("g", lin, "cpu", q)
        j.quant_w()
        j.quant_x()
        j.gemm()
    assert q.calls.count("qlin_gemm") == len(lins)


def test_mis_sized_arguments_are_refused_before_the_library(q):
    F, L = q.Fmt, q.Layout
    args, kw = operands(q, "FP8_BLOCK128", "FP8_TOKEN", "CANONICAL", 200, 512, 384)
    wf, xf, M, N, K, xa, xs, wc, ws = args
    n = len(q.calls)
    bad = [
        dict(y=torch.empty(M, N + 1, dtype=torch.bfloat16)),                    # wrong shape
        dict(y=torch.empty(N, M, dtype=torch.bfloat16).t()),                     # column stride != 1
        dict(y=torch.empty(M, N, dtype=torch.float32)),                          # wrong dtype
        dict(bias=torch.zeros(N - 1, dtype=torch.bfloat16)),                     # short bias
    ]
    for extra in bad:
        with pytest.raises(ValueError):
            q.gemm(*args, **{**kw, **extra})
    with pytest.raises(ValueError):
        q.gemm(wf, xf, M, N, K, xa[:-1], xs, wc, ws, **kw)                       # short X codes
    with pytest.raises(ValueError):
        q.gemm(wf, xf, M, N, K, xa, xs[:-1], wc, ws, **kw)                       # short X scales
    with pytest.raises(ValueError):
        q.gemm(wf, xf, M, N, K, xa, xs, wc[::2], ws, **kw)                       # non-contiguous W codes
    with pytest.raises(ValueError):
        q.gemm(wf, xf, M, N, K, xa, None, wc, ws, **kw)                          # missing X scales
    x = inputs.normal_bf16((64, 256), 1.0, 5)
    with pytest.raises(ValueError):                                             # BF16 X of the wrong shape
        q.gemm(F.INT4_G128_ASYM, F.BF16, 64, 256, 256, x[:, :128], None, wc, ws, w_zeros=wc)
    b = q.alloc_quant(F.NVFP4, 64, 256, L.MMA, "cpu")
    for key, short in (("codes", b["codes"][:-1]), ("scales", b["scales"][:-16]), ("global", None),
                       ("workspace", None)):
        with pytest.raises(ValueError):
            q.quantize_act(F.NVFP4, x, L.MMA, bufs={**b, key: short})
    assert len(q.calls) == n                                                    # the library was never called
