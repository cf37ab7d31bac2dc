"""Host-side checks of the C-ABI library: it builds for sm_103a, loads without
a GPU, exports every entry point include/qlin.h declares, answers size
queries, and rejects bad arguments before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    from serving_amax_reduce_gb300 import build
    build.build()
    from serving_amax_reduce_gb300 import qlin
    return qlin


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qlin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(q):
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(q.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(q):
    assert "sm_103a" in q.qlin_version()
    assert q.qlin_last_cuda_error() == 0
    for s in q.Status:
        assert q.qlin_status_string(s)


def test_size_queries(q):
    F, L = q.Fmt, q.Layout
    assert q.qlin_codes_bytes(F.FP8_TOKEN, 20280, 5120) == 20280 * 5120
    assert q.qlin_codes_bytes(F.NVFP4, 32768, 3072) == 32768 * 1536
    assert q.qlin_codes_bytes(F.INT4_G128_ASYM, 4096, 12288) == 12288 // 8 * 4096 * 4
    assert q.qlin_scales_bytes(F.FP8_TENSOR, L.CANONICAL, 128, 1024) == 4
    assert q.qlin_scales_bytes(F.FP8_BLOCK128, L.CANONICAL, 12288, 3072) == 96 * 24 * 4
    assert q.qlin_scales_bytes(F.MXFP8, L.CANONICAL, 20280, 5120) == 20280 * 160
    assert q.qlin_scales_bytes(F.MXFP8, L.MMA, 20280, 5120) == 20352 * 160
    assert q.qlin_scales_bytes(F.NVFP4, L.MMA, 200, 3072) == 256 * 192
    assert q.qlin_scales_bytes(F.INT4_G128_ASYM, L.CANONICAL, 4096, 12288) == 96 * 4096 * 2
    assert q.qlin_zeros_bytes(F.INT4_G128_ASYM, 4096, 12288) == 96 * 512 * 4
    assert q.qlin_zeros_bytes(F.FP8_TOKEN, 4096, 12288) == 0
    assert q.qlin_quant_workspace_bytes(F.FP8_TENSOR, 128, 1024) > 0
    assert q.qlin_quant_workspace_bytes(F.FP8_TOKEN, 128, 1024) == 0
    # MXFP4: E2M1 codes two per byte, one E8M0 byte per 32, no workspace
    assert q.qlin_codes_bytes(F.MXFP4, 20280, 5120) == 20280 * 2560
    assert q.qlin_scales_bytes(F.MXFP4, L.CANONICAL, 20280, 5120) == 20280 * 160
    assert q.qlin_scales_bytes(F.MXFP4, L.MMA, 20280, 5120) == 20352 * 160
    assert q.qlin_quant_workspace_bytes(F.MXFP4, 20280, 5120) == 0
    # FP8 1 x 128 groups: one float per row and 128 K
    assert q.qlin_codes_bytes(F.FP8_GROUP128, 4096, 3072) == 4096 * 3072
    assert q.qlin_scales_bytes(F.FP8_GROUP128, L.CANONICAL, 4096, 3072) == 4096 * 24 * 4
    # INT8 per row: one byte per code, one float per row, no workspace
    assert q.qlin_codes_bytes(F.INT8_ROW, 4096, 3072) == 4096 * 3072
    assert q.qlin_scales_bytes(F.INT8_ROW, L.CANONICAL, 4096, 3072) == 4096 * 4
    assert q.qlin_quant_workspace_bytes(F.INT8_ROW, 4096, 3072) == 0
    assert q.qlin_gemm_workspace_bytes(F.INT8_ROW, F.INT8_ROW, 4096, 12288, 3072) == 0
    # MXFP4 dual-scale: MXFP4's codes and fine scales, coarse fp32 scales per 512 in `global`
    assert q.qlin_codes_bytes(F.MXFP4_DUAL, 20280, 5120) == 20280 * 2560
    assert q.qlin_scales_bytes(F.MXFP4_DUAL, L.MMA, 20280, 5120) == 20352 * 160
    assert q.qlin_global_bytes(F.MXFP4_DUAL, 20280, 5120) == 20280 * 10 * 4
    assert q.qlin_global_bytes(F.NVFP4, 20280, 5120) == 4 and q.qlin_global_bytes(F.MXFP4, 20280, 5120) == 0
    # symmetric int4: the asymmetric variant's layouts
    for fn in (q.qlin_codes_bytes, q.qlin_zeros_bytes, q.qlin_quant_workspace_bytes):
        assert fn(F.INT4_G128_SYM, 4096, 12288) == fn(F.INT4_G128_ASYM, 4096, 12288)
    assert q.qlin_scales_bytes(F.INT4_G128_SYM, L.CANONICAL, 4096, 12288) == 96 * 4096 * 2
    assert q.qlin_gemm_workspace_bytes(F.INT4_G128_SYM, F.BF16, 16, 4096, 4096) == 0


FAKE = 1 << 20          # a 16-byte aligned non-null value; never dereferenced by these calls


def test_quantize_rejects_bad_arguments(q):
    F, L, S = q.Fmt, q.Layout, q.Status
    ws = q.qlin_quant_workspace_bytes(F.FP8_TENSOR, 128, 1024)
    # null source / outputs
    assert q.qlin_quantize_act(F.FP8_TOKEN, None, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE, 128, 1024, 1024, None, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG
    # K not a multiple of 8, ld < K, empty
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE, 128, 1020, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE, 128, 1024, 512, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE, 0, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG
    # misaligned source
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE + 2, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0,
                               None, None) == S.ALIGNMENT
    # per-tensor without workspace
    assert q.qlin_quantize_act(F.FP8_TENSOR, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.WORKSPACE
    assert q.qlin_quantize_act(F.FP8_TENSOR, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, FAKE, ws - 4,
                               None, None) == S.WORKSPACE
    # block-128 shape rules
    assert q.qlin_quantize_weight(F.FP8_BLOCK128, FAKE, 200, 1024, 1024, FAKE, FAKE, None, None, L.CANONICAL,
                                  None, 0, None, None) == S.INVALID_ARG
    # MMA layout only for MX / NVFP4; MX MMA layout needs K % 128
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.MMA, None, 0, None,
                               None) == S.UNSUPPORTED
    assert q.qlin_quantize_act(F.MXFP8, FAKE, 128, 96, 96, FAKE, FAKE, None, L.MMA, None, 0, None,
                               None) == S.INVALID_ARG
    assert q.qlin_quantize_act(F.MXFP4, FAKE, 128, 96, 96, FAKE, FAKE, None, L.MMA, None, 0, None,
                               None) == S.INVALID_ARG
    assert q.qlin_quantize_act(F.MXFP4, FAKE, 128, 80, 80, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG                  # K % 32
    assert q.qlin_quantize_act(F.FP8_GROUP128, FAKE, 128, 96, 96, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG                  # K % 128
    assert q.qlin_quantize_act(F.FP8_GROUP128, FAKE, 128, 128, 128, FAKE, FAKE, None, L.MMA, None, 0, None,
                               None) == S.UNSUPPORTED                  # no tensor-core scale layout
    assert q.qlin_quantize_act(F.INT8_ROW, FAKE, 128, 1020, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG                  # K % 8
    assert q.qlin_quantize_weight(F.INT8_ROW, FAKE, 128, 1024, 1024, FAKE, FAKE + 2, None, None, L.CANONICAL,
                                  None, 0, None, None) == S.ALIGNMENT  # float scales
    assert q.qlin_quantize_weight(F.INT8_ROW, FAKE, 128, 1024, 1024, FAKE, FAKE, None, None, L.MMA, None, 0,
                                  None, None) == S.UNSUPPORTED
    # NVFP4 needs the global-scale output
    assert q.qlin_quantize_act(F.NVFP4, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, FAKE, 1 << 20,
                               None, None) == S.INVALID_ARG
    # int4 is weight-only, and needs zeros
    assert q.qlin_quantize_act(F.INT4_G128_ASYM, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0,
                               None, None) == S.UNSUPPORTED
    assert q.qlin_quantize_weight(F.INT4_G128_ASYM, FAKE, 128, 1024, 1024, FAKE, FAKE, None, None, L.CANONICAL,
                                  None, 0, None, None) == S.INVALID_ARG
    assert q.qlin_quantize_weight(F.BF16, FAKE, 128, 1024, 1024, FAKE, FAKE, None, None, L.CANONICAL, None, 0,
                                  None, None) == S.UNSUPPORTED
    assert q.qlin_quantize_act(F.INT4_G128_SYM, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.CANONICAL, None, 0,
                               None, None) == S.UNSUPPORTED
    assert q.qlin_quantize_weight(F.INT4_G128_SYM, FAKE, 128, 1024, 1024, FAKE, FAKE, None, None, L.CANONICAL,
                                  None, 0, None, None) == S.INVALID_ARG                 # zeros missing
    assert q.qlin_quantize_weight(F.INT4_G128_SYM, FAKE, 100, 1024, 1024, FAKE, FAKE, FAKE, None, L.CANONICAL,
                                  None, 0, None, None) == S.INVALID_ARG                 # N % 8
    assert q.qlin_quantize_weight(F.INT4_G128_SYM, FAKE, 128, 1024, 1024, FAKE, FAKE, FAKE, None, L.MMA,
                                  None, 0, None, None) == S.UNSUPPORTED
    # MXFP4 dual-scale: K % 512, and the coarse-scale buffer is required
    assert q.qlin_quantize_act(F.MXFP4_DUAL, FAKE, 128, 768, 768, FAKE, FAKE, FAKE, L.MMA, None, 0,
                               None, None) == S.INVALID_ARG
    assert q.qlin_quantize_act(F.MXFP4_DUAL, FAKE, 128, 1024, 1024, FAKE, FAKE, None, L.MMA, None, 0,
                               None, None) == S.INVALID_ARG


def test_gemm_rejects_bad_arguments(q):
    F, L, S = q.Fmt, q.Layout, q.Status

    def g(wf, xf, M, N, K, layout=L.CANONICAL, x=FAKE, y=FAKE, ldy=None, xs=FAKE, ws=FAKE, xg=FAKE, wg=FAKE,
          wz=FAKE, work=None, work_bytes=0):
        return q.qlin_gemm(wf, xf, M, N, K, x, xs, xg, FAKE, ws, wz, wg, None, y, N if ldy is None else ldy, layout,
                           work, work_bytes, None, None)

    assert g(F.FP8_TENSOR, F.FP8_TENSOR, 0, 1024, 1024) == S.INVALID_ARG
    assert g(F.FP8_TENSOR, F.FP8_TENSOR, 128, 1024, 1024, x=None) == S.INVALID_ARG
    assert g(F.FP8_TENSOR, F.FP8_TENSOR, 128, 1024, 1024, y=FAKE + 8) == S.ALIGNMENT
    assert g(F.FP8_TENSOR, F.FP8_TENSOR, 128, 1024, 1024, ldy=1000) == S.INVALID_ARG
    assert g(F.FP8_TENSOR, F.FP8_TENSOR, 128, 1024, 1024, xs=None) == S.INVALID_ARG
    assert g(F.FP8_BLOCK128, F.FP8_TOKEN, 128, 1000, 1024) == S.INVALID_ARG
    assert g(F.MXFP8, F.MXFP8, 128, 1024, 1024) == S.UNSUPPORTED          # canonical scales
    assert g(F.MXFP8, F.MXFP8, 128, 1024, 1056, layout=L.MMA) == S.INVALID_ARG
    assert g(F.NVFP4, F.NVFP4, 128, 1024, 1024, layout=L.MMA, xg=None) == S.INVALID_ARG
    assert g(F.NVFP4, F.FP8_TOKEN, 128, 1024, 1024, layout=L.MMA) == S.UNSUPPORTED
    assert g(F.MXFP4, F.MXFP4, 128, 1024, 1024) == S.UNSUPPORTED          # canonical scales
    assert g(F.MXFP4, F.MXFP4, 128, 1024, 1152, layout=L.MMA) == S.INVALID_ARG   # K % 256
    assert g(F.MXFP4, F.MXFP8, 128, 1024, 1024, layout=L.MMA) == S.UNSUPPORTED
    assert g(F.FP8_BLOCK128, F.FP8_GROUP128, 128, 1024, 1000) == S.INVALID_ARG   # K % 128
    assert g(F.FP8_BLOCK128, F.FP8_GROUP128, 128, 1024, 1024, xs=None) == S.INVALID_ARG
    assert g(F.FP8_TENSOR, F.FP8_GROUP128, 128, 1024, 1024) == S.UNSUPPORTED
    assert g(F.FP8_TENSOR, F.FP8_TOKEN, 128, 1024, 1024) == S.UNSUPPORTED
    assert g(F.FP8_TENSOR, F.BF16, 129, 1024, 1024) == S.UNSUPPORTED           # fused X: M <= 128
    assert g(F.FP8_TENSOR, F.BF16, 128, 1024, 1000) == S.INVALID_ARG           # K % 16
    assert g(F.FP8_TENSOR, F.BF16, 128, 1024, 1024, ws=None) == S.INVALID_ARG
    assert g(F.INT8_ROW, F.INT8_ROW, 128, 1024, 1000) == S.INVALID_ARG         # K % 16
    assert g(F.INT8_ROW, F.INT8_ROW, 128, 1024, 1024, ws=None) == S.INVALID_ARG
    assert g(F.INT8_ROW, F.FP8_TOKEN, 128, 1024, 1024) == S.UNSUPPORTED
    assert g(F.MXFP4_DUAL, F.MXFP4_DUAL, 128, 1024, 1024) == S.UNSUPPORTED        # canonical scales
    assert g(F.MXFP4_DUAL, F.MXFP4_DUAL, 128, 1024, 768, layout=L.MMA) == S.INVALID_ARG   # K % 512
    assert g(F.MXFP4_DUAL, F.MXFP4_DUAL, 128, 1024, 1024, layout=L.MMA, wg=None) == S.INVALID_ARG
    assert g(F.MXFP4_DUAL, F.MXFP4, 128, 1024, 1024, layout=L.MMA) == S.UNSUPPORTED
    assert g(F.FP8_BLOCK128, F.INT8_ROW, 128, 1024, 1024) == S.UNSUPPORTED
    assert g(F.INT4_G128_ASYM, F.BF16, 16, 4096, 4000) == S.INVALID_ARG
    need = q.qlin_gemm_workspace_bytes(F.INT4_G128_ASYM, F.BF16, 16, 4096, 4096)
    if need:
        assert g(F.INT4_G128_ASYM, F.BF16, 16, 4096, 4096, work=None) == S.WORKSPACE


def test_shapes_past_the_32_bit_limits_are_rejected_before_any_launch(q):
    F, L, S = q.Fmt, q.Layout, q.Status
    big = 1 << 31
    # quantizers: K, and rows x 256-element tasks, within 32 bits
    assert q.qlin_quantize_act(F.FP8_TOKEN, FAKE, 1, big, big, FAKE, FAKE, None, L.CANONICAL, None, 0, None,
                               None) == S.INVALID_ARG
    for fmt in (F.FP8_TENSOR, F.MXFP8, F.NVFP4, F.FP8_GROUP128, F.INT8_ROW):
        assert q.qlin_quantize_act(fmt, FAKE, 1 << 24, 1 << 16, 1 << 16, FAKE, FAKE, FAKE, L.CANONICAL, FAKE,
                                   1 << 30, None, None) == S.INVALID_ARG, fmt
    # rows padded to 128 for the MMA scale layout count too
    rows = (1 << 31) - 1
    assert q.qlin_quantize_act(F.MXFP8, FAKE, rows, 128, 128, FAKE, FAKE, None, L.MMA, None, 0, None,
                               None) == S.INVALID_ARG

    def g(wf, xf, M, N, K, layout=L.CANONICAL):
        return q.qlin_gemm(wf, xf, M, N, K, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, N, layout, None,
                           0, None, None)

    assert g(F.FP8_TENSOR, F.FP8_TENSOR, 16, 16, big) == S.INVALID_ARG
    assert g(F.FP8_BLOCK128, F.FP8_TOKEN, big - 1, big - 128, 128) == S.INVALID_ARG     # tiles past 2^31
    # W4A16: 128-channel tiles and 64-token tiles on grid dimensions y and z
    assert g(F.INT4_G128_ASYM, F.BF16, 65535 * 64 + 1, 4096, 4096) == S.INVALID_ARG
    assert g(F.INT4_G128_ASYM, F.BF16, 16, 65535 * 128 + 8, 4096) == S.INVALID_ARG


def test_mma_layout_reader_matches_the_documented_formula():
    from layouts import mma_to_canonical
    rows, nsc = 200, 8
    buf = np.zeros(2 * 2 * 512, np.uint8)
    canon = (np.arange(rows * nsc) % 251).astype(np.uint8).reshape(rows, nsc)
    for r in range(rows):
        for j in range(nsc):
            tile, rr, chunk, jj = r // 128, r % 128, j // 4, j % 4
            buf[(tile * 2 + chunk) * 512 + 16 * (rr % 32) + 4 * (rr // 32) + jj] = canon[r, j]
    assert np.array_equal(mma_to_canonical(buf, rows, nsc), canon)


def test_plain_c_consumer_compiles_links_and_passes(q, tmp_path):
    """include/qlin.h is plain C99 (no C++ or CUDA headers) and libqlin.so links
    into a C program; the program checks sizes and validation without a GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_check")
    libdir = os.path.dirname(q.LIB_PATH)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-o", exe, q.LIB_PATH, f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c abi ok" in r.stdout, r.stdout + r.stderr
