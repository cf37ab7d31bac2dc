"""Slow, obviously-correct CPU oracle for the quantized-linear hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library shares no code with it and never calls it.

Two layers:

* ``qlin_oracle.c`` (built here into ``_build/liboracle.so`` with gcc, strict
  IEEE binary32, no contraction): scalar codecs and quantizers, written one
  element at a time from the format definitions.  See its header for the
  readings R1..R5, R11..R13, R15 and R16 taken where the pages name a format but print no
  formula.
* this module: numpy marshalling, and the GEMM reference, which is the plain
  definition Y = Xhat @ What^T evaluated in float64 over the dequantized
  operands (``numpy.matmul`` as the one library step).

Sources for what is computed: "[vLLM] 기타 양자화: FP8, ModelOpt, INC, TorchAO,
Quark" section "FP8: vLLM의 핵심 양자화" (FP8 granularities);
"vLLM-Omni 在线量化（Online Quantization）完全指南" section "在线量化的底层工作原理"
(load-time weight quantization, dynamic activation quantization, then the
quantized matmul; MXFP8's E8M0 scale per 32 K elements); "vLLM-Omni 量化推理实践"
Table 1 (mixed FP8/NVFP4 linears); "vLLM-Omni는 AutoRound 양자화로 추론을
가속화합니다" section "새로운 모델 양자화" (int4, group 128, auto_gptq packing,
``--iters 0``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlin_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations", "-frounding-math"]


def build(force: bool = False) -> str:
    """Compile ``qlin_oracle.c`` into ``_build/liboracle.so`` (gcc) if stale."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
        sig = {
            "oracle_bf16_to_f32": ([ctypes.c_uint16], F),
            "oracle_f32_to_bf16": ([F], ctypes.c_uint16),
            "oracle_floor_log2": ([F], ctypes.c_int),
            "oracle_dec_e4m3": ([ctypes.c_uint8], ctypes.c_double),
            "oracle_enc_e4m3": ([F], ctypes.c_uint8),
            "oracle_dec_e2m1": ([ctypes.c_uint8], ctypes.c_double),
            "oracle_enc_e2m1": ([F], ctypes.c_uint8),
            "oracle_dec_e8m0": ([ctypes.c_uint8], ctypes.c_double),
            "oracle_quant_fp8_tensor": ([P, I64, I64, I64, P, P], None),
            "oracle_quant_fp8_token": ([P, I64, I64, I64, P, P], None),
            "oracle_quant_fp8_block128": ([P, I64, I64, I64, P, P], None),
            "oracle_quant_fp8_group128": ([P, I64, I64, I64, P, P], None),
            "oracle_quant_mxfp8": ([P, I64, I64, I64, P, P], None),
            "oracle_quant_nvfp4": ([P, I64, I64, I64, P, P, P], None),
            "oracle_quant_mxfp4": ([P, I64, I64, I64, P, P], None),
            "oracle_quant_int4_g128": ([P, I64, I64, I64, P, P, P], None),
            "oracle_quant_int4_g128_sym": ([P, I64, I64, I64, P, P, P], None),
            "oracle_quant_mxfp4_dual": ([P, I64, I64, I64, P, P, P], None),
            "oracle_dequant_mxfp4_dual": ([P, I64, I64, P, P, P], None),
            "oracle_quant_int8_row": ([P, I64, I64, I64, P, P], None),
            "oracle_dequant_fp8_tensor": ([P, I64, I64, F, P], None),
            "oracle_dequant_fp8_token": ([P, I64, I64, P, P], None),
            "oracle_dequant_fp8_block128": ([P, I64, I64, P, P], None),
            "oracle_dequant_fp8_group128": ([P, I64, I64, P, P], None),
            "oracle_dequant_mxfp8": ([P, I64, I64, P, P], None),
            "oracle_dequant_nvfp4": ([P, I64, I64, P, F, P], None),
            "oracle_dequant_mxfp4": ([P, I64, I64, P, P], None),
            "oracle_dequant_int4_g128": ([P, P, P, I64, I64, P], None),
            "oracle_dequant_int8_row": ([P, I64, I64, P, P], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a 2-D uint16 array of bf16 bits (or a torch bf16 CPU tensor)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(getattr(x, "dtype", "")) == "torch.bfloat16":
        import torch
        x = x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError("oracle expects a 2-D array of bf16 bit patterns (uint16)")
    return x


# ---------------------------------------------------------------- scalar codecs
def bf16_to_f32(h: int) -> float:
    return _load().oracle_bf16_to_f32(h)


def f32_to_bf16(f: float) -> int:
    return _load().oracle_f32_to_bf16(f)


def floor_log2(a: float) -> int:
    return _load().oracle_floor_log2(a)


def dec_e4m3(c: int) -> float:
    return _load().oracle_dec_e4m3(c)


def enc_e4m3(v: float) -> int:
    return _load().oracle_enc_e4m3(v)


def dec_e2m1(c: int) -> float:
    return _load().oracle_dec_e2m1(c)


def enc_e2m1(v: float) -> int:
    return _load().oracle_enc_e2m1(v)


def dec_e8m0(c: int) -> float:
    return _load().oracle_dec_e8m0(c)


# ---------------------------------------------------------------- quantizers
def quant_fp8_tensor(x):
    """Per-tensor dynamic E4M3 -> (codes uint8 [R,K], scale float32)."""
    x = _bf16_bits(x)
    R, K = x.shape
    codes = np.empty((R, K), np.uint8)
    s = np.zeros(1, np.float32)
    _load().oracle_quant_fp8_tensor(_p(x), R, K, K, _p(codes), _p(s))
    return codes, s[0]


def quant_fp8_token(x):
    """Per-row dynamic E4M3 -> (codes uint8 [R,K], scales float32 [R])."""
    x = _bf16_bits(x)
    R, K = x.shape
    codes = np.empty((R, K), np.uint8)
    s = np.empty(R, np.float32)
    _load().oracle_quant_fp8_token(_p(x), R, K, K, _p(codes), _p(s))
    return codes, s


def quant_int8_row(x):
    """Symmetric INT8, one scale per row (a token of X or a channel of W)
    -> (codes int8 [R,K], scales float32 [R])."""
    x = _bf16_bits(x)
    R, K = x.shape
    codes = np.empty((R, K), np.int8)
    s = np.empty(R, np.float32)
    _load().oracle_quant_int8_row(_p(x), R, K, K, _p(codes), _p(s))
    return codes, s


def quant_fp8_group128(x):
    """Dynamic E4M3 per 1 x 128 group -> (codes uint8 [R,K], scales float32 [R, K/128])."""
    x = _bf16_bits(x)
    R, K = x.shape
    if K % 128:
        raise ValueError("FP8 group-128 needs K multiple of 128")
    codes = np.empty((R, K), np.uint8)
    s = np.empty((R, K // 128), np.float32)
    _load().oracle_quant_fp8_group128(_p(x), R, K, K, _p(codes), _p(s))
    return codes, s


def quant_fp8_block128(x):
    """128x128-tile E4M3 -> (codes uint8 [R,K], scales float32 [R/128, K/128])."""
    x = _bf16_bits(x)
    R, K = x.shape
    if R % 128 or K % 128:
        raise ValueError("block-128 needs rows and K multiples of 128")
    codes = np.empty((R, K), np.uint8)
    s = np.empty((R // 128, K // 128), np.float32)
    _load().oracle_quant_fp8_block128(_p(x), R, K, K, _p(codes), _p(s))
    return codes, s


def quant_mxfp8(x):
    """MXFP8 -> (codes uint8 [R,K], E8M0 scale codes uint8 [R, K/32])."""
    x = _bf16_bits(x)
    R, K = x.shape
    if K % 32:
        raise ValueError("MXFP8 needs K multiple of 32")
    codes = np.empty((R, K), np.uint8)
    sc = np.empty((R, K // 32), np.uint8)
    _load().oracle_quant_mxfp8(_p(x), R, K, K, _p(codes), _p(sc))
    return codes, sc


def quant_nvfp4(x):
    """NVFP4 -> (packed uint8 [R,K/2], UE4M3 scale codes uint8 [R,K/16], global float32)."""
    x = _bf16_bits(x)
    R, K = x.shape
    if K % 16:
        raise ValueError("NVFP4 needs K multiple of 16")
    packed = np.empty((R, K // 2), np.uint8)
    sc = np.empty((R, K // 16), np.uint8)
    g = np.zeros(1, np.float32)
    _load().oracle_quant_nvfp4(_p(x), R, K, K, _p(packed), _p(sc), _p(g))
    return packed, sc, g[0]


def quant_mxfp4(x):
    """MXFP4 -> (packed E2M1 uint8 [R,K/2], E8M0 scale codes uint8 [R,K/32])."""
    x = _bf16_bits(x)
    R, K = x.shape
    if K % 32:
        raise ValueError("MXFP4 needs K multiple of 32")
    packed = np.empty((R, K // 2), np.uint8)
    sc = np.empty((R, K // 32), np.uint8)
    _load().oracle_quant_mxfp4(_p(x), R, K, K, _p(packed), _p(sc))
    return packed, sc


def quant_mxfp4_dual(x):
    """MXFP4 dual-scale (reading R16) -> (packed E2M1 uint8 [R,K/2], fine E8M0
    scale codes uint8 [R,K/32], coarse fp32 scales [R,K/512])."""
    x = _bf16_bits(x)
    R, K = x.shape
    if K % 512:
        raise ValueError("MXFP4 dual-scale needs K multiple of 512")
    packed = np.empty((R, K // 2), np.uint8)
    sc = np.empty((R, K // 32), np.uint8)
    coarse = np.empty((R, K // 512), np.float32)
    _load().oracle_quant_mxfp4_dual(_p(x), R, K, K, _p(packed), _p(sc), _p(coarse))
    return packed, sc, coarse


def quant_int4_g128(w):
    """int4 asymmetric g128 RTN of W [N,K] -> (qweight int32 [K/8,N],
    scales bf16 bits uint16 [K/128,N], qzeros int32 [K/128,N/8])."""
    w = _bf16_bits(w)
    N, K = w.shape
    if N % 8 or K % 128:
        raise ValueError("int4 g128 needs N multiple of 8 and K multiple of 128")
    qw = np.empty((K // 8, N), np.int32)
    sc = np.empty((K // 128, N), np.uint16)
    qz = np.empty((K // 128, N // 8), np.int32)
    _load().oracle_quant_int4_g128(_p(w), N, K, K, _p(qw), _p(sc), _p(qz))
    return qw, sc, qz


def quant_int4_g128_sym(w):
    """int4 symmetric g128 RTN of W [N,K] (reading R15: range [-a, a], zero
    point 8) -> (qweight int32 [K/8,N], scales bf16 bits uint16 [K/128,N],
    qzeros int32 [K/128,N/8], every zero point 8).  Dequantize with
    dequant_int4_g128."""
    w = _bf16_bits(w)
    N, K = w.shape
    if N % 8 or K % 128:
        raise ValueError("int4 g128 needs N multiple of 8 and K multiple of 128")
    qw = np.empty((K // 8, N), np.int32)
    sc = np.empty((K // 128, N), np.uint16)
    qz = np.empty((K // 128, N // 8), np.int32)
    _load().oracle_quant_int4_g128_sym(_p(w), N, K, K, _p(qw), _p(sc), _p(qz))
    return qw, sc, qz


# ---------------------------------------------------------------- dequantizers
def _f64(shape):
    return np.empty(shape, np.float64)


def dequant_fp8_tensor(codes, scale):
    codes = np.ascontiguousarray(codes, np.uint8)
    out = _f64(codes.shape)
    _load().oracle_dequant_fp8_tensor(_p(codes), codes.shape[0], codes.shape[1], float(scale), _p(out))
    return out


def dequant_fp8_token(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    out = _f64(codes.shape)
    _load().oracle_dequant_fp8_token(_p(codes), codes.shape[0], codes.shape[1], _p(scales), _p(out))
    return out


def dequant_int8_row(codes, scales):
    codes = np.ascontiguousarray(codes, np.int8)
    scales = np.ascontiguousarray(scales, np.float32)
    out = _f64(codes.shape)
    _load().oracle_dequant_int8_row(_p(codes), codes.shape[0], codes.shape[1], _p(scales), _p(out))
    return out


def dequant_fp8_group128(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    out = _f64(codes.shape)
    _load().oracle_dequant_fp8_group128(_p(codes), codes.shape[0], codes.shape[1], _p(scales), _p(out))
    return out


def dequant_fp8_block128(codes, scales):
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    out = _f64(codes.shape)
    _load().oracle_dequant_fp8_block128(_p(codes), codes.shape[0], codes.shape[1], _p(scales), _p(out))
    return out


def dequant_mxfp8(codes, scale_codes):
    codes = np.ascontiguousarray(codes, np.uint8)
    scale_codes = np.ascontiguousarray(scale_codes, np.uint8)
    out = _f64(codes.shape)
    _load().oracle_dequant_mxfp8(_p(codes), codes.shape[0], codes.shape[1], _p(scale_codes), _p(out))
    return out


def dequant_nvfp4(packed, scale_codes, global_scale):
    packed = np.ascontiguousarray(packed, np.uint8)
    scale_codes = np.ascontiguousarray(scale_codes, np.uint8)
    R, K = packed.shape[0], packed.shape[1] * 2
    out = _f64((R, K))
    _load().oracle_dequant_nvfp4(_p(packed), R, K, _p(scale_codes), float(global_scale), _p(out))
    return out


def dequant_mxfp4(packed, scale_codes):
    packed = np.ascontiguousarray(packed, np.uint8)
    scale_codes = np.ascontiguousarray(scale_codes, np.uint8)
    R, K = packed.shape[0], packed.shape[1] * 2
    out = _f64((R, K))
    _load().oracle_dequant_mxfp4(_p(packed), R, K, _p(scale_codes), _p(out))
    return out


def dequant_mxfp4_dual(packed, scale_codes, coarse):
    packed = np.ascontiguousarray(packed, np.uint8)
    scale_codes = np.ascontiguousarray(scale_codes, np.uint8)
    coarse = np.ascontiguousarray(coarse, np.float32)
    R, K = packed.shape[0], packed.shape[1] * 2
    out = _f64((R, K))
    _load().oracle_dequant_mxfp4_dual(_p(packed), R, K, _p(scale_codes), _p(coarse), _p(out))
    return out


def dequant_int4_g128(qweight, scales, qzeros):
    qweight = np.ascontiguousarray(qweight, np.int32)
    scales = np.ascontiguousarray(scales, np.uint16)
    qzeros = np.ascontiguousarray(qzeros, np.int32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    out = _f64((N, K))
    _load().oracle_dequant_int4_g128(_p(qweight), _p(scales), _p(qzeros), N, K, _p(out))
    return out


def bf16_values(x) -> np.ndarray:
    """bf16 bit patterns -> exact float64 values (bf16 is the top half of binary32)."""
    x = _bf16_bits(x)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- GEMM reference
def gemm_ref(xhat: np.ndarray, what: np.ndarray, alpha: float = 1.0, bias=None) -> np.ndarray:
    """Y = alpha * Xhat @ What^T (+ bias), all in float64.

    The quantized matmul of "vLLM-Omni 在线量化（Online Quantization）完全指南"
    section "在线量化的底层工作原理" stage 3, with the scales already folded into
    the dequantized operands (they are exact in binary64)."""
    y = np.matmul(np.asarray(xhat, np.float64), np.asarray(what, np.float64).T)
    if alpha != 1.0:
        y = y * alpha
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


def bf16_round(y: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 (via nearest binary32, then bf16 RNE), as float64."""
    f = np.asarray(y, np.float64).astype(np.float32)
    flat = f.reshape(-1)
    out = np.empty(flat.shape, np.float64)
    u = flat.view(np.uint32)
    kept = (u >> 16).astype(np.uint64)
    rest = (u & 0xFFFF).astype(np.uint64)
    up = (rest > 0x8000) | ((rest == 0x8000) & ((kept & 1) == 1))
    kept = (kept + up.astype(np.uint64)).astype(np.uint32)
    out[:] = (kept << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    return out.reshape(f.shape)


def gemm_metrics(y_test: np.ndarray, y_ref: np.ndarray) -> dict:
    """The output-similarity set of "vLLM-Omni 在线量化（Online Quantization）完全指南"
    section "验证与注意事项" item 1 (cosine, mae, mse/rmse, max_abs, relative_l2,
    psnr_db), evaluated on GEMM outputs, plus the bf16-rounding floor of Y_ref."""
    yt = np.asarray(y_test, np.float64)
    yr = np.asarray(y_ref, np.float64)
    d = yt - yr
    ref_norm = np.linalg.norm(yr)
    mse = float(np.mean(d * d))
    peak = float(np.max(np.abs(yr))) if yr.size else 0.0
    rel_l2 = float(np.linalg.norm(d) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(d))
    bf = bf16_round(yr)
    floor = float(np.linalg.norm(bf - yr) / ref_norm) if ref_norm > 0 else 0.0
    denom = float(np.linalg.norm(yt) * ref_norm)
    return {
        "relative_l2": rel_l2,
        "bf16_floor": floor,
        "max_abs": float(np.max(np.abs(d))) if d.size else 0.0,
        "mae": float(np.mean(np.abs(d))) if d.size else 0.0,
        "mse": mse,
        "rmse": mse ** 0.5,
        "cosine": float(np.sum(yt * yr) / denom) if denom > 0 else 1.0,
        "psnr_db": float(10 * np.log10(peak * peak / mse)) if mse > 0 and peak > 0 else float("inf"),
    }


GEMM_REL_TOL = 2e-3


def gemm_pass(y_test: np.ndarray, y_ref: np.ndarray) -> tuple[bool, dict]:
    """Pass criterion: relative Frobenius error <= 2e-3 + the relative Frobenius
    error that rounding Y_ref itself to bf16 costs."""
    m = gemm_metrics(y_test, y_ref)
    return m["relative_l2"] <= GEMM_REL_TOL + m["bf16_floor"], m
