"""Thin ctypes binding over ``libqlin.so``.

The ``qlin_*`` functions mirror the C ABI in ``include/qlin.h`` one to one
(device pointers as integers, the stream as an integer handle).  The
lower-case helpers below them only marshal torch tensors: they allocate the
output buffers with torch (plumbing), pass pointers and the current stream,
and raise if the library returns an error.  Every step of the computation
runs in the library's CUDA kernels; there is no other path.
"""
from __future__ import annotations

import ctypes
import enum
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqlin.so")


class Fmt(enum.IntEnum):
    FP8_TENSOR = 0
    FP8_TOKEN = 1
    FP8_BLOCK128 = 2
    MXFP8 = 3
    NVFP4 = 4
    INT4_G128_ASYM = 5
    BF16 = 6
    MXFP4 = 7
    FP8_GROUP128 = 8
    INT8_ROW = 9
    INT4_G128_SYM = 10
    MXFP4_DUAL = 11


class Layout(enum.IntEnum):
    CANONICAL = 0
    MMA = 1


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    ALIGNMENT = 3
    WORKSPACE = 4
    CUDA = 5
    DEVICE_TIMEOUT = 6


class QlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        extra = f", cudaError {qlin_last_cuda_error()}" if self.status == Status.CUDA else ""
        super().__init__(f"{where}: {self.status.name} ({qlin_status_string(status)}{extra})")


_lib = None

_P, _I64, _SZ, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run serving_amax_reduce_gb300.build.build() "
                           "(or __graft_entry__.build()) first; there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    sigs = {
        "qlin_status_string": ([_I], ctypes.c_char_p),
        "qlin_version": ([], ctypes.c_char_p),
        "qlin_last_cuda_error": ([], _I),
        "qlin_codes_bytes": ([_I, _I64, _I64], _SZ),
        "qlin_scales_bytes": ([_I, _I, _I64, _I64], _SZ),
        "qlin_zeros_bytes": ([_I, _I64, _I64], _SZ),
        "qlin_global_bytes": ([_I, _I64, _I64], _SZ),
        "qlin_quant_workspace_bytes": ([_I, _I64, _I64], _SZ),
        "qlin_gemm_workspace_bytes": ([_I, _I, _I64, _I64, _I64], _SZ),
        "qlin_quantize_weight": ([_I, _P, _I64, _I64, _I64, _P, _P, _P, _P, _I, _P, _SZ, _P, _P], _I),
        "qlin_quantize_act": ([_I, _P, _I64, _I64, _I64, _P, _P, _P, _I, _P, _SZ, _P, _P], _I),
        "qlin_gemm": ([_I, _I, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _P, _SZ, _P, _P],
                      _I),
        "qlin_debug_expire_wait": ([_P, ctypes.c_uint32, _P], _I),
        "qlin_quantize_fp8_tensor_noalloc": ([_P, _I64, _I64, _I64, _P, _P, _P], _I),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def lib_handle():
    return _load()


# ------------------------------------------------------------------ C ABI, 1:1
def qlin_status_string(s: int) -> str:
    return _load().qlin_status_string(int(s)).decode()


def qlin_version() -> str:
    return _load().qlin_version().decode()


def qlin_last_cuda_error() -> int:
    return _load().qlin_last_cuda_error()


def qlin_codes_bytes(fmt, rows, K) -> int:
    return _load().qlin_codes_bytes(int(fmt), rows, K)


def qlin_scales_bytes(fmt, layout, rows, K) -> int:
    return _load().qlin_scales_bytes(int(fmt), int(layout), rows, K)


def qlin_zeros_bytes(fmt, rows, K) -> int:
    return _load().qlin_zeros_bytes(int(fmt), rows, K)


def qlin_global_bytes(fmt, rows, K) -> int:
    return _load().qlin_global_bytes(int(fmt), rows, K)


def qlin_quant_workspace_bytes(fmt, rows, K) -> int:
    return _load().qlin_quant_workspace_bytes(int(fmt), rows, K)


def qlin_gemm_workspace_bytes(w_fmt, x_fmt, M, N, K) -> int:
    return _load().qlin_gemm_workspace_bytes(int(w_fmt), int(x_fmt), M, N, K)


def qlin_quantize_weight(fmt, w, N, K, ldw, codes, scales, zeros, global_, layout, ws, ws_bytes, status,
                         stream) -> int:
    return _load().qlin_quantize_weight(int(fmt), w, N, K, ldw, codes, scales, zeros, global_, int(layout), ws,
                                        ws_bytes, status, stream)


def qlin_quantize_act(fmt, x, M, K, ldx, codes, scales, global_, layout, ws, ws_bytes, status, stream) -> int:
    return _load().qlin_quantize_act(int(fmt), x, M, K, ldx, codes, scales, global_, int(layout), ws, ws_bytes,
                                     status, stream)


def qlin_gemm(w_fmt, x_fmt, M, N, K, x, x_scales, x_global, w_codes, w_scales, w_zeros, w_global, bias, y, ldy,
              layout, ws, ws_bytes, status, stream) -> int:
    return _load().qlin_gemm(int(w_fmt), int(x_fmt), M, N, K, x, x_scales, x_global, w_codes, w_scales, w_zeros,
                             w_global, bias, y, ldy, int(layout), ws, ws_bytes, status, stream)


def qlin_debug_expire_wait(status, max_polls, stream) -> int:
    return _load().qlin_debug_expire_wait(status, max_polls, stream)


NOALLOC_MAX_ELEMENTS = 4096 * 16384


def qlin_quantize_fp8_tensor_noalloc(x, rows, K, ld, codes, scale, stream) -> int:
    """Per-tensor FP8 quantization that allocates nothing and takes no
    workspace (for callers that cannot allocate device memory); see qlin.h."""
    return _load().qlin_quantize_fp8_tensor_noalloc(x, rows, K, ld, codes, scale, stream)


# ------------------------------------------------------------------ torch marshalling
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


_status_bufs: dict = {}


def device_status(device=None) -> torch.Tensor:
    """The int32 device word the helpers below pass as dev_status when the
    caller gives none (one per device, zeroed on creation)."""
    dev = torch.device(device if device is not None else "cuda")
    key = (dev.type, dev.index if dev.index is not None else torch.cuda.current_device())
    if key not in _status_bufs:
        _status_bufs[key] = torch.zeros(1, dtype=torch.int32, device=dev)
    return _status_bufs[key]


def read_device_status(device=None, reset: bool = True) -> int:
    """Synchronizing read of the default status word (test/debug helper)."""
    st = device_status(device)
    v = int(st.item())
    if reset and v:
        st.zero_()
    return v


def _check(rc: int, where: str):
    if rc != 0:
        raise QlinError(rc, where)


def _need(t, nbytes: int, what: str):
    """The library writes or reads `nbytes` bytes at t's address: refuse a
    smaller or non-contiguous buffer before any pointer is handed over."""
    if not nbytes:
        return
    if t is None:
        raise ValueError(f"{what}: a buffer of {nbytes} bytes is required")
    if not t.is_contiguous() or t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{what}: needs {nbytes} contiguous bytes, got {t.numel() * t.element_size()}"
                         f"{'' if t.is_contiguous() else ' (not contiguous)'}")


def _check_quant_bufs(fmt: Fmt, rows: int, K: int, layout: Layout, b: dict):
    _need(b["codes"], qlin_codes_bytes(fmt, rows, K), "codes")
    _need(b["scales"], qlin_scales_bytes(fmt, layout, rows, K), "scales")
    _need(b.get("zeros"), qlin_zeros_bytes(fmt, rows, K), "zeros")
    _need(b.get("global"), qlin_global_bytes(fmt, rows, K), "global")
    wsb = qlin_quant_workspace_bytes(fmt, rows, K)
    _need(b.get("workspace"), wsb, "workspace")
    if b.get("workspace_bytes", 0) < wsb:
        raise ValueError(f"workspace_bytes: {wsb} required")


def _empty(nbytes: int, device, dtype=torch.uint8):
    item = torch.empty((), dtype=dtype).element_size()
    return torch.empty(max(1, (nbytes + item - 1) // item), dtype=dtype, device=device)


def alloc_quant(fmt: Fmt, rows: int, K: int, layout: Layout, device) -> dict:
    """Torch buffers sized by the library's own size queries."""
    out = {"codes": _empty(qlin_codes_bytes(fmt, rows, K), device)}
    sb = qlin_scales_bytes(fmt, layout, rows, K)
    if fmt in (Fmt.FP8_TENSOR, Fmt.FP8_TOKEN, Fmt.FP8_BLOCK128, Fmt.FP8_GROUP128, Fmt.INT8_ROW):
        out["scales"] = _empty(sb, device, torch.float32)
    elif fmt in (Fmt.INT4_G128_ASYM, Fmt.INT4_G128_SYM):
        out["scales"] = _empty(sb, device, torch.int16)
        out["zeros"] = _empty(qlin_zeros_bytes(fmt, rows, K), device, torch.int32)
    else:
        out["scales"] = _empty(sb, device)
    gb = qlin_global_bytes(fmt, rows, K)
    if gb:
        out["global"] = _empty(gb, device, torch.float32)
    wsb = qlin_quant_workspace_bytes(fmt, rows, K)
    out["workspace"] = _empty(wsb, device, torch.float32) if wsb else None
    out["workspace_bytes"] = wsb
    return out


def quantize_weight(fmt: Fmt, w: torch.Tensor, layout: Layout = Layout.CANONICAL, bufs: dict | None = None,
                    status: torch.Tensor | None = None, stream=None) -> dict:
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.stride(1) == 1
    N, K = w.shape
    b = bufs if bufs is not None else alloc_quant(fmt, N, K, layout, w.device)
    _check_quant_bufs(fmt, N, K, layout, b)
    rc = qlin_quantize_weight(fmt, w.data_ptr(), N, K, w.stride(0), b["codes"].data_ptr(), b["scales"].data_ptr(),
                              _ptr(b.get("zeros")), _ptr(b.get("global")), layout, _ptr(b["workspace"]),
                              b["workspace_bytes"], _ptr(status if status is not None else device_status(w.device)),
                              _stream(stream))
    _check(rc, "qlin_quantize_weight")
    return b


def quantize_act(fmt: Fmt, x: torch.Tensor, layout: Layout = Layout.CANONICAL, bufs: dict | None = None,
                 status: torch.Tensor | None = None, stream=None) -> dict:
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    b = bufs if bufs is not None else alloc_quant(fmt, M, K, layout, x.device)
    _check_quant_bufs(fmt, M, K, layout, b)
    rc = qlin_quantize_act(fmt, x.data_ptr(), M, K, x.stride(0), b["codes"].data_ptr(), b["scales"].data_ptr(),
                           _ptr(b.get("global")), layout, _ptr(b["workspace"]), b["workspace_bytes"],
                           _ptr(status if status is not None else device_status(x.device)), _stream(stream))
    _check(rc, "qlin_quantize_act")
    return b


def gemm(w_fmt: Fmt, x_fmt: Fmt, M: int, N: int, K: int, x, x_scales, w_codes, w_scales, *, x_global=None,
         w_zeros=None, w_global=None, bias=None, y=None, layout: Layout = Layout.CANONICAL, workspace=None,
         status=None, stream=None) -> torch.Tensor:
    dev = w_codes.device
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    # the kernels write Y[M, N] with leading dimension y.stride(0) and read every operand in full
    if y.dtype != torch.bfloat16 or tuple(y.shape) != (M, N) or y.stride(1) != 1:
        raise ValueError(f"y: a bf16 [{M}, {N}] matrix with unit column stride is required")
    if x_fmt == Fmt.BF16:
        if x.dtype != torch.bfloat16 or tuple(x.shape) != (M, K) or not x.is_contiguous():
            raise ValueError(f"x: contiguous bf16 [{M}, {K}] activations are required")
    else:
        _need(x, qlin_codes_bytes(x_fmt, M, K), "x codes")
        _need(x_scales, qlin_scales_bytes(x_fmt, layout, M, K), "x_scales")
        _need(x_global, qlin_global_bytes(x_fmt, M, K), "x_global")
    _need(w_codes, qlin_codes_bytes(w_fmt, N, K), "w_codes")
    _need(w_scales, qlin_scales_bytes(w_fmt, layout, N, K), "w_scales")
    _need(w_zeros, qlin_zeros_bytes(w_fmt, N, K), "w_zeros")
    _need(w_global, qlin_global_bytes(w_fmt, N, K), "w_global")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.numel() < N or not bias.is_contiguous()):
        raise ValueError(f"bias: {N} contiguous bf16 values are required")
    wsb = qlin_gemm_workspace_bytes(w_fmt, x_fmt, M, N, K)
    if workspace is None:
        if wsb:
            workspace = _empty(wsb, dev)
    else:
        _need(workspace, wsb, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = qlin_gemm(w_fmt, x_fmt, M, N, K, x.data_ptr(), _ptr(x_scales), _ptr(x_global), w_codes.data_ptr(),
                   _ptr(w_scales), _ptr(w_zeros), _ptr(w_global), _ptr(bias), y.data_ptr(), y.stride(0), layout,
                   _ptr(workspace), ws_bytes,
                   _ptr(status if status is not None else device_status(dev)), _stream(stream))
    _check(rc, "qlin_gemm")
    return y
