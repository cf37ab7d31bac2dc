// C ABI: argument validation, buffer-size queries and dispatch to the
// kernels.  Nothing here allocates, synchronizes or falls back to another
// path: a call that cannot run returns an error code before any launch.
#include <cuda_runtime.h>

#include "qlin_internal.h"

using namespace qlin;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_quant_format(qlin_format f) {
    return (f >= QLIN_FP8_TENSOR && f <= QLIN_INT4_G128_ASYM) || f == QLIN_MXFP4 || f == QLIN_FP8_GROUP128 ||
           f == QLIN_INT8_ROW || f == QLIN_INT4_G128_SYM || f == QLIN_MXFP4_DUAL;
}

bool is_int4(qlin_format f) { return f == QLIN_INT4_G128_ASYM || f == QLIN_INT4_G128_SYM;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

thread_local int g_last_cuda_error = 0;   // the calling thread's last failed CUDA call (cudaError_t)

qlin_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return QLIN_OK;
    g_last_cuda_error = (int)e;
    return QLIN_ERR_CUDA;
}

// Shape rules per format (see qlin.h).
qlin_status check_quant_shape(qlin_format fmt, qlin_scale_layout layout, int64_t rows, int64_t K) {
    if (rows < 1 || K < 8 || (K & 7) || rows > 0x7FFFFFFFll || K > 0x7FFFFFFFll) return QLIN_ERR_INVALID_ARG;
    if (layout != QLIN_SCALE_CANONICAL && layout != QLIN_SCALE_MMA) return QLIN_ERR_INVALID_ARG;
    // the tensor-amax walks number their 256-element row tasks in 32 bits
    const int64_t rows_pad = layout == QLIN_SCALE_MMA ? ceil_div(rows, 128) * 128 : rows;
    if (rows_pad * ceil_div(K, 256) > 0x7FFFFFFFll) return QLIN_ERR_INVALID_ARG;
    if (layout == QLIN_SCALE_MMA && fmt != QLIN_MXFP8 && fmt != QLIN_MXFP4 && fmt != QLIN_NVFP4 &&
        fmt != QLIN_MXFP4_DUAL)
        return QLIN_ERR_UNSUPPORTED;
    // the row-chunk walks (1 x 128 groups, MX, NVFP4) put a row's 1024-element chunks on grid y
    if ((fmt == QLIN_FP8_GROUP128 || fmt == QLIN_MXFP8 || fmt == QLIN_MXFP4 || fmt == QLIN_NVFP4 ||
         fmt == QLIN_MXFP4_DUAL) &&
        ceil_div(K, 1024) > 65535)
        return QLIN_ERR_INVALID_ARG;
    switch (fmt) {
        case QLIN_FP8_TENSOR:
        case QLIN_FP8_TOKEN:
        case QLIN_INT8_ROW: return QLIN_OK;
        case QLIN_FP8_BLOCK128: return (rows % 128 || K % 128) ? QLIN_ERR_INVALID_ARG : QLIN_OK;
        case QLIN_FP8_GROUP128: return (K % 128) ? QLIN_ERR_INVALID_ARG : QLIN_OK;
        case QLIN_MXFP8:
        case QLIN_MXFP4:
            if (K % 32) return QLIN_ERR_INVALID_ARG;
            return (layout == QLIN_SCALE_MMA && K % 128) ? QLIN_ERR_INVALID_ARG : QLIN_OK;
        case QLIN_NVFP4:
            if (K % 16) return QLIN_ERR_INVALID_ARG;
            return (layout == QLIN_SCALE_MMA && K % 64) ? QLIN_ERR_INVALID_ARG : QLIN_OK;
        case QLIN_MXFP4_DUAL: return (K % 512) ? QLIN_ERR_INVALID_ARG : QLIN_OK;
        case QLIN_INT4_G128_ASYM:
        case QLIN_INT4_G128_SYM: return (rows % 8 || K % 128) ? QLIN_ERR_INVALID_ARG : QLIN_OK;
        default: return QLIN_ERR_UNSUPPORTED;
    }
}

qlin_status quantize(qlin_format fmt, const void* src, int64_t rows, int64_t K, int64_t ld, void* codes,
                     void* scales, void* zeros, float* global, qlin_scale_layout layout, void* ws,
                     size_t ws_bytes, cudaStream_t st) {
    if (!is_quant_format(fmt)) return QLIN_ERR_UNSUPPORTED;
    qlin_status s = check_quant_shape(fmt, layout, rows, K);
    if (s != QLIN_OK) return s;
    if (!src || !codes || !scales || ld < K) return QLIN_ERR_INVALID_ARG;
    if (is_int4(fmt) && !zeros) return QLIN_ERR_INVALID_ARG;
    if ((fmt == QLIN_NVFP4 || fmt == QLIN_MXFP4_DUAL) && !global) return QLIN_ERR_INVALID_ARG;
    if (fmt == QLIN_MXFP4_DUAL && (reinterpret_cast<uintptr_t>(global) & 3u)) return QLIN_ERR_ALIGNMENT;
    if (!aligned16(src) || (ld * 2) % 16 || !aligned16(codes)) return QLIN_ERR_ALIGNMENT;
    if (fmt == QLIN_FP8_TOKEN || fmt == QLIN_FP8_BLOCK128 || fmt == QLIN_FP8_TENSOR || fmt == QLIN_FP8_GROUP128 ||
        fmt == QLIN_INT8_ROW) {
        if (reinterpret_cast<uintptr_t>(scales) & 3u) return QLIN_ERR_ALIGNMENT;
    }
    if (is_int4(fmt) &&
        ((reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(zeros) & 3u)))
        return QLIN_ERR_ALIGNMENT;
    const size_t need = qlin_quant_workspace_bytes(fmt, rows, K);
    if (need && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 3u))) return QLIN_ERR_WORKSPACE;

    const uint16_t* x = static_cast<const uint16_t*>(src);
    uint8_t* c = static_cast<uint8_t*>(codes);
    const bool mma = layout == QLIN_SCALE_MMA;
    switch (fmt) {
        case QLIN_FP8_TENSOR:
            return launch_status(launch_fp8_tensor(x, rows, K, ld, c, static_cast<float*>(scales),
                                                   static_cast<float*>(ws), amax_partials(rows, K), st));
        case QLIN_FP8_TOKEN:
            return launch_status(launch_fp8_rowwise(x, rows, K, ld, c, static_cast<float*>(scales), st));
        case QLIN_INT8_ROW:
            return launch_status(launch_int8_rowwise(x, rows, K, ld, c, static_cast<float*>(scales), st));
        case QLIN_FP8_BLOCK128:
            return launch_status(launch_fp8_block128(x, rows, K, ld, c, static_cast<float*>(scales), st));
        case QLIN_FP8_GROUP128:
            return launch_status(launch_fp8_group128(x, rows, K, ld, c, static_cast<float*>(scales), st));
        case QLIN_MXFP8:
            return launch_status(launch_mxfp8(x, rows, K, ld, c, static_cast<uint8_t*>(scales), mma, st));
        case QLIN_MXFP4:
            return launch_status(launch_mxfp4(x, rows, K, ld, c, static_cast<uint8_t*>(scales), mma, st));
        case QLIN_MXFP4_DUAL:
            return launch_status(launch_mxfp4_dual(x, rows, K, ld, c, static_cast<uint8_t*>(scales), global, mma, st));
        case QLIN_NVFP4:
            return launch_status(launch_nvfp4(x, rows, K, ld, c, static_cast<uint8_t*>(scales), global, mma,
                                              static_cast<float*>(ws), amax_partials(rows, K), st));
        case QLIN_INT4_G128_ASYM:
        case QLIN_INT4_G128_SYM:
            return launch_status(launch_int4_g128(x, rows, K, ld, reinterpret_cast<int32_t*>(codes),
                                                  static_cast<uint16_t*>(scales), static_cast<int32_t*>(zeros),
                                                  fmt == QLIN_INT4_G128_SYM, st));
        default: return QLIN_ERR_UNSUPPORTED;
    }
}

}  // namespace

extern "C" {

const char* qlin_status_string(qlin_status s) {
    switch (s) {
        case QLIN_OK: return "ok";
        case QLIN_ERR_INVALID_ARG: return "invalid argument (null pointer, size or leading dimension)";
        case QLIN_ERR_UNSUPPORTED: return "unsupported format, layout or format pair";
        case QLIN_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
        case QLIN_ERR_WORKSPACE: return "workspace missing or too small";
        case QLIN_ERR_CUDA: return "CUDA launch or call failed";
        case QLIN_ERR_DEVICE_TIMEOUT: return "a bounded device wait expired";
        default: return "unknown status";
    }
}

const char* qlin_version(void) { return "qlin 0.1 sm_103a"; }

int qlin_last_cuda_error(void) { return g_last_cuda_error; }

size_t qlin_codes_bytes(qlin_format fmt, int64_t rows, int64_t K) {
    if (rows < 1 || K < 1) return 0;
    switch (fmt) {
        case QLIN_FP8_TENSOR:
        case QLIN_FP8_TOKEN:
        case QLIN_FP8_BLOCK128:
        case QLIN_FP8_GROUP128:
        case QLIN_INT8_ROW:
        case QLIN_MXFP8: return (size_t)(rows * K);
        case QLIN_NVFP4:
        case QLIN_MXFP4:
        case QLIN_MXFP4_DUAL: return (size_t)(rows * (K / 2));
        case QLIN_INT4_G128_ASYM:
        case QLIN_INT4_G128_SYM: return (size_t)((K / 8) * rows * 4);
        default: return 0;
    }
}

size_t qlin_scales_bytes(qlin_format fmt, qlin_scale_layout layout, int64_t rows, int64_t K) {
    if (rows < 1 || K < 1) return 0;
    const int64_t rows_pad = ceil_div(rows, 128) * 128;
    switch (fmt) {
        case QLIN_FP8_TENSOR: return 4;
        case QLIN_FP8_TOKEN:
        case QLIN_INT8_ROW: return (size_t)(rows * 4);
        case QLIN_FP8_BLOCK128: return (size_t)((rows / 128) * (K / 128) * 4);
        case QLIN_FP8_GROUP128: return (size_t)(rows * (K / 128) * 4);
        case QLIN_MXFP8:
        case QLIN_MXFP4:
        case QLIN_MXFP4_DUAL: return (size_t)((layout == QLIN_SCALE_MMA ? rows_pad : rows) * (K / 32));
        case QLIN_NVFP4: return (size_t)((layout == QLIN_SCALE_MMA ? rows_pad : rows) * (K / 16));
        case QLIN_INT4_G128_ASYM:
        case QLIN_INT4_G128_SYM: return (size_t)((K / 128) * rows * 2);
        default: return 0;
    }
}

size_t qlin_zeros_bytes(qlin_format fmt, int64_t rows, int64_t K) {
    if (!is_int4(fmt) || rows < 1 || K < 1) return 0;
    return (size_t)((K / 128) * (rows / 8) * 4);
}

size_t qlin_global_bytes(qlin_format fmt, int64_t rows, int64_t K) {
    if (rows < 1 || K < 1) return 0;
    if (fmt == QLIN_NVFP4) return 4;
    if (fmt == QLIN_MXFP4_DUAL) return (size_t)(rows * (K / 512) * 4);
    return 0;
}

size_t qlin_quant_workspace_bytes(qlin_format fmt, int64_t rows, int64_t K) {
    if (rows < 1 || K < 1) return 0;
    if (fmt == QLIN_FP8_TENSOR || fmt == QLIN_NVFP4) return (size_t)amax_partials(rows, K) * sizeof(float);
    return 0;
}

size_t qlin_gemm_workspace_bytes(qlin_format w_fmt, qlin_format x_fmt, int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1) return 0;
    if (is_int4(w_fmt) && x_fmt == QLIN_BF16) return w4a16_workspace_bytes(M, N, K);
    return 0;
}

qlin_status qlin_quantize_weight(qlin_format fmt, const void* w_bf16_dev, int64_t N, int64_t K, int64_t ldw,
                                 void* codes_dev, void* scales_dev, void* zeros_dev, float* global_dev,
                                 qlin_scale_layout layout, void* workspace_dev, size_t workspace_bytes,
                                 int* dev_status_dev, qlin_stream_t stream) {
    (void)dev_status_dev;   // the quantizers have no device-side waits
    return quantize(fmt, w_bf16_dev, N, K, ldw, codes_dev, scales_dev, zeros_dev, global_dev, layout,
                    workspace_dev, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status qlin_quantize_act(qlin_format fmt, const void* x_bf16_dev, int64_t M, int64_t K, int64_t ldx,
                              void* codes_dev, void* scales_dev, float* global_dev, qlin_scale_layout layout,
                              void* workspace_dev, size_t workspace_bytes, int* dev_status_dev,
                              qlin_stream_t stream) {
    (void)dev_status_dev;
    if (is_int4(fmt)) return QLIN_ERR_UNSUPPORTED;   // int4 is weight-only (W4A16)
    return quantize(fmt, x_bf16_dev, M, K, ldx, codes_dev, scales_dev, nullptr, global_dev, layout,
                    workspace_dev, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status qlin_gemm(qlin_format w_fmt, qlin_format x_fmt, int64_t M, int64_t N, int64_t K, const void* x_dev,
                      const void* x_scales_dev, const float* x_global_dev, const void* w_codes_dev,
                      const void* w_scales_dev, const void* w_zeros_dev, const float* w_global_dev,
                      const void* bias_bf16_dev, void* y_bf16_dev, int64_t ldy, qlin_scale_layout layout,
                      void* workspace_dev, size_t workspace_bytes, int* dev_status_dev, qlin_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (M < 1 || N < 1 || K < 1 || M > 0x7FFFFFFFll || N > 0x7FFFFFFFll || K > 0x7FFFFFFFll || ldy < N)
        return QLIN_ERR_INVALID_ARG;
    // the kernels count K and the 128 x 128 output tiles in 32 bits
    if (ceil_div(M, 128) * ceil_div(N, 128) > 0x7FFFFFFFll) return QLIN_ERR_INVALID_ARG;
    if (!x_dev || !w_codes_dev || !y_bf16_dev) return QLIN_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(w_codes_dev) || !aligned16(y_bf16_dev) || (ldy * 2) % 16 ||
        (bias_bf16_dev && !aligned16(bias_bf16_dev)))
        return QLIN_ERR_ALIGNMENT;
    GemmArgs a{M, N, K, ldy, x_dev, x_scales_dev, x_global_dev, w_codes_dev, w_scales_dev, w_zeros_dev,
               w_global_dev, static_cast<const uint16_t*>(bias_bf16_dev), static_cast<uint16_t*>(y_bf16_dev),
               workspace_dev, workspace_bytes, dev_status_dev, /*x_group128=*/false};
    if (w_fmt == QLIN_FP8_TENSOR && x_fmt == QLIN_FP8_TENSOR) {
        if (!x_scales_dev || !w_scales_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 16) return QLIN_ERR_INVALID_ARG;
        return launch_status(launch_gemm_fp8_tensor(a, st));
    }
    if (w_fmt == QLIN_FP8_BLOCK128 && (x_fmt == QLIN_FP8_TOKEN || x_fmt == QLIN_FP8_GROUP128)) {
        if (!x_scales_dev || !w_scales_dev) return QLIN_ERR_INVALID_ARG;
        if (N % 128 || K % 128) return QLIN_ERR_INVALID_ARG;
        a.x_group128 = (x_fmt == QLIN_FP8_GROUP128);
        return launch_status(launch_gemm_fp8_block(a, st));
    }
    if (w_fmt == QLIN_MXFP8 && x_fmt == QLIN_MXFP8) {
        if (layout != QLIN_SCALE_MMA) return QLIN_ERR_UNSUPPORTED;
        if (!x_scales_dev || !w_scales_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 128) return QLIN_ERR_INVALID_ARG;
        if (!aligned16(x_scales_dev) || !aligned16(w_scales_dev)) return QLIN_ERR_ALIGNMENT;
        return launch_status(launch_gemm_mxfp8(a, st));
    }
    if (w_fmt == QLIN_MXFP4 && x_fmt == QLIN_MXFP4) {
        if (layout != QLIN_SCALE_MMA) return QLIN_ERR_UNSUPPORTED;
        if (!x_scales_dev || !w_scales_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 256) return QLIN_ERR_INVALID_ARG;
        if (!aligned16(x_scales_dev) || !aligned16(w_scales_dev)) return QLIN_ERR_ALIGNMENT;
        return launch_status(launch_gemm_mxfp4(a, st));
    }
    if (w_fmt == QLIN_MXFP4_DUAL && x_fmt == QLIN_MXFP4_DUAL) {
        if (layout != QLIN_SCALE_MMA) return QLIN_ERR_UNSUPPORTED;
        if (!x_scales_dev || !w_scales_dev || !x_global_dev || !w_global_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 512) return QLIN_ERR_INVALID_ARG;
        if (!aligned16(x_scales_dev) || !aligned16(w_scales_dev) ||
            (reinterpret_cast<uintptr_t>(x_global_dev) & 3u) || (reinterpret_cast<uintptr_t>(w_global_dev) & 3u))
            return QLIN_ERR_ALIGNMENT;
        return launch_status(launch_gemm_mxfp4_dual(a, st));
    }
    if (w_fmt == QLIN_NVFP4 && x_fmt == QLIN_NVFP4) {
        if (layout != QLIN_SCALE_MMA) return QLIN_ERR_UNSUPPORTED;
        if (!x_scales_dev || !w_scales_dev || !x_global_dev || !w_global_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 256) return QLIN_ERR_INVALID_ARG;
        if (!aligned16(x_scales_dev) || !aligned16(w_scales_dev)) return QLIN_ERR_ALIGNMENT;
        return launch_status(launch_gemm_nvfp4(a, st));
    }
    if (w_fmt == QLIN_FP8_TENSOR && x_fmt == QLIN_BF16) {
        // activation quantization fused into the GEMM: single-request row counts
        if (!w_scales_dev) return QLIN_ERR_INVALID_ARG;
        if (M > 128) return QLIN_ERR_UNSUPPORTED;
        if (K % 16) return QLIN_ERR_INVALID_ARG;
        return launch_status(launch_gemm_fp8_tensor_fused_x(a, st));
    }
    if (w_fmt == QLIN_INT8_ROW && x_fmt == QLIN_INT8_ROW) {
        if (!x_scales_dev || !w_scales_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 16) return QLIN_ERR_INVALID_ARG;
        return launch_status(launch_gemm_int8(a, st));
    }
    if (is_int4(w_fmt) && x_fmt == QLIN_BF16) {      // the stored zero points serve both int4 variants
        if (!w_scales_dev || !w_zeros_dev) return QLIN_ERR_INVALID_ARG;
        if (K % 128 || N % 8) return QLIN_ERR_INVALID_ARG;
        // 128-channel tiles and 64-token tiles run on grid dimensions y and z (at most 65535 each)
        if (ceil_div(N, 128) > 65535 || ceil_div(M, 64) > 65535) return QLIN_ERR_INVALID_ARG;
        const size_t need = w4a16_workspace_bytes(M, N, K);
        if (need && (!workspace_dev || workspace_bytes < need || !aligned16(workspace_dev)))
            return QLIN_ERR_WORKSPACE;
        return launch_status(launch_gemm_w4a16(a, st));
    }
    return QLIN_ERR_UNSUPPORTED;
}

qlin_status qlin_debug_expire_wait(int* dev_status_dev, uint32_t max_polls, qlin_stream_t stream) {
    if (!dev_status_dev) return QLIN_ERR_INVALID_ARG;
    return launch_status(launch_debug_expire_wait(dev_status_dev, max_polls, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
