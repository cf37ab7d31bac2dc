/*
 * qlin.h -- C ABI of the GB300 (sm_103a) quantized-linear library.
 *
 * The operations are the online-quantization linear method of
 * "vLLM-Omni 在线量化（Online Quantization）完全指南：加载期动态量化 FP8 / Int8 /
 * MXFP8 / MXFP4", section "在线量化的底层工作原理":
 *   stage 2  the BF16 weight is quantized once after loading
 *            (process_weights_after_loading)        -> qlin_quantize_weight
 *   stage 3  every call quantizes the activation dynamically
 *            (_quantize_activation)                 -> qlin_quantize_act
 *            and runs the quantized matmul
 *            (_quant_matmul)                        -> qlin_gemm
 * The callers flatten 3-D activations to 2-D first, as the same stage's
 * apply() skeleton does.  Formats and granularities:
 *   FP8 per-tensor / per-token / 128x128 block: "[vLLM] 기타 양자화: FP8,
 *     ModelOpt, INC, TorchAO, Quark", section "FP8: vLLM의 핵심 양자화".
 *   MXFP8 (E8M0 scale per 32 K elements): stage 2 of the section above.
 *   NVFP4 (mixed FP8/NVFP4 linears): "vLLM-Omni 量化推理实践", Table 1.
 *   int4 asymmetric, group 128, auto_gptq packing, round-to-nearest
 *     ("--iters 0"): "vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다",
 *     section "새로운 모델 양자화".
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers; the caller owns all memory
 *     (inputs, outputs, workspace).  Entry points that take a stream never
 *     allocate, never synchronize and never fall back to another path; they
 *     enqueue kernels on `stream` and return.
 *   - Matrices are row-major with the leading dimension in ELEMENTS.  X is
 *     [M, K] (activations), W is [N, K] (nn.Linear weight), Y is [M, N].
 *   - The return value covers host-side validation and launch errors only.
 *     `dev_status_dev` (optional, may be NULL) is a device int that the
 *     caller zeroes; a kernel writes QLIN_ERR_DEVICE_TIMEOUT into it if one
 *     of its bounded waits gives up.  Such a kernel leaves its outputs
 *     unspecified but returns, and the context stays usable.
 *   - Inputs are finite.  NaN or Inf inputs give unspecified codes.
 *   - One device per process.  The first qlin_gemm call of each format pair
 *     sets that kernel's shared-memory size on the device current at the
 *     time, and later calls skip the step.  A call on another device of the
 *     same process then fails to launch and returns QLIN_ERR_CUDA; nothing is
 *     written.  Calls from several host threads at once, each on its own
 *     stream and buffers, are safe, first calls included: the one-time
 *     setups (device queries, driver entry-point lookups, kernel attributes)
 *     are thread-safe and idempotent.  The exception is
 *     qlin_quantize_fp8_tensor_noalloc, whose calls share one device array:
 *     calls that overlap on the GPU must not be issued (see its entry).
 *
 * Numeric rules (bit-exact; the pages name the formats but print no formula,
 * so these are the plainest readings of the public format definitions):
 *   FP8 (tensor, token, block): s = amax/448, code = E4M3(x * (448/amax)),
 *     s = 1 and multiplier 1 when amax == 0.
 *   MXFP8: e = clamp(floor(log2 amax) - 8, -127, 127); scale code e + 127;
 *     code = E4M3(x * 2^-e).
 *   NVFP4: g = A/2688 (A = tensor amax); block scale sb = UE4M3(b * (448/A));
 *     code = E2M1(x * ((2688/A)/dec(sb))), 0 when dec(sb) == 0.
 *   INT4: per (n, group of 128 k): range [min(0,min), max(0,max)],
 *     s = bf16((max-min)/15) (1 if 0), r = 1/s in fp32, z = clamp(rint(-min*r)),
 *     q = clamp(rint(x*r) + z), clamps to [0, 15].  INT4_SYM: the same with
 *     max = a, min = -a (a = max |x|) and z = 8.
 *   INT8 (per row): s = amax/127, code = clamp(rint(x * (127/amax)), -127,
 *     127), s = 1 and multiplier 1 when amax == 0.
 *   MXFP4_DUAL: per 512 K, c = A/6 and r = 6/A (1, 1 when A == 0); v = x * r;
 *     per 32, e = clamp(floor(log2 max|v|) - 2, -127, 127), code =
 *     E2M1(v * 2^-e); dequant dec(code) * 2^e * c.
 *   Conversions round to nearest even and saturate (satfinite); a zero keeps
 *   its sign.  Every fp32 operation is a single correctly rounded op.
 */
#ifndef QLIN_H
#define QLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qlin_stream_t;   /* same handle as cudaStream_t */

typedef enum {
    QLIN_FP8_TENSOR = 0,     /* E4M3 codes, one fp32 scale for the tensor          */
    QLIN_FP8_TOKEN = 1,      /* E4M3 codes, one fp32 scale per row                 */
    QLIN_FP8_BLOCK128 = 2,   /* E4M3 codes, one fp32 scale per 128x128 tile        */
    QLIN_MXFP8 = 3,          /* E4M3 codes, one E8M0 scale byte per 32 along K     */
    QLIN_NVFP4 = 4,          /* E2M1 codes 2/byte, UE4M3 per 16, fp32 per tensor   */
    QLIN_INT4_G128_ASYM = 5, /* uint4 codes 8/int32, bf16 scale + uint4 zero / 128 */
    QLIN_BF16 = 6,           /* unquantized bf16 (the activation side of W4A16)    */
    /* E2M1 codes 2/byte (lower k in the low nibble), one E8M0 scale byte per
     * 32 along K by the MX shared-exponent rule with the E2M1 element:
     * "vLLM-Omni 在线量化（Online Quantization）完全指南", section
     * "在线量化的底层工作原理" (the online MXFP4 path mirrors MXFP8 with
     * float4_e2m1fn_x2 codes; W4A4).                                          */
    QLIN_MXFP4 = 7,
    /* E4M3 codes, one fp32 scale per row and 128 consecutive K (1 x 128
     * groups): the block-128 dynamic symmetric FP8 scheme of "[vLLM] 기타
     * 양자화: FP8, ModelOpt, INC, TorchAO, Quark", section "FP8: vLLM의 핵심
     * 양자화", on activations; pairs with FP8_BLOCK128 weights in qlin_gemm.   */
    QLIN_FP8_GROUP128 = 8,
    /* int8 codes (two's complement), one fp32 scale per row: per output
     * channel for a weight, per token for an activation.  The CUDA online
     * INT8 W8A8 path of "vLLM-Omni 在线量化（Online Quantization）完全指南",
     * section "在线量化的底层工作原理" (weights and their scales from a scaled
     * int8 quantizer), with the dynamic activation scheme of section
     * "核心参数详解"; pairs with itself in qlin_gemm.                           */
    QLIN_INT8_ROW = 9,
    /* int4 symmetric, group 128 along K: the "sym": true variant of the
     * AutoRound page's checkpoint config ("vLLM-Omni는 AutoRound 양자화로
     * 추론을 가속화합니다", section "새로운 모델 양자화").  Range [-a, a] with
     * a = max |x| over the group, scale bf16(2a/15), zero point fixed at 8;
     * stored exactly like QLIN_INT4_G128_ASYM (qzeros all 8), so qlin_gemm
     * takes it with bf16 activations through the same W4A16 kernels.         */
    QLIN_INT4_G128_SYM = 10,
    /* MXFP4 with two scale levels: a coarse fp32 scale per 512 consecutive K
     * (A/6, A the amax of the 512) and, on the values divided by it, the MX
     * shared exponent per 32 (E8M0 bytes, as QLIN_MXFP4); E2M1 codes two per
     * byte.  The online mxfp4_dualscale path of "vLLM-Omni 在线量化（Online
     * Quantization）完全指南", section "在线量化的底层工作原理" (per-32 fine and
     * per-512 coarse levels computed at run time, the calibrated mul_scale
     * absent and taken as ones).  The coarse scales go in the `global`
     * buffer: float [rows, K/512].  Pairs with itself in qlin_gemm.           */
    QLIN_MXFP4_DUAL = 11
} qlin_format;

typedef enum {
    /* Row-major [rows, K/G] scale tensor (G = 32 MXFP8 / MXFP4, 16 NVFP4).   */
    QLIN_SCALE_CANONICAL = 0,
    /* Tensor-core-ready tiling, MXFP8, MXFP4 and NVFP4 only: for each 128-row tile
     * (rows padded up to a multiple of 128 with scale code 0) and each chunk
     * of 4 consecutive scales along K, 512 contiguous bytes; the scale of
     * row r (r < 128 within the tile) and chunk position j (0..3) sits at
     * byte 16*(r % 32) + 4*(r / 32) + j.  Tiles are ordered
     * [row_tile][k_chunk].  This is the layout qlin_gemm consumes.            */
    QLIN_SCALE_MMA = 1
} qlin_scale_layout;

typedef enum {
    QLIN_OK = 0,
    QLIN_ERR_INVALID_ARG = 1,    /* null pointer, bad size or leading dimension */
    QLIN_ERR_UNSUPPORTED = 2,    /* format / layout / pair not provided          */
    QLIN_ERR_ALIGNMENT = 3,      /* a pointer or stride breaks the 16-byte rule  */
    QLIN_ERR_WORKSPACE = 4,      /* workspace missing or smaller than required   */
    QLIN_ERR_CUDA = 5,           /* a CUDA call or launch failed                 */
    QLIN_ERR_DEVICE_TIMEOUT = 6  /* written to dev_status by a kernel whose bounded wait expired */
} qlin_status;

const char *qlin_status_string(qlin_status s);

/* ---------------------------------------------------------------- sizes
 * Byte sizes of the buffers the quantizers write, for `rows` rows of K
 * elements (rows = N for weights, M for activations).  0 means "not used by
 * this format" or invalid arguments.  The layouts are those of the formats'
 * sources cited above (the GPTQ packing of the int4 page's
 * auto_round:auto_gptq format; the E8M0 and UE4M3 scale bytes of the MX and
 * NVFP4 formats).                                                           */

/* Codes: FP8 formats and INT8_ROW rows*K; NVFP4 and MXFP4 rows*K/2 (lower k in the low nibble);
 * INT4 (both variants) (K/8)*rows*4 as int32 [K/8, rows], k = 8i+j in bits [4j,4j+4). */
size_t qlin_codes_bytes(qlin_format fmt, int64_t rows, int64_t K);

/* Scales: FP8_TENSOR 4 (one float); FP8_TOKEN and INT8_ROW rows*4; FP8_GROUP128
 * rows*(K/128)*4, float [rows, K/128] row-major; FP8_BLOCK128
 * (rows/128)*(K/128)*4 row-major; MXFP8 rows*K/32 (canonical) or
 * ceil(rows/128)*128*K/32 (MMA), the same for MXFP4; NVFP4 rows*K/16 or
 * ceil(rows/128)*128*K/16;
 * INT4 (K/128)*rows*2, bf16 [K/128, rows].                                  */
size_t qlin_scales_bytes(qlin_format fmt, qlin_scale_layout layout, int64_t rows, int64_t K);

/* Zero points: INT4 only, (K/128)*(rows/8)*4 as int32 [K/128, rows/8],
 * n = 8i+j in bits [4j,4j+4); no "-1" offset is applied.                     */
size_t qlin_zeros_bytes(qlin_format fmt, int64_t rows, int64_t K);

/* Second-level scale buffer (`global`): NVFP4 4 bytes (one float, the
 * per-tensor scale); MXFP4_DUAL rows*(K/512)*4 (float [rows, K/512], the
 * coarse scales); 0 otherwise.                                              */
size_t qlin_global_bytes(qlin_format fmt, int64_t rows, int64_t K);

/* Workspace (device scratch) a quantizer call needs: the per-tensor
 * formats (FP8_TENSOR, NVFP4) keep one float per reduction block; others 0. */
size_t qlin_quant_workspace_bytes(qlin_format fmt, int64_t rows, int64_t K);

/* Workspace a qlin_gemm call needs for this pair and shape.  Every GEMM
 * here returns 0: the W4A16 split-K reduction runs through distributed
 * shared memory inside a thread-block cluster.                             */
size_t qlin_gemm_workspace_bytes(qlin_format w_fmt, qlin_format x_fmt,
                                 int64_t M, int64_t N, int64_t K);

/* ---------------------------------------------------------------- quantizers
 * Quantize a bf16 matrix src[rows, K] (leading dimension ld >= K, elements)
 * into caller-owned buffers, on `stream`.  Both entry points apply the
 * numeric rules above; they differ in where the pages place them (below).
 *   codes_dev          qlin_codes_bytes(fmt, rows, K) bytes, 16-byte aligned
 *   scales_dev         qlin_scales_bytes(fmt, layout, rows, K) bytes
 *   zeros_dev          INT4 only (else NULL)
 *   global_dev         NVFP4: one float, the per-tensor scale g; MXFP4_DUAL:
 *                      the coarse scales, qlin_global_bytes(...) bytes
 *   layout             QLIN_SCALE_MMA is accepted for MXFP8, MXFP4, MXFP4_DUAL and NVFP4 only
 *   workspace_dev      qlin_quant_workspace_bytes(...) bytes (NULL if 0)
 * Requirements: src and ld*2 bytes 16-byte aligned; K % 8 == 0;
 *   rows < 2^31, K < 2^31 and rows' * ceil(K/256) < 2^31, rows' being rows
 *   rounded up to a multiple of 128 for the MMA layout (about 1 TB of bf16);
 *   FP8_GROUP128, MXFP8, MXFP4 and NVFP4 also K <= 65535 * 1024;
 *   FP8_BLOCK128: rows % 128 == 0 and K % 128 == 0; FP8_GROUP128: K % 128 == 0;
 *   MXFP8: K % 32 == 0
 *   (K % 128 == 0 for the MMA layout), the same for MXFP4; MXFP4_DUAL: K % 512 == 0;
 *   NVFP4: K % 16 == 0
 *   (K % 64 for MMA);
 *   INT4 (both variants): rows % 8 == 0 and K % 128 == 0.
 * Errors: QLIN_ERR_INVALID_ARG, QLIN_ERR_ALIGNMENT, QLIN_ERR_UNSUPPORTED
 *   (QLIN_BF16, or INT4 through qlin_quantize_act), QLIN_ERR_WORKSPACE,
 *   QLIN_ERR_CUDA.                                                          */
/* Load-time weight quantization, once per weight: "vLLM-Omni 在线量化（Online
 * Quantization）完全指南", section "在线量化的底层工作原理", stage 2 (the BF16
 * weight is quantized after loading, process_weights_after_loading, and the
 * original is released).  Every format except QLIN_BF16; rows = N output
 * channels of W[N, K].                                                      */
qlin_status qlin_quantize_weight(qlin_format fmt, const void *w_bf16_dev, int64_t N, int64_t K,
                                 int64_t ldw, void *codes_dev, void *scales_dev, void *zeros_dev,
                                 float *global_dev, qlin_scale_layout layout, void *workspace_dev,
                                 size_t workspace_bytes, int *dev_status_dev, qlin_stream_t stream);

/* Dynamic activation quantization, every call: the same section, stage 3
 * (_quantize_activation on the flattened input; activation scales are
 * dynamic only, section "核心参数详解").  Every format except QLIN_BF16 and
 * QLIN_INT4_G128_ASYM (int4 is weight-only: W4A16 takes bf16 activations);
 * rows = M tokens of X[M, K].                                               */
qlin_status qlin_quantize_act(qlin_format fmt, const void *x_bf16_dev, int64_t M, int64_t K,
                              int64_t ldx, void *codes_dev, void *scales_dev, float *global_dev,
                              qlin_scale_layout layout, void *workspace_dev, size_t workspace_bytes,
                              int *dev_status_dev, qlin_stream_t stream);

/* ---------------------------------------------------------------- GEMM
 * Y[M, N] (bf16, leading dimension ldy) = sum over k of dequant(X)[m,k] *
 * dequant(W)[n,k], fp32 accumulation, optional bf16 bias[N] added before the
 * final round to bf16 (the fused alpha*(A@B)+bias epilogue of
 * "vLLM-Omni 在线量化（Online Quantization）完全指南" section
 * "在线量化的底层工作原理", FP8 paragraph).
 * Supported (w_fmt, x_fmt) pairs and their operands:
 *   FP8_TENSOR, FP8_TENSOR : x = codes [M,K]; x_scales, w_scales = one float each
 *   FP8_TENSOR, BF16       : activation quantization fused into the GEMM: x =
 *                            bf16 activations [M,K] (M <= 128, else
 *                            QLIN_ERR_UNSUPPORTED), quantized per tensor inside
 *                            the kernel by the FP8_TENSOR rule; x_scales unused;
 *                            w_scales one float; K % 16 == 0.  Y is bit-identical
 *                            to qlin_quantize_act(FP8_TENSOR) followed by the
 *                            FP8_TENSOR pair, in one launch.
 *   FP8_BLOCK128, FP8_TOKEN: x_scales float [M]; w_scales float [N/128, K/128]
 *                            (N % 128 == 0, K % 128 == 0)
 *   FP8_BLOCK128, FP8_GROUP128: x_scales float [M, K/128]; otherwise as above
 *   MXFP8, MXFP8           : scales in QLIN_SCALE_MMA layout (K % 128 == 0)
 *   NVFP4, NVFP4           : scales in QLIN_SCALE_MMA layout, x_global and
 *                            w_global one float each (K % 256 == 0)
 *   MXFP4, MXFP4           : scales in QLIN_SCALE_MMA layout (K % 256 == 0)
 *   MXFP4_DUAL, MXFP4_DUAL : fine scales in QLIN_SCALE_MMA layout, x_global and
 *                            w_global the coarse scales [M, K/512] and
 *                            [N, K/512] (K % 512 == 0); each 512-K partial is
 *                            scaled by x_global[m,b] * w_global[n,b] in fp32
 *   INT8_ROW, INT8_ROW     : x_scales float [M], w_scales float [N] (K % 16 == 0).
 *                            sm_103a has no integer tensor-core MMA, so the
 *                            kernel turns the codes into exact fp16 values on
 *                            chip and multiplies them with fp32 accumulation:
 *                            every product is exact, and so is every partial sum
 *                            below 2^24 in magnitude.
 *   INT4_G128_ASYM, BF16   : (and INT4_G128_SYM, BF16)
 *                            x = bf16 activations [M,K] row-major; w_codes
 *                            qweight, w_scales bf16, w_zeros qzeros (K % 128 == 0,
 *                            N % 8 == 0, N <= 65535*128, M <= 65535*64);
 *                            workspace per qlin_gemm_workspace_bytes
 * Other pairs return QLIN_ERR_UNSUPPORTED.  All operand rows are contiguous
 * (leading dimension K, or K/2 bytes for NVFP4 / MXFP4 codes); ldy >= N and ldy*2
 * bytes 16-byte aligned.  M may be any value >= 1 (the row tail is handled
 * in the kernels; buffers are not padded).  M, N, K < 2^31 and
 * ceil(M/128)*ceil(N/128) < 2^31; larger shapes return QLIN_ERR_INVALID_ARG. */
qlin_status qlin_gemm(qlin_format w_fmt, qlin_format x_fmt, int64_t M, int64_t N, int64_t K,
                      const void *x_dev, const void *x_scales_dev, const float *x_global_dev,
                      const void *w_codes_dev, const void *w_scales_dev, const void *w_zeros_dev,
                      const float *w_global_dev, const void *bias_bf16_dev, void *y_bf16_dev,
                      int64_t ldy, qlin_scale_layout layout, void *workspace_dev,
                      size_t workspace_bytes, int *dev_status_dev, qlin_stream_t stream);

/* ---------------------------------------------------------------- no-allocation variant
 * The pages have no counterpart to this entry point.
 *
 * Per-tensor FP8 quantization (QLIN_FP8_TENSOR rules, same codes and scale
 * as qlin_quantize_act / qlin_quantize_weight) for callers that cannot
 * allocate device memory or hand over a workspace -- for example a plugin
 * inside a serving engine that has already reserved the device memory for its
 * own pool, or code that must keep the memory footprint fixed after start-up.
 * The per-tensor amax partials live in a fixed device array inside the
 * library (QLIN_NOALLOC_MAX_PARTIALS floats, 16 KB), which every device that
 * loads the library holds until exit.  One partial covers 16384 elements, so
 * rows*K may be at most QLIN_NOALLOC_MAX_ELEMENTS; larger tensors return
 * QLIN_ERR_WORKSPACE before any launch.
 *   x_bf16_dev  [rows, K] bf16, leading dimension ld (elements), 16-byte aligned
 *   codes_dev   rows*K E4M3 codes, row-major, 16-byte aligned
 *   scale_dev   one float, the tensor scale s = amax/448
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, so make the first call
 * before any stream capture, and call with the stream's device current.
 * The address is kept per device and context; after cudaDeviceReset the next
 * call looks it up again in the new context (again outside any capture).
 * The array is shared by all calls on a device and keeps the last call's
 * contents (each call rewrites the slots it reads, nothing needs clearing);
 * calls that overlap on the GPU race on it.  Allocates nothing; errors as
 * qlin_quantize_act.                                                        */
#define QLIN_NOALLOC_MAX_PARTIALS 4096
#define QLIN_NOALLOC_MAX_ELEMENTS (4096LL * 16384LL)
qlin_status qlin_quantize_fp8_tensor_noalloc(const void *x_bf16_dev, int64_t rows, int64_t K, int64_t ld,
                                             void *codes_dev, float *scale_dev, qlin_stream_t stream);

/* ---------------------------------------------------------------- diagnostics
 * Runs the library's bounded device wait on an mbarrier that nothing ever
 * completes, with at most `max_polls` polls, then writes
 * QLIN_ERR_DEVICE_TIMEOUT into *dev_status_dev.  Exists so that the timeout
 * path can be exercised without hanging or faulting a GPU.                  */
qlin_status qlin_debug_expire_wait(int *dev_status_dev, uint32_t max_polls, qlin_stream_t stream);

/* The cudaError_t value of the CUDA call that made this thread's most
 * recent QLIN_ERR_CUDA return (0 if none has failed), for diagnostics. */
int qlin_last_cuda_error(void);

/* Library version string, e.g. "qlin 0.1 sm_103a". */
const char *qlin_version(void);

#ifdef __cplusplus
}
#endif
#endif /* QLIN_H */
