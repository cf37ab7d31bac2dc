// Online quantizers: bf16 -> FP8 E4M3 (tensor / token / 1x128 group /
// 128x128 block), MXFP8, MXFP4 (single and dual scale), NVFP4, int4 g128 and
// INT8 per row.  Each
// reads its bf16 input once from HBM in 16-byte vectors, reduces amax (or
// min/max) with warp shuffles, and writes codes and scales in the same pass.
// The per-tensor formats need the tensor amax before any code exists, so they
// add one read-only amax pass.
//
// Formats: "[vLLM] 기타 양자화: FP8, ModelOpt, INC, TorchAO, Quark" section
// "FP8: vLLM의 핵심 양자화" (tensor/token/block-128 dynamic scales);
// "vLLM-Omni 在线量化（Online Quantization）完全指南" section
// "在线量化的底层工作原理" stage 2 (E4M3 + float8_e8m0fnu per 32 along K);
// "vLLM-Omni 量化推理实践" Table 1 (NVFP4 in the mixed FP8/NVFP4 model);
// "vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다" section "새로운 모델
// 양자화" (int4, group_size 128, auto_round:auto_gptq packing, --iters 0;
// the checkpoint config's "sym": true for the symmetric variant);
// "vLLM-Omni 在线量化（Online Quantization）完全指南" sections "在线量化的底层
// 工作原理" and "核心参数详解" (INT8 W8A8: per-channel weight scales, dynamic
// per-token activation scales).
//
// Bit-exactness: every fp32 step is one explicitly rounded intrinsic
// (__fmul_rn, __fdiv_rn, __fsub_rn), this file is compiled with
// -fmad=false -ftz=false -prec-div=true, and the E4M3/E2M1 conversions are
// the hardware cvt.rn.satfinite instructions.
#include <atomic>

#include <cuda_bf16.h>

#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr float kE4M3Max = 448.0f;
constexpr float kNvfp4Global = 2688.0f;   // 448 (E4M3 max) * 6 (E2M1 max)

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint4 ld16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

__device__ __forceinline__ float absmax8(const uint4& v) {
    float a = fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x)));
    a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
    a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))));
    a = fmaxf(a, fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w))));
    return a;
}

// The same maximum on bf16 pairs: clear the sign bits, three packed maxima
// (exact: a max of bf16 values is one of them), then the last pair in fp32.
__device__ __forceinline__ float absmax8_bf16x2(const uint4& v) {
    const uint32_t u[4] = {v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu, v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu};
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u[0]),
                                     *reinterpret_cast<const __nv_bfloat162*>(&u[1]));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&u[2]),
                                     *reinterpret_cast<const __nv_bfloat162*>(&u[3]));
    const __nv_bfloat162 m = __hmax2(a, b);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(&m);
    return fmaxf(bf16_lo(w), bf16_hi(w));
}

// Two fp32 -> two E4M3 codes, round to nearest even, saturating; `lo` lands
// in bits 0..7.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One E4M3 code -> its value (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    uint16_t in = (uint16_t)(code & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n}" : "=f"(f) : "r"(h2));
    return f;
}

// Four fp32 -> four E4M3 codes in one word (a, b in the low half, lo first).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 t0, t1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t1, %4, %3;\n\t"
        "mov.b32 %0, {t0, t1};\n}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// 8 bf16 (one 16-byte vector) times r -> 8 E4M3 codes.
__device__ __forceinline__ uint2 enc8_e4m3(const uint4& v, float r) {
    return make_uint2(cvt_e4m3x4(__fmul_rn(bf16_lo(v.x), r), __fmul_rn(bf16_hi(v.x), r), __fmul_rn(bf16_lo(v.y), r),
                                 __fmul_rn(bf16_hi(v.y), r)),
                      cvt_e4m3x4(__fmul_rn(bf16_lo(v.z), r), __fmul_rn(bf16_hi(v.z), r), __fmul_rn(bf16_lo(v.w), r),
                                 __fmul_rn(bf16_hi(v.w), r)));
}

// Eight fp32 (pairs lo, hi in each of the four slots) -> eight E2M1 codes
// in one word, pair i in byte i (lo in its low nibble): four conversions into
// byte registers, packed by one vector move.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float l0, float h0, float l1, float h1, float l2, float h2, float l3,
                                               float h3) {
    uint32_t r;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n}"
        : "=r"(r)
        : "f"(l0), "f"(h0), "f"(l1), "f"(h1), "f"(l2), "f"(h2), "f"(l3), "f"(h3));
    return r;
}

// 8 bf16 times r -> 8 E2M1 codes packed in 4 bytes.
__device__ __forceinline__ uint32_t enc8_e2m1(const uint4& v, float r) {
    return cvt_e2m1x8(__fmul_rn(bf16_lo(v.x), r), __fmul_rn(bf16_hi(v.x), r), __fmul_rn(bf16_lo(v.y), r),
                      __fmul_rn(bf16_hi(v.y), r), __fmul_rn(bf16_lo(v.z), r), __fmul_rn(bf16_hi(v.z), r),
                      __fmul_rn(bf16_lo(v.w), r), __fmul_rn(bf16_hi(v.w), r));
}

// 8 bf16 times r (rounded), then times the power of two m (exact) -> 8
// E2M1 codes packed in 4 bytes: the two steps of the dual-scale rule.
__device__ __forceinline__ uint32_t enc8_e2m1_2(const uint4& v, float r, float m) {
    return cvt_e2m1x8(__fmul_rn(__fmul_rn(bf16_lo(v.x), r), m), __fmul_rn(__fmul_rn(bf16_hi(v.x), r), m),
                      __fmul_rn(__fmul_rn(bf16_lo(v.y), r), m), __fmul_rn(__fmul_rn(bf16_hi(v.y), r), m),
                      __fmul_rn(__fmul_rn(bf16_lo(v.z), r), m), __fmul_rn(__fmul_rn(bf16_hi(v.z), r), m),
                      __fmul_rn(__fmul_rn(bf16_lo(v.w), r), m), __fmul_rn(__fmul_rn(bf16_hi(v.w), r), m));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Max over the block; every thread receives the result.
template <int T>
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = lane < T / 32 ? red[lane] : 0.0f;
        w = warp_max(w);
        if (lane == 0) red[32] = w;
    }
    __syncthreads();
    return red[32];
}

// FP8 granule: s = amax/448 and encode multiplier 448/amax (1, 1 for amax 0).
__device__ __forceinline__ void fp8_params(float amax, float& s, float& r) {
    if (amax == 0.0f) { s = 1.0f; r = 1.0f; return; }
    s = __fdiv_rn(amax, kE4M3Max);
    r = __fdiv_rn(kE4M3Max, amax);
}

// INT8 granule: s = amax/127 and encode multiplier 127/amax (1, 1 for amax 0).
__device__ __forceinline__ void int8_params(float amax, float& s, float& r) {
    if (amax == 0.0f) { s = 1.0f; r = 1.0f; return; }
    s = __fdiv_rn(amax, 127.0f);
    r = __fdiv_rn(127.0f, amax);
}

// v * r -> int8 code clamp(rint(v * r), -127, 127) in the low byte.  |v * r|
// <= 127 (up to one rounding), so adding 1.5 * 2^23 lands in [2^23, 2^24),
// where the fp32 spacing is 1: the add rounds the product to an integer,
// ties to even, and the bits minus those of 1.5 * 2^23 are that integer.
__device__ __forceinline__ uint32_t int8_code(float v, float r) {
    const int t = (int)__float_as_uint(__fadd_rn(__fmul_rn(v, r), 12582912.0f)) - 0x4B400000;
    return (uint32_t)min(max(t, -127), 127) & 0xFFu;
}

// 8 bf16 (one 16-byte vector) times r -> 8 int8 codes.
__device__ __forceinline__ uint2 enc8_int8(const uint4& v, float r) {
    const uint32_t w0 = int8_code(bf16_lo(v.x), r) | (int8_code(bf16_hi(v.x), r) << 8) |
                        (int8_code(bf16_lo(v.y), r) << 16) | (int8_code(bf16_hi(v.y), r) << 24);
    const uint32_t w1 = int8_code(bf16_lo(v.z), r) | (int8_code(bf16_hi(v.z), r) << 8) |
                        (int8_code(bf16_lo(v.w), r) << 16) | (int8_code(bf16_hi(v.w), r) << 24);
    return make_uint2(w0, w1);
}

// One row granule, FP8 (s = amax/448, E4M3 codes) or INT8 (s = amax/127).
template <bool INT8>
__device__ __forceinline__ void row_params(float amax, float& s, float& r) {
    if constexpr (INT8) int8_params(amax, s, r);
    else fp8_params(amax, s, r);
}

template <bool INT8>
__device__ __forceinline__ uint2 enc8_row(const uint4& v, float r) {
    if constexpr (INT8) return enc8_int8(v, r);
    else return enc8_e4m3(v, r);
}

// Byte offset of scale (row, j).  In the tensor-core tiling (see qlin.h),
// 512-byte chunks of 128 rows x 4 scales ordered [row_tile][chunk]:
//   ((row / 128 * chunks + j / 4) << 9) + (row % 32) * 16 + (row % 128 / 32) * 4 + j % 4;
// in the canonical layout row * gs + j.  Split into a per-row base and a
// per-scale part, so that a warp working on one row computes the 64-bit base
// once: offset(row, j) = scale_row_base(row) + scale_col_part(j) (gs = scales
// per row in the canonical layout, chunks = 4-scale chunks per row in the tiling).
__device__ __forceinline__ int64_t scale_row_base(int64_t row, int64_t gs, int64_t chunks, int mma) {
    if (!mma) return row * gs;
    const int64_t rr = row & 127;
    return (((row >> 7) * chunks) << 9) + ((rr & 31) << 4) + ((rr >> 5) << 2);
}
__device__ __forceinline__ int scale_col_part(int j, int mma) { return mma ? (((j >> 2) << 9) + (j & 3)) : j; }

// ---------------------------------------------------------------- row tasks
// The tensor-amax passes (per-tensor FP8, the NVFP4 global scale) walk
// "tasks": 32 consecutive 16-byte vectors (256 elements) of one row, one task
// per warp and one vector per lane, so each row is read in 512-byte coalesced
// segments.  A warp keeps kUnroll tasks
// in flight; row and column come from one 32-bit division per task.  The
// task count fits in 32 bits for any tensor that fits in device memory (the
// host checks).
constexpr int kUnroll = 4;

struct TaskPos {
    uint32_t row, c;   // c: 16-byte vector index within the row
    bool in;           // the task exists and c < vectors per row
};

__device__ __forceinline__ TaskPos task_pos(uint32_t t, uint32_t total, uint32_t tpr, uint32_t nvr, int lane) {
    TaskPos q{0, 0, false};
    if (t < total) {
        q.row = t / tpr;
        q.c = (t - q.row * tpr) * 32 + (uint32_t)lane;
        q.in = q.c < nvr;
    }
    return q;
}

// ---------------------------------------------------------------- per row
// One CTA per row; each thread keeps VPT 16-byte vectors in registers so the
// row is read from HBM once.  FP8 per-token and INT8 per-row (a token of X or
// an output channel of W) share this body and differ in the granule rule.
template <int T, int VPT, bool INT8>
__device__ __forceinline__ void rows_body(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                          uint8_t* __restrict__ codes, float* __restrict__ scales) {
    __shared__ float red[33];
    const int64_t row = blockIdx.x;
    const uint16_t* src = x + row * ld;
    const int nv = (int)(K >> 3);
    uint4 v[VPT];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; i++) {
        const int j = threadIdx.x + i * T;
        if (j < nv) {
            v[i] = ld16(src + 8 * j);
            amax = fmaxf(amax, absmax8(v[i]));
        }
    }
    amax = block_max<T>(amax, red);
    float s, r;
    row_params<INT8>(amax, s, r);
    uint2* dst = reinterpret_cast<uint2*>(codes + row * K);
#pragma unroll
    for (int i = 0; i < VPT; i++) {
        const int j = threadIdx.x + i * T;
        if (j < nv) dst[j] = enc8_row<INT8>(v[i], r);
    }
    if (threadIdx.x == 0) scales[row] = s;
}

template <int T, int VPT>
__global__ void __launch_bounds__(T) k_fp8_rows(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                                uint8_t* __restrict__ codes, float* __restrict__ scales) {
    rows_body<T, VPT, false>(x, K, ld, codes, scales);
}

template <int T, int VPT>
__global__ void __launch_bounds__(T) k_int8_rows(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                                 uint8_t* __restrict__ codes, float* __restrict__ scales) {
    rows_body<T, VPT, true>(x, K, ld, codes, scales);
}

// Rows too long for registers: amax pass then encode pass (second read hits L2).
template <bool INT8>
__device__ __forceinline__ void rows_long_body(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                               uint8_t* __restrict__ codes, float* __restrict__ scales) {
    __shared__ float red[33];
    const int64_t row = blockIdx.x;
    const uint16_t* src = x + row * ld;
    const int64_t nv = K >> 3;
    float amax = 0.0f;
    for (int64_t j = threadIdx.x; j < nv; j += 256) amax = fmaxf(amax, absmax8(ld16(src + 8 * j)));
    amax = block_max<256>(amax, red);
    float s, r;
    row_params<INT8>(amax, s, r);
    uint2* dst = reinterpret_cast<uint2*>(codes + row * K);
    for (int64_t j = threadIdx.x; j < nv; j += 256) dst[j] = enc8_row<INT8>(ld16(src + 8 * j), r);
    if (threadIdx.x == 0) scales[row] = s;
}

__global__ void __launch_bounds__(256) k_fp8_rows_long(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                                       uint8_t* __restrict__ codes, float* __restrict__ scales) {
    rows_long_body<false>(x, K, ld, codes, scales);
}

__global__ void __launch_bounds__(256) k_int8_rows_long(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                                        uint8_t* __restrict__ codes, float* __restrict__ scales) {
    rows_long_body<true>(x, K, ld, codes, scales);
}

// ---------------------------------------------------------------- per tensor
// Pass 1: partial amax per CTA into partials[blockIdx.x].
__global__ void __launch_bounds__(256) k_amax_partial(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                      int64_t ld, float* __restrict__ partials) {
    __shared__ float red[33];
    const uint32_t nvr = (uint32_t)(K >> 3), tpr = (nvr + 31) / 32, total = (uint32_t)rows * tpr;
    const uint32_t warps = gridDim.x * 8, w0 = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    float amax = 0.0f;
    for (uint32_t t = w0; t < total; t += warps * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; u++) {
            const TaskPos q = task_pos(t + u * warps, total, tpr, nvr, lane);
            v[u] = q.in ? ld16(x + (int64_t)q.row * ld + 8 * q.c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; u++) amax = fmaxf(amax, absmax8(v[u]));
    }
    amax = block_max<256>(amax, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = amax;
}

__device__ __forceinline__ float reduce_partials(const float* __restrict__ partials, int nparts, float* red) {
    float a = 0.0f;
    for (int i = threadIdx.x; i < nparts; i += 256) a = fmaxf(a, partials[i]);
    return block_max<256>(a, red);
}

// Pass 2: every CTA folds the partials (a few KB from L2), then encodes.
__global__ void __launch_bounds__(256) k_fp8_tensor_encode(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                           int64_t ld, uint8_t* __restrict__ codes,
                                                           float* __restrict__ scale,
                                                           const float* __restrict__ partials, int nparts) {
    __shared__ float red[33];
    const float amax = reduce_partials(partials, nparts, red);
    float s, r;
    fp8_params(amax, s, r);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
    const uint32_t nvr = (uint32_t)(K >> 3), tpr = (nvr + 31) / 32, total = (uint32_t)rows * tpr;
    const uint32_t warps = gridDim.x * 8, w0 = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (uint32_t t = w0; t < total; t += warps * kUnroll) {
        uint4 v[kUnroll];
        TaskPos q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; u++) {
            q[u] = task_pos(t + u * warps, total, tpr, nvr, lane);
            if (q[u].in) v[u] = ld16(x + (int64_t)q[u].row * ld + 8 * q[u].c);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; u++)
            if (q[u].in) reinterpret_cast<uint2*>(codes + (int64_t)q[u].row * K)[q[u].c] = enc8_e4m3(v[u], r);
    }
}

// 16-byte global -> shared copy that bypasses the registers (zero-filled when
// src_bytes is 0); completion through cp.async.wait_group, no spin.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

// ---------------------------------------------------------------- 128x128 block
// One CTA per 128x128 tile: 256 threads x 8 vectors; thread t covers rows
// t/16 + 16i and the 16-byte column t%16 (256-byte coalesced row segments).
__global__ void __launch_bounds__(256) k_fp8_block128(const uint16_t* __restrict__ x, int64_t K, int64_t ld,
                                                      uint8_t* __restrict__ codes, float* __restrict__ scales) {
    // The tile waits in shared memory rather than in registers, so more CTAs (and
    // more of their loads) fit on an SM.  Each thread reads back only the vectors
    // it copied itself, so its own cp.async.wait_group is the only wait needed.
    __shared__ __align__(16) uint4 tile[8][256];
    __shared__ float red[33];
    const int64_t kt = K >> 7, bi = (int64_t)blockIdx.x / kt, bj = (int64_t)blockIdx.x - bi * kt;
    const int r0 = threadIdx.x >> 4, cv = threadIdx.x & 15;
    const uint16_t* src = x + (bi * 128 + r0) * ld + bj * 128 + cv * 8;   // row r0 + 16 i for i = 0..7
#pragma unroll
    for (int i = 0; i < 8; i++) cp_async16(&tile[i][threadIdx.x], src + (int64_t)(16 * i) * ld, 16u);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) amax = fmaxf(amax, absmax8(tile[i][threadIdx.x]));
    amax = block_max<256>(amax, red);
    float s, r;
    fp8_params(amax, s, r);
    uint8_t* dst = codes + (bi * 128 + r0) * K + bj * 128 + cv * 8;
#pragma unroll
    for (int i = 0; i < 8; i++)
        *reinterpret_cast<uint2*>(dst + (int64_t)(16 * i) * K) = enc8_e4m3(tile[i][threadIdx.x], r);
    if (threadIdx.x == 0) scales[bi * (K >> 7) + bj] = s;
}

// ---------------------------------------------------------------- row chunks
// The 1 x 128-group, MX and NVFP4 quantizers walk "row chunks": warp w of a
// CTA owns one row and kChunk = 32 * kChunkU consecutive 16-byte vectors of
// it, kChunkU per lane (lane + 32 u), so each vector slot of the warp reads
// 512 contiguous bytes and the row and column come from the block and warp
// indices without a division.  Row blocks of 8 rows run along grid x, chunks
// along grid y.  A granule (32, 16 or 128 elements: 4, 2 or 16 lanes) never
// straddles a chunk, and every lane of a warp runs the same shuffles.
constexpr int kChunkU = 4;
constexpr int kChunk = 32 * kChunkU;           // vectors per warp chunk (1024 elements)

// ---------------------------------------------------------------- 1 x 128 groups
// Sixteen lanes own one 128-element group; the group amax comes from four
// xor-shuffles inside the 16 lanes.  A half-warp holds kChunkU groups; lane
// l works out the scale and multiplier (two divisions) of group l & 3 only,
// and the others take them by shuffle.  K % 128 == 0.
static_assert(kChunkU == 4, "one group per lane & 3");
__global__ void __launch_bounds__(256) k_fp8_group128(const uint16_t* __restrict__ x, int rows, int K, int64_t ld,
                                                      uint8_t* __restrict__ codes, float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int nvr = K >> 3, c0 = blockIdx.y * kChunk + lane;
    const uint16_t* src = x + (int64_t)row * ld;
    uint4 v[kChunkU];
#pragma unroll
    for (int u = 0; u < kChunkU; u++) {
        const int c = c0 + 32 * u;
        v[u] = c < nvr ? ld16(src + 8 * c) : make_uint4(0, 0, 0, 0);
    }
    float a[kChunkU];
#pragma unroll
    for (int u = 0; u < kChunkU; u++) {
        a[u] = absmax8_bf16x2(v[u]);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) a[u] = fmaxf(a[u], __shfl_xor_sync(0xFFFFFFFFu, a[u], o));
    }
    const int mine = lane & 3;
    const float am = mine == 0 ? a[0] : mine == 1 ? a[1] : mine == 2 ? a[2] : a[3];
    float sc_m, r_m;
    fp8_params(am, sc_m, r_m);
    uint2* dst = reinterpret_cast<uint2*>(codes + (int64_t)row * K);
    float* srow = scales + (int64_t)row * (K >> 7);
#pragma unroll
    for (int u = 0; u < kChunkU; u++) {
        const int c = c0 + 32 * u;
        const float r = __shfl_sync(0xFFFFFFFFu, r_m, (lane & 16) | u);
        const float sc = __shfl_sync(0xFFFFFFFFu, sc_m, (lane & 16) | u);
        if (c >= nvr) continue;
        dst[c] = enc8_e4m3(v[u], r);
        if ((c & 15) == 0) srow[c >> 4] = sc;
    }
}

// ---------------------------------------------------------------- MXFP8 / MXFP4
// The MX rule with the element format's largest power-of-two exponent: 8 for
// E4M3 (MXFP8), 2 for E2M1 (MXFP4, codes two per byte).  Four consecutive
// lanes own one 32-element granule (8 elements each).  Rows from `rows` up to
// `rows_pad` exist only in the MMA scale layout: they get scale code 0 and no
// codes.
template <bool FP4>
__global__ void __launch_bounds__(256) k_mx(const uint16_t* __restrict__ x, int rows, int rows_pad, int K, int64_t ld,
                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int mma) {
    constexpr int kEmax = FP4 ? 2 : 8;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows_pad) return;
    const bool live = row < rows;
    const int nvr = K >> 3, c0 = blockIdx.y * kChunk + lane;
    const uint16_t* src = x + (int64_t)row * ld;
    uint4 v[kChunkU];
#pragma unroll
    for (int u = 0; u < kChunkU; u++) {
        const int c = c0 + 32 * u;
        v[u] = (live && c < nvr) ? ld16(src + 8 * c) : make_uint4(0, 0, 0, 0);
    }
    uint8_t* crow = codes + (int64_t)row * (FP4 ? (K >> 1) : K);
    uint8_t* srow = scales + scale_row_base(row, K >> 5, K >> 7, mma);
#pragma unroll
    for (int u = 0; u < kChunkU; u++) {
        const int c = c0 + 32 * u;
        float a = absmax8_bf16x2(v[u]);
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        if (c >= nvr) continue;
        // e = clamp(floor(log2 a) - kEmax, -127, 127); subnormal a lands below -127.
        const int biased = (int)(__float_as_uint(a) >> 23);
        int e = (a == 0.0f || biased == 0) ? -127 : max(biased - 127 - kEmax, -127);
        e = min(e, 127);
        const float mult = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e, e <= 126 here
        if (live) {
            if (FP4) reinterpret_cast<uint32_t*>(crow)[c] = enc8_e2m1(v[u], mult);
            else reinterpret_cast<uint2*>(crow)[c] = enc8_e4m3(v[u], mult);
        }
        if ((c & 3) == 0) srow[scale_col_part(c >> 2, mma)] = (uint8_t)(e + 127);
    }
}

// ---------------------------------------------------------------- MXFP4 dual-scale
// A warp chunk (1024 elements of a row) holds two 512-element coarse blocks:
// vector slots u = 0, 1 of every lane form the first, u = 2, 3 the second
// (K % 512 == 0).  The coarse amax is a full-warp maximum, the coarse scale
// A / 6 and multiplier 6 / A follow, and each 32-element granule (four lanes)
// takes the MX rule on its normalized values: its amax times 6 / A, rounded,
// is the maximum of the rounded products because rounding is monotone.
__global__ void __launch_bounds__(256) k_mx_dual(const uint16_t* __restrict__ x, int rows, int rows_pad, int K,
                                                 int64_t ld, uint8_t* __restrict__ codes,
                                                 uint8_t* __restrict__ scales, float* __restrict__ coarse, int mma) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows_pad) return;
    const bool live = row < rows;
    const int nvr = K >> 3, c0 = blockIdx.y * kChunk + lane;
    const uint16_t* src = x + (int64_t)row * ld;
    uint4 v[kChunkU];
#pragma unroll
    for (int u = 0; u < kChunkU; u++) {
        const int c = c0 + 32 * u;
        v[u] = (live && c < nvr) ? ld16(src + 8 * c) : make_uint4(0, 0, 0, 0);
    }
    uint32_t* crow = reinterpret_cast<uint32_t*>(codes + (int64_t)row * (K >> 1));
    uint8_t* srow = scales + scale_row_base(row, K >> 5, K >> 7, mma);
#pragma unroll
    for (int blk = 0; blk < 2; blk++) {
        const float A = warp_max(fmaxf(absmax8_bf16x2(v[2 * blk]), absmax8_bf16x2(v[2 * blk + 1])));
        float cs = 1.0f, rc = 1.0f;
        if (A != 0.0f) {
            cs = __fdiv_rn(A, 6.0f);
            rc = __fdiv_rn(6.0f, A);
        }
        const int cb0 = blockIdx.y * kChunk + 64 * blk;          // first vector of this coarse block
        if (cb0 >= nvr) break;                                    // K % 1024 == 512: the chunk's last block is absent
        if (live && lane == 0) coarse[(int64_t)row * (K >> 9) + (cb0 >> 6)] = cs;
#pragma unroll
        for (int uu = 0; uu < 2; uu++) {
            const int u = 2 * blk + uu, c = c0 + 32 * u;
            float a = absmax8_bf16x2(v[u]);
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
            a = __fmul_rn(a, rc);
            const int biased = (int)(__float_as_uint(a) >> 23);
            int e = (a == 0.0f || biased == 0) ? -127 : max(biased - 127 - 2, -127);
            e = min(e, 127);
            const float mult = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e, e <= 126 here
            if (live) crow[c] = enc8_e2m1_2(v[u], rc, mult);
            if ((c & 3) == 0) srow[scale_col_part(c >> 2, mma)] = (uint8_t)(e + 127);
        }
    }
}

// ---------------------------------------------------------------- NVFP4
// After the amax pass: two consecutive lanes own one 16-element block.  The
// code multiplier rg / dsb depends only on the block's UE4M3 scale code, so
// each CTA tabulates it once for all 256 codes (same division, same bits).
// That prologue (and folding the partial maxima) makes the grid persistent:
// a CTA takes the chunk ids blockIdx.x, blockIdx.x + gridDim.x, ..., chunk
// id = row block * chunks per row + chunk (one division per id).
__global__ void __launch_bounds__(256) k_nvfp4_encode(const uint16_t* __restrict__ x, int rows, int rows_pad, int K,
                                                      int64_t ld, uint8_t* __restrict__ codes,
                                                      uint8_t* __restrict__ scales, float* __restrict__ global,
                                                      const float* __restrict__ partials, int nparts, int mma) {
    __shared__ float red[33];
    __shared__ float rb_of[256];
    const float A = reduce_partials(partials, nparts, red);
    float g = 1.0f, qm = 1.0f, rg = 1.0f;
    if (A != 0.0f) {
        g = __fdiv_rn(A, kNvfp4Global);
        qm = __fdiv_rn(kE4M3Max, A);
        rg = __fdiv_rn(kNvfp4Global, A);
    }
    {
        const float dsb = e4m3_value((uint32_t)threadIdx.x);
        rb_of[threadIdx.x] = (dsb == 0.0f) ? 0.0f : __fdiv_rn(rg, dsb);
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) *global = g;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nvr = K >> 3, nch = (nvr + kChunk - 1) / kChunk;
    const uint32_t ids = (uint32_t)((rows_pad + 7) / 8) * (uint32_t)nch;
    for (uint32_t id = blockIdx.x; id < ids; id += gridDim.x) {
        const uint32_t rb = id / (uint32_t)nch;
        const int row = (int)rb * 8 + warp;
        if (row >= rows_pad) continue;                   // warp-uniform
        const bool live = row < rows;
        const int c0 = (int)(id - rb * (uint32_t)nch) * kChunk + lane;
        const uint16_t* src = x + (int64_t)row * ld;
        uint4 v[kChunkU];
#pragma unroll
        for (int u = 0; u < kChunkU; u++) {
            const int c = c0 + 32 * u;
            v[u] = (live && c < nvr) ? ld16(src + 8 * c) : make_uint4(0, 0, 0, 0);
        }
        uint32_t* crow = reinterpret_cast<uint32_t*>(codes + (int64_t)row * (K >> 1));
        uint8_t* srow = scales + scale_row_base(row, K >> 4, K >> 6, mma);
#pragma unroll
        for (int u = 0; u < kChunkU; u++) {
            const int c = c0 + 32 * u;
            float b = absmax8_bf16x2(v[u]);
            b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
            if (c >= nvr) continue;
            const uint32_t sb = cvt_e4m3x2(__fmul_rn(b, qm), 0.0f) & 0xFFu;   // non-negative: UE4M3
            if (live) crow[c] = enc8_e2m1(v[u], rb_of[sb]);
            if ((c & 1) == 0) srow[scale_col_part(c >> 1, mma)] = (uint8_t)sb;
        }
    }
}

// ---------------------------------------------------------------- int4 g128
constexpr int kInt4Pitch = 272;   // bytes per staged row: 256 + 16, so 8 lanes reading 8 rows hit 8 bank groups

// One thread per output channel and 128-K group: it takes the group's 256
// contiguous bytes of its weight row (16 vectors), so min/max, the scale, the
// zero point and the 16 packed words are all computed once, by one thread.
// The CTA's 128 x 128 tile is first copied into shared memory with coalesced
// 16-byte copies (a warp moves two 256-byte row segments per instruction)
// instead of each lane loading from its own row.
// A warp covers 32 consecutive channels, so each qweight row store (fixed
// k-octet, consecutive n) and each scale store is coalesced; the zero points
// of 8 channels are OR-ed into one word across 8 lanes.
// SYM takes the range symmetric, [-a, a] with a = max |x|, and stores the
// fixed zero point 8 (the "sym": true int4 variant); otherwise the range is
// [min(0, min), max(0, max)] and the zero point is derived from it.
template <bool SYM>
__global__ void __launch_bounds__(128) k_int4_g128(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                   int64_t ld, int32_t* __restrict__ qweight,
                                                   uint16_t* __restrict__ scales, int32_t* __restrict__ qzeros) {
    __shared__ __align__(16) uint8_t tile[128 * kInt4Pitch];
    const int64_t nb = (N + 127) >> 7, g = (int64_t)blockIdx.x / nb, k0 = g * 128;
    const int64_t n0 = ((int64_t)blockIdx.x - g * nb) * 128, n = n0 + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const bool valid = n < N;
    // copy j of thread t: row 8 j + t / 16, 16-byte column t % 16 (rows past N zero-filled)
#pragma unroll
    for (int j = 0; j < 16; j++) {
        const int r = 8 * j + (threadIdx.x >> 4), c = threadIdx.x & 15;
        const bool in = n0 + r < N;
        cp_async16(tile + r * kInt4Pitch + 16 * c, w + (in ? n0 + r : 0) * ld + k0 + 8 * c, in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    uint4 v[16];
#pragma unroll
    for (int o = 0; o < 16; o++) v[o] = *reinterpret_cast<const uint4*>(tile + threadIdx.x * kInt4Pitch + 16 * o);
    // min and max on bf16 pairs (exact), four independent chains of each,
    // then combined
    __nv_bfloat162 mn2[4], mx2[4];
#pragma unroll
    for (int i = 0; i < 4; i++) { mn2[i] = __floats2bfloat162_rn(0.0f, 0.0f); mx2[i] = mn2[i]; }
#pragma unroll
    for (int o = 0; o < 16; o++) {
        const uint32_t u[4] = {v[o].x, v[o].y, v[o].z, v[o].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&u[i]);
            mn2[i] = __hmin2(mn2[i], h);
            mx2[i] = __hmax2(mx2[i], h);
        }
    }
    const __nv_bfloat162 m0 = __hmin2(__hmin2(mn2[0], mn2[1]), __hmin2(mn2[2], mn2[3]));
    const __nv_bfloat162 m1 = __hmax2(__hmax2(mx2[0], mx2[1]), __hmax2(mx2[2], mx2[3]));
    float mn = fminf(__low2float(m0), __high2float(m0));
    float mx = fmaxf(__low2float(m1), __high2float(m1));
    if constexpr (SYM) {
        mx = fmaxf(mx, -mn);          // a = max |x|; the range [-a, a]
        mn = -mx;
    }
    const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
    float s = __bfloat162float(sb);
    uint16_t sbits = __bfloat16_as_ushort(sb);
    if (s == 0.0f) { s = 1.0f; sbits = 0x3F80u; }
    const float r = __fdiv_rn(1.0f, s);
    const int z = SYM ? 8 : min(max(__float2int_rn(__fmul_rn(-mn, r)), 0), 15);
    // rint(x*r) + z without a float->int conversion per element: |x*r| <= 15,
    // and adding 1.5 * 2^23 rounds it to an integer (nearest even) in the low
    // mantissa bits, so bits(x*r + 1.5*2^23) - bits(1.5*2^23) = rint(x*r).
    constexpr float kRound = 12582912.0f;
    const int zoff = (int)0x4B400000 - z;
#pragma unroll
    for (int o = 0; o < 16; o++) {
        const uint32_t u[4] = {v[o].x, v[o].y, v[o].z, v[o].w};
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int ta = (int)__float_as_uint(__fadd_rn(__fmul_rn(bf16_lo(u[i]), r), kRound)) - zoff;
            const int tb = (int)__float_as_uint(__fadd_rn(__fmul_rn(bf16_hi(u[i]), r), kRound)) - zoff;
            const int qa = min(max(ta, 0), 15), qb = min(max(tb, 0), 15);
            word |= ((uint32_t)qa << (8 * i)) | ((uint32_t)qb << (8 * i + 4));
        }
        if (valid) qweight[(k0 / 8 + o) * N + n] = (int32_t)word;
    }
    if (valid) scales[g * N + n] = sbits;
    // N is a multiple of 8, so an aligned group of 8 lanes is all valid or all not
    uint32_t zw = (uint32_t)z << (4 * (lane & 7));
    zw |= __shfl_xor_sync(0xFFFFFFFFu, zw, 1);
    zw |= __shfl_xor_sync(0xFFFFFFFFu, zw, 2);
    zw |= __shfl_xor_sync(0xFFFFFFFFu, zw, 4);
    if (valid && (lane & 7) == 0) qzeros[g * (N / 8) + n / 8] = (int32_t)zw;
}

int sm_count() {
    static const int n = [] {     // initialised once, thread-safe
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            return v;
        return kNumSMs;
    }();
    return n;
}

// Grid of the per-tensor task walks (8 warps per CTA, kUnroll tasks per warp
// per round): the FP8 per-tensor encode pass begins by folding the partial
// maxima, so it stays persistent with one resident wave of CTAs and that
// prologue runs once per resident CTA.  Tasks of one tensor, or -1 when their count does
// not fit the 32-bit walk.
int64_t task_count(int64_t rows, int64_t K) {
    const int64_t t = rows * (((K >> 3) + 31) / 32);
    return t > 0x7FFFFFFFll ? -1 : t;
}

int64_t task_rounds(int64_t tasks) { return (tasks + 8 * kUnroll - 1) / (8 * kUnroll); }

// CTAs of a kernel that fit on one SM at once (256 threads, no dynamic shared
// memory), asked of the runtime once per kernel; a persistent grid larger
// than one resident wave would leave its last CTAs to start late.
template <typename Kern>
int resident_ctas(Kern k, std::atomic<int>& cache) {
    int c = cache.load(std::memory_order_relaxed);
    if (!c) {     // several threads may ask at once; they all get the same answer
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, k, 256, 0) != cudaSuccess || c < 1) {
            (void)cudaGetLastError();
            c = 4;
        }
        cache.store(c, std::memory_order_relaxed);
    }
    return c;
}

int task_grid_persistent(int64_t tasks, int per_sm) {
    int64_t b = task_rounds(tasks);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (b > cap) b = cap;
    return (int)(b < 1 ? 1 : b);
}

template <int T, bool INT8>
cudaError_t rows_dispatch(int vpt, const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                          float* scales, cudaStream_t st) {
    dim3 grid((unsigned)rows);
#define QLIN_ROWS(V)                                                                              \
    case V:                                                                                       \
        if constexpr (INT8) k_int8_rows<T, V><<<grid, T, 0, st>>>(x, K, ld, codes, scales);        \
        else k_fp8_rows<T, V><<<grid, T, 0, st>>>(x, K, ld, codes, scales);                        \
        break;
    switch (vpt) {
        QLIN_ROWS(1)
        QLIN_ROWS(2)
        QLIN_ROWS(3)
        QLIN_ROWS(4)
        QLIN_ROWS(5)
        QLIN_ROWS(6)
        QLIN_ROWS(7)
        default:
        QLIN_ROWS(8)
    }
#undef QLIN_ROWS
    return cudaGetLastError();
}

template <bool INT8>
cudaError_t rowwise(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes, float* scales,
                    cudaStream_t st) {
    const int64_t nv = K >> 3;
    if (nv <= 128 * 8) return rows_dispatch<128, INT8>((int)((nv + 127) / 128), x, rows, K, ld, codes, scales, st);
    if (nv <= 256 * 8) return rows_dispatch<256, INT8>((int)((nv + 255) / 256), x, rows, K, ld, codes, scales, st);
    if constexpr (INT8) k_int8_rows_long<<<(unsigned)rows, 256, 0, st>>>(x, K, ld, codes, scales);
    else k_fp8_rows_long<<<(unsigned)rows, 256, 0, st>>>(x, K, ld, codes, scales);
    return cudaGetLastError();
}

}  // namespace

int amax_partials(int64_t rows, int64_t K) {
    const int64_t nv = rows * (K >> 3);
    int64_t p = (nv + 1023) / 1024;
    if (p > 1024) p = 1024;
    return (int)(p < 1 ? 1 : p);
}

cudaError_t launch_fp8_rowwise(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                               float* scales, cudaStream_t st) {
    return rowwise<false>(x, rows, K, ld, codes, scales, st);
}

cudaError_t launch_int8_rowwise(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                                float* scales, cudaStream_t st) {
    return rowwise<true>(x, rows, K, ld, codes, scales, st);
}

cudaError_t launch_fp8_tensor(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                              float* scale, float* partials, int nparts, cudaStream_t st) {
    const int64_t tasks = task_count(rows, K);
    if (tasks < 0) return cudaErrorInvalidValue;
    k_amax_partial<<<nparts, 256, 0, st>>>(x, rows, K, ld, partials);
    static std::atomic<int> per_sm{0};
    k_fp8_tensor_encode<<<task_grid_persistent(tasks, resident_ctas(k_fp8_tensor_encode, per_sm)), 256, 0, st>>>(
        x, rows, K, ld, codes, scale, partials, nparts);
    return cudaGetLastError();
}

cudaError_t launch_fp8_block128(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                                float* scales, cudaStream_t st) {
    k_fp8_block128<<<(unsigned)((K / 128) * (rows / 128)), 256, 0, st>>>(x, K, ld, codes, scales);
    return cudaGetLastError();
}

// Grid of a row-chunk walk: row blocks of 8 along x, chunks of a row along y.
dim3 chunk_grid(int64_t rows, int64_t K) {
    const int64_t nch = ((K >> 3) + kChunk - 1) / kChunk;
    return dim3((unsigned)((rows + 7) / 8), (unsigned)nch);
}

cudaError_t launch_fp8_group128(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                                float* scales, cudaStream_t st) {
    k_fp8_group128<<<chunk_grid(rows, K), 256, 0, st>>>(x, (int)rows, (int)K, ld, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_mxfp8(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                         uint8_t* scales, bool mma_layout, cudaStream_t st) {
    const int64_t rows_pad = mma_layout ? (rows + 127) / 128 * 128 : rows;
    k_mx<false><<<chunk_grid(rows_pad, K), 256, 0, st>>>(x, (int)rows, (int)rows_pad, (int)K, ld, codes, scales,
                                                         mma_layout ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_mxfp4(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                         uint8_t* scales, bool mma_layout, cudaStream_t st) {
    const int64_t rows_pad = mma_layout ? (rows + 127) / 128 * 128 : rows;
    k_mx<true><<<chunk_grid(rows_pad, K), 256, 0, st>>>(x, (int)rows, (int)rows_pad, (int)K, ld, codes, scales,
                                                        mma_layout ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_mxfp4_dual(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                              uint8_t* scales, float* coarse, bool mma_layout, cudaStream_t st) {
    const int64_t rows_pad = mma_layout ? (rows + 127) / 128 * 128 : rows;
    k_mx_dual<<<chunk_grid(rows_pad, K), 256, 0, st>>>(x, (int)rows, (int)rows_pad, (int)K, ld, codes, scales, coarse,
                                                        mma_layout ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                         uint8_t* scales, float* global, bool mma_layout, float* partials, int nparts,
                         cudaStream_t st) {
    const int64_t rows_pad = mma_layout ? (rows + 127) / 128 * 128 : rows;
    const dim3 g = chunk_grid(rows_pad, K);
    const int64_t ids = (int64_t)g.x * g.y;
    static std::atomic<int> per_sm{0};       // one resident wave of the persistent encode pass
    int64_t grid = (int64_t)sm_count() * resident_ctas(k_nvfp4_encode, per_sm);
    if (grid > ids) grid = ids;
    k_amax_partial<<<nparts, 256, 0, st>>>(x, rows, K, ld, partials);
    k_nvfp4_encode<<<(unsigned)grid, 256, 0, st>>>(x, (int)rows, (int)rows_pad, (int)K, ld, codes, scales, global,
                                                  partials, nparts, mma_layout ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_int4_g128(const uint16_t* w, int64_t N, int64_t K, int64_t ld, int32_t* qweight,
                             uint16_t* scales, int32_t* qzeros, bool sym, cudaStream_t st) {
    const unsigned grid = (unsigned)(((N + 127) / 128) * (K / 128));
    if (sym) k_int4_g128<true><<<grid, 128, 0, st>>>(w, N, K, ld, qweight, scales, qzeros);
    else k_int4_g128<false><<<grid, 128, 0, st>>>(w, N, K, ld, qweight, scales, qzeros);
    return cudaGetLastError();
}

}  // namespace qlin
