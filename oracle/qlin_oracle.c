/*
 * qlin_oracle.c -- slow, scalar CPU oracle for the quantized-linear hot path.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The CUDA library
 * never links, includes or calls it, and it shares no code with the kernels.
 *
 * What it computes (the pages name the formats, not their arithmetic):
 *   - "[vLLM] 기타 양자화: FP8, ModelOpt, INC, TorchAO, Quark", section
 *     "FP8: vLLM의 핵심 양자화": FP8 E4M3 with per-tensor, per-token and
 *     128x128-block dynamic symmetric scales.
 *   - "vLLM-Omni 在线量化（Online Quantization）完全指南", section
 *     "在线量化的底层工作原理", stage 2: MXFP8 = E4M3 codes plus one
 *     float8_e8m0fnu exponent scale shared by 32 consecutive K elements.
 *   - "vLLM-Omni 量化推理实践", Table 1 (mixed FP8/NVFP4): NVFP4 = E2M1 codes,
 *     an E4M3 scale per 16 elements and an fp32 per-tensor scale.
 *   - "vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다", section
 *     "새로운 모델 양자화": int4, group_size 128, packing auto_round:auto_gptq,
 *     and the "--iters 0" no-tuning (round-to-nearest) mode.
 * Bit layouts follow the public definitions those names refer to: OCP OFP8
 * (E4M3 "fn"), OCP Microscaling v1.0 (E8M0, E2M1, the MX shared-exponent rule)
 * and NVIDIA's NVFP4 description (E2M1 + E4M3 per 16 + fp32 per tensor).
 *
 * Arithmetic contract: every float operation here is one IEEE-754 binary32
 * operation, round-to-nearest-even, denormals kept.  Build with
 * -ffp-contract=off and without -ffast-math so that no multiply-add is fused
 * and no division is turned into a reciprocal multiply.
 *
 * Readings where the pages leave the rule open (all of them, since the pages
 * print no formula; R6-R10 are not arithmetic readings, they fix inputs,
 * layouts and the pass rule):
 *   R1  FP8 dynamic granule: s = amax/448, codes = E4M3(x * (448/amax));
 *       amax == 0 gives s = 1 and multiplier 1.
 *   R2  MX shared exponent: e = clamp(floor(log2 amax) - 8, -127, 127)
 *       (OCP MX v1.0 rule, 8 = exponent of the largest E4M3 power of two);
 *       codes = E4M3(x * 2^-e); amax == 0 gives scale code 0.
 *   R3  NVFP4: g = A/2688 with A the tensor amax; block scale
 *       sb = UE4M3(b * (448/A)); element multiplier (2688/A)/dec(sb), or 0
 *       when dec(sb) == 0; E2M1 codes packed two per byte, lower K index in
 *       the low nibble.  A == 0 gives g = 1 and both helpers 1.
 *   R4  int4 asymmetric RTN: range [min(0,min), max(0,max)],
 *       s = bf16((max-min)/15) (1 if that is 0), r = 1/s, z = clamp(rint(-min*r)),
 *       q = clamp(rint(x*r) + z); z stored without the "-1" offset.
 *   R5  conversions to E4M3/E2M1 round to nearest, ties to the even code,
 *       saturate to the largest finite magnitude and keep the sign of zero.
 *   R11 MXFP4 (the same page and section: the online MXFP4 path mirrors
 *       MXFP8 with float4_e2m1fn_x2 codes, two per byte): the R2 rule with
 *       the E2M1 exponent, e = clamp(floor(log2 amax) - 2, -127, 127)
 *       (2 = exponent of 6, the largest E2M1 power-of-two range), codes =
 *       E2M1(x * 2^-e) packed two per byte, lower K index in the low nibble;
 *       amax == 0 gives scale code 0.
 *   R12 dynamic FP8 128-group activations ("[vLLM] 기타 양자화", section
 *       "FP8: vLLM의 핵심 양자화", the block-128 dynamic symmetric scheme
 *       applied to activations): the R1 granule is 1 x 128, one token times
 *       128 consecutive K elements, with one fp32 scale per (row, K/128).
 *   R13 INT8 W8A8 ("vLLM-Omni 在线量化（Online Quantization）完全指南",
 *       section "在线量化的底层工作原理": the CUDA online INT8 path makes
 *       the weight codes and their scales with a scaled int8 quantizer;
 *       section "核心参数详解": activations are dynamic only): symmetric
 *       per-row granule, one fp32 scale per weight output channel and one
 *       per activation token, s = amax/127, codes = clamp(rint(x * (127/amax)),
 *       -127, 127) as two's-complement bytes; amax == 0 gives s = 1 and
 *       multiplier 1.
 *   R15 int4 symmetric ("vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다",
 *       section "새로운 모델 양자화": the checkpoint's quantization_config
 *       has "sym": true): the R4 group with its range taken symmetric,
 *       [-a, a] with a = max |x| over the 128 elements, so s = bf16((a - (-a))/15)
 *       (1 if that is 0) and r = 1/s as in R4; the zero point is the fixed
 *       mid-code 8, not derived from the range, and q = clamp(rint(x*r) + 8)
 *       in [0, 15].  Stored exactly like R4 (qzeros all 8).
 *   R16 MXFP4 dual-scale online ("vLLM-Omni 在线量化（Online Quantization）完全指南",
 *       section "在线量化的底层工作原理": the online mxfp4_dualscale path computes
 *       a fine (per 32) and a coarse (per 512) scale level at run time and
 *       fills the absent calibrated mul_scale with ones): per row and 512
 *       consecutive K elements, A = max |x|, coarse fp32 scale c = A/6 and
 *       multiplier r = 6/A (both 1 when A == 0); the block is normalized,
 *       v = x * r (x * 1 for the all-ones mul_scale first, which is exact),
 *       and the R11 MX rule runs on v per 32: e = clamp(floor(log2 max|v|) - 2,
 *       -127, 127), codes E2M1(v * 2^-e) two per byte, scale byte e + 127.
 *       Dequant: dec(code) * 2^e * c.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bit helpers                                                         */
/* ------------------------------------------------------------------ */

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of a binary32. */
float oracle_bf16_to_f32(uint16_t h) { return from_bits((uint32_t)h << 16); }

/* binary32 -> bf16, round to nearest, ties to even (finite inputs). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = to_bits(f);
    uint32_t kept = u >> 16;          /* truncated result            */
    uint32_t rest = u & 0xFFFFu;      /* the dropped low half        */
    if (rest > 0x8000u || (rest == 0x8000u && (kept & 1u)))
        kept += 1u;                   /* carries into the exponent if needed */
    return (uint16_t)kept;
}

/* floor(log2(a)) for finite a > 0, read off the binary32 encoding. */
int oracle_floor_log2(float a)
{
    uint32_t u = to_bits(a) & 0x7FFFFFFFu;
    int biased = (int)(u >> 23);
    if (biased != 0)
        return biased - 127;
    /* subnormal: a = m * 2^-149 with 0 < m < 2^23 */
    uint32_t m = u & 0x7FFFFFu;
    int top = -1;
    while (m) { top++; m >>= 1; }
    return top - 149;
}

/* ------------------------------------------------------------------ */
/* element codecs                                                      */
/* ------------------------------------------------------------------ */

/* E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa; no infinities,
 * S.1111.111 is NaN, largest finite 448, smallest subnormal 2^-9. */
double oracle_dec_e4m3(uint8_t c)
{
    int sign = c >> 7, ex = (c >> 3) & 0xF, man = c & 7;
    double v;
    if (ex == 0xF && man == 7) return NAN;
    if (ex == 0) v = ldexp((double)man, -9);              /* man/8 * 2^-6 */
    else v = ldexp((double)(8 + man), ex - 7 - 3);        /* (1+man/8) * 2^(ex-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 code to v: ties to the even code, saturate at 448 (R5). */
uint8_t oracle_enc_e4m3(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    float a = fabsf(v);
    if (a > 448.0f) return sign | 0x7E;
    /* binade of a; the subnormal range shares the spacing of binade -6 */
    int e = (a >= 0x1p-6f) ? oracle_floor_log2(a) : -6;
    float spacing = ldexpf(1.0f, e - 3);                  /* 3 mantissa bits */
    float n = rintf(a / spacing);                         /* exact scaling, RNE */
    if (n == 16.0f) { e += 1; n = 8.0f; }                 /* rounded up into the next binade */
    int ni = (int)n;
    if (ni < 8) return sign | (uint8_t)ni;                /* subnormal, exponent field 0 */
    return sign | (uint8_t)(((e + 7) << 3) | (ni - 8));
}

/* E2M1: values +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; exponent bias 1. */
double oracle_dec_e2m1(uint8_t c)
{
    int sign = (c >> 3) & 1, ex = (c >> 1) & 3, man = c & 1;
    double v = (ex == 0) ? 0.5 * man : ldexp((double)(2 + man), ex - 2);
    return sign ? -v : v;
}

uint8_t oracle_enc_e2m1(float v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    float a = fabsf(v);
    if (a > 6.0f) return sign | 0x7;
    int e = (a >= 1.0f) ? oracle_floor_log2(a) : 0;
    float spacing = ldexpf(1.0f, e - 1);                  /* 1 mantissa bit */
    float n = rintf(a / spacing);
    if (n == 4.0f) { e += 1; n = 2.0f; }
    int ni = (int)n;
    if (ni < 2) return sign | (uint8_t)ni;                /* 0 or 0.5 */
    return sign | (uint8_t)(((e + 1) << 1) | (ni - 2));
}

/* E8M0: code c is 2^(c-127); 0xFF is NaN and never produced here. */
double oracle_dec_e8m0(uint8_t c)
{
    if (c == 0xFF) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 with an fp32 scale per granule (R1)                        */
/* ------------------------------------------------------------------ */

static void fp8_granule(float amax, float *s, float *r)
{
    if (amax == 0.0f) { *s = 1.0f; *r = 1.0f; return; }
    *s = amax / 448.0f;
    *r = 448.0f / amax;
}

/* One scale for the whole rows x K tensor.  codes: rows x K, row-major. */
void oracle_quant_fp8_tensor(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                             uint8_t *codes, float *scale)
{
    float amax = 0.0f, s, r;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(x[i * ld + k])));
    fp8_granule(amax, &s, &r);
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            codes[i * K + k] = oracle_enc_e4m3(oracle_bf16_to_f32(x[i * ld + k]) * r);
    *scale = s;
}

/* One scale per row ("per token").  scales: rows. */
void oracle_quant_fp8_token(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                            uint8_t *codes, float *scales)
{
    for (int64_t i = 0; i < rows; i++) {
        float amax = 0.0f, s, r;
        for (int64_t k = 0; k < K; k++)
            amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(x[i * ld + k])));
        fp8_granule(amax, &s, &r);
        for (int64_t k = 0; k < K; k++)
            codes[i * K + k] = oracle_enc_e4m3(oracle_bf16_to_f32(x[i * ld + k]) * r);
        scales[i] = s;
    }
}

/* One scale per 128 x 128 tile.  rows, K multiples of 128.
 * scales: (rows/128) x (K/128), row-major. */
/* FP8 E4M3 with one dynamic scale per 1 x 128 group along K (R12)      */
void oracle_quant_fp8_group128(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                               uint8_t *codes, float *scales)
{
    int64_t ng = K / 128;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t g = 0; g < ng; g++) {
            const uint16_t *grp = x + i * ld + g * 128;
            float amax = 0.0f, s, r;
            for (int k = 0; k < 128; k++)
                amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(grp[k])));
            fp8_granule(amax, &s, &r);
            for (int k = 0; k < 128; k++)
                codes[i * K + g * 128 + k] = oracle_enc_e4m3(oracle_bf16_to_f32(grp[k]) * r);
            scales[i * ng + g] = s;
        }
}

void oracle_quant_fp8_block128(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                               uint8_t *codes, float *scales)
{
    int64_t kb = K / 128;
    for (int64_t bi = 0; bi < rows / 128; bi++)
        for (int64_t bj = 0; bj < kb; bj++) {
            float amax = 0.0f, s, r;
            for (int64_t i = bi * 128; i < bi * 128 + 128; i++)
                for (int64_t k = bj * 128; k < bj * 128 + 128; k++)
                    amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(x[i * ld + k])));
            fp8_granule(amax, &s, &r);
            for (int64_t i = bi * 128; i < bi * 128 + 128; i++)
                for (int64_t k = bj * 128; k < bj * 128 + 128; k++)
                    codes[i * K + k] = oracle_enc_e4m3(oracle_bf16_to_f32(x[i * ld + k]) * r);
            scales[bi * kb + bj] = s;
        }
}

/* ------------------------------------------------------------------ */
/* MXFP8: E4M3 codes + E8M0 exponent per 32 along K (R2)               */
/* ------------------------------------------------------------------ */

/* K multiple of 32.  codes: rows x K; scale codes: rows x (K/32). */
void oracle_quant_mxfp8(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                        uint8_t *codes, uint8_t *scale_codes)
{
    int64_t nb = K / 32;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t b = 0; b < nb; b++) {
            const uint16_t *g = x + i * ld + b * 32;
            float amax = 0.0f;
            for (int k = 0; k < 32; k++)
                amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(g[k])));
            int e;
            if (amax == 0.0f) {
                e = -127;
            } else {
                e = oracle_floor_log2(amax) - 8;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            float mult = ldexpf(1.0f, -e);                /* 2^-e, exact */
            for (int k = 0; k < 32; k++)
                codes[i * K + b * 32 + k] = oracle_enc_e4m3(oracle_bf16_to_f32(g[k]) * mult);
            scale_codes[i * nb + b] = (uint8_t)(e + 127);
        }
}

/* ------------------------------------------------------------------ */
/* NVFP4: E2M1 codes, UE4M3 scale per 16, fp32 scale per tensor (R3)   */
/* ------------------------------------------------------------------ */

/* K multiple of 16.  packed codes: rows x (K/2) bytes (lower K index in the
 * low nibble); block scale codes: rows x (K/16); global: one float. */
/* MXFP4: E2M1 codes + E8M0 exponent per 32 along K (R11)              */
void oracle_quant_mxfp4(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                        uint8_t *packed, uint8_t *scale_codes)
{
    int64_t nb = K / 32;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t b = 0; b < nb; b++) {
            const uint16_t *g = x + i * ld + b * 32;
            float amax = 0.0f;
            for (int k = 0; k < 32; k++)
                amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(g[k])));
            int e;
            if (amax == 0.0f) {
                e = -127;
            } else {
                e = oracle_floor_log2(amax) - 2;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            float mult = ldexpf(1.0f, -e);                /* 2^-e, exact */
            for (int k = 0; k < 32; k += 2) {
                uint8_t lo = oracle_enc_e2m1(oracle_bf16_to_f32(g[k]) * mult);
                uint8_t hi = oracle_enc_e2m1(oracle_bf16_to_f32(g[k + 1]) * mult);
                packed[i * (K / 2) + (b * 32 + k) / 2] = (uint8_t)(lo | (hi << 4));
            }
            scale_codes[i * nb + b] = (uint8_t)(e + 127);
        }
}

void oracle_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                        uint8_t *packed, uint8_t *scale_codes, float *global)
{
    float A = 0.0f;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            A = fmaxf(A, fabsf(oracle_bf16_to_f32(x[i * ld + k])));
    float g, q, rg;
    if (A == 0.0f) { g = 1.0f; q = 1.0f; rg = 1.0f; }
    else { g = A / 2688.0f; q = 448.0f / A; rg = 2688.0f / A; }   /* 2688 = 448 * 6 */

    int64_t nb = K / 16;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t b = 0; b < nb; b++) {
            const uint16_t *blk = x + i * ld + b * 16;
            float bmax = 0.0f;
            for (int k = 0; k < 16; k++)
                bmax = fmaxf(bmax, fabsf(oracle_bf16_to_f32(blk[k])));
            uint8_t sb = oracle_enc_e4m3(bmax * q);         /* non-negative: UE4M3 */
            float dsb = (float)oracle_dec_e4m3(sb);         /* exact in binary32 */
            float rb = (dsb == 0.0f) ? 0.0f : rg / dsb;
            for (int k = 0; k < 16; k += 2) {
                uint8_t lo = oracle_enc_e2m1(oracle_bf16_to_f32(blk[k]) * rb);
                uint8_t hi = oracle_enc_e2m1(oracle_bf16_to_f32(blk[k + 1]) * rb);
                packed[i * (K / 2) + (b * 16 + k) / 2] = (uint8_t)(lo | (hi << 4));
            }
            scale_codes[i * nb + b] = sb;
        }
    *global = g;
}

/* MXFP4 dual-scale (R16): K multiple of 512.  packed codes: rows x (K/2)
 * bytes (lower K index in the low nibble); fine scale codes: rows x (K/32);
 * coarse scales: rows x (K/512) floats. */
void oracle_quant_mxfp4_dual(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                             uint8_t *packed, uint8_t *scale_codes, float *coarse)
{
    int64_t nc = K / 512, nb = K / 32;
    for (int64_t i = 0; i < rows; i++)
        for (int64_t cb = 0; cb < nc; cb++) {
            const uint16_t *blk = x + i * ld + cb * 512;
            float A = 0.0f, c = 1.0f, r = 1.0f;
            for (int k = 0; k < 512; k++)
                A = fmaxf(A, fabsf(oracle_bf16_to_f32(blk[k])));
            if (A != 0.0f) { c = A / 6.0f; r = 6.0f / A; }
            coarse[i * nc + cb] = c;
            for (int f = 0; f < 16; f++) {
                const uint16_t *g = blk + f * 32;
                float v[32], a = 0.0f;
                for (int k = 0; k < 32; k++) {
                    v[k] = (oracle_bf16_to_f32(g[k]) * 1.0f) * r;     /* mul_scale = 1, then the coarse level */
                    a = fmaxf(a, fabsf(v[k]));
                }
                int e;
                if (a == 0.0f) {
                    e = -127;
                } else {
                    e = oracle_floor_log2(a) - 2;
                    if (e < -127) e = -127;
                    if (e > 127) e = 127;
                }
                float mult = ldexpf(1.0f, -e);                 /* 2^-e, exact */
                for (int k = 0; k < 32; k += 2) {
                    uint8_t lo = oracle_enc_e2m1(v[k] * mult);
                    uint8_t hi = oracle_enc_e2m1(v[k + 1] * mult);
                    packed[i * (K / 2) + (cb * 512 + f * 32 + k) / 2] = (uint8_t)(lo | (hi << 4));
                }
                scale_codes[i * nb + cb * 16 + f] = (uint8_t)(e + 127);
            }
        }
}

void oracle_dequant_mxfp4_dual(const uint8_t *packed, int64_t rows, int64_t K,
                               const uint8_t *scale_codes, const float *coarse, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++) {
            uint8_t byte = packed[i * (K / 2) + k / 2];
            uint8_t c = (k % 2) ? (byte >> 4) : (byte & 0xF);
            out[i * K + k] = oracle_dec_e2m1(c) * oracle_dec_e8m0(scale_codes[i * (K / 32) + k / 32])
                             * (double)coarse[i * (K / 512) + k / 512];
        }
}

/* ------------------------------------------------------------------ */
/* int4 asymmetric, group 128 along K, round to nearest (R4)           */
/* ------------------------------------------------------------------ */

/* W: N x K (nn.Linear layout), N multiple of 8, K multiple of 128.
 * qweight: (K/8) x N int32, k = 8i + j in bits [4j, 4j+4) of qweight[i][n];
 * scales:  (K/128) x N bf16 bits;
 * qzeros:  (K/128) x (N/8) int32, n = 8i + j in bits [4j, 4j+4). */
void oracle_quant_int4_g128(const uint16_t *w, int64_t N, int64_t K, int64_t ld,
                            int32_t *qweight, uint16_t *scales, int32_t *qzeros)
{
    int64_t ng = K / 128;
    memset(qweight, 0, sizeof(int32_t) * (size_t)(K / 8) * (size_t)N);
    memset(qzeros, 0, sizeof(int32_t) * (size_t)ng * (size_t)(N / 8));
    for (int64_t n = 0; n < N; n++)
        for (int64_t g = 0; g < ng; g++) {
            const uint16_t *grp = w + n * ld + g * 128;
            float mn = 0.0f, mx = 0.0f;                    /* range always holds 0 */
            for (int k = 0; k < 128; k++) {
                float v = oracle_bf16_to_f32(grp[k]);
                mn = fminf(mn, v);
                mx = fmaxf(mx, v);
            }
            uint16_t sbits = oracle_f32_to_bf16((mx - mn) / 15.0f);
            float s = oracle_bf16_to_f32(sbits);
            if (s == 0.0f) { s = 1.0f; sbits = oracle_f32_to_bf16(1.0f); }
            float r = 1.0f / s;
            float zf = rintf(-mn * r);
            if (zf < 0.0f) zf = 0.0f;
            if (zf > 15.0f) zf = 15.0f;
            int z = (int)zf;
            for (int k = 0; k < 128; k++) {
                float qf = rintf(oracle_bf16_to_f32(grp[k]) * r) + (float)z;
                if (qf < 0.0f) qf = 0.0f;
                if (qf > 15.0f) qf = 15.0f;
                int64_t kk = g * 128 + k;
                uint32_t word = (uint32_t)qweight[(kk / 8) * N + n];
                word |= (uint32_t)(int)qf << (4 * (kk % 8));
                qweight[(kk / 8) * N + n] = (int32_t)word;
            }
            scales[g * N + n] = sbits;
            uint32_t zw = (uint32_t)qzeros[g * (N / 8) + n / 8];
            zw |= (uint32_t)z << (4 * (n % 8));
            qzeros[g * (N / 8) + n / 8] = (int32_t)zw;
        }
}

/* int4 symmetric, group 128 along K, round to nearest (R15).  Same
 * layouts as oracle_quant_int4_g128; every stored zero point is 8. */
void oracle_quant_int4_g128_sym(const uint16_t *w, int64_t N, int64_t K, int64_t ld,
                                int32_t *qweight, uint16_t *scales, int32_t *qzeros)
{
    int64_t ng = K / 128;
    memset(qweight, 0, sizeof(int32_t) * (size_t)(K / 8) * (size_t)N);
    memset(qzeros, 0, sizeof(int32_t) * (size_t)ng * (size_t)(N / 8));
    for (int64_t n = 0; n < N; n++)
        for (int64_t g = 0; g < ng; g++) {
            const uint16_t *grp = w + n * ld + g * 128;
            float a = 0.0f;
            for (int k = 0; k < 128; k++)
                a = fmaxf(a, fabsf(oracle_bf16_to_f32(grp[k])));
            uint16_t sbits = oracle_f32_to_bf16((a - (-a)) / 15.0f);
            float s = oracle_bf16_to_f32(sbits);
            if (s == 0.0f) { s = 1.0f; sbits = oracle_f32_to_bf16(1.0f); }
            float r = 1.0f / s;
            const int z = 8;
            for (int k = 0; k < 128; k++) {
                float qf = rintf(oracle_bf16_to_f32(grp[k]) * r) + (float)z;
                if (qf < 0.0f) qf = 0.0f;
                if (qf > 15.0f) qf = 15.0f;
                int64_t kk = g * 128 + k;
                uint32_t word = (uint32_t)qweight[(kk / 8) * N + n];
                word |= (uint32_t)(int)qf << (4 * (kk % 8));
                qweight[(kk / 8) * N + n] = (int32_t)word;
            }
            scales[g * N + n] = sbits;
            uint32_t zw = (uint32_t)qzeros[g * (N / 8) + n / 8];
            zw |= (uint32_t)z << (4 * (n % 8));
            qzeros[g * (N / 8) + n / 8] = (int32_t)zw;
        }
}

/* ------------------------------------------------------------------ */
/* INT8 symmetric, one fp32 scale per row (R13)                         */
/* ------------------------------------------------------------------ */

/* codes: rows x K int8, row-major; scales: rows.  A row is one token of X or
 * one output channel of W. */
void oracle_quant_int8_row(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                           int8_t *codes, float *scales)
{
    for (int64_t i = 0; i < rows; i++) {
        float amax = 0.0f, s = 1.0f, r = 1.0f;
        for (int64_t k = 0; k < K; k++)
            amax = fmaxf(amax, fabsf(oracle_bf16_to_f32(x[i * ld + k])));
        if (amax != 0.0f) {
            s = amax / 127.0f;
            r = 127.0f / amax;
        }
        for (int64_t k = 0; k < K; k++) {
            float q = rintf(oracle_bf16_to_f32(x[i * ld + k]) * r);
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            codes[i * K + k] = (int8_t)(int)q;
        }
        scales[i] = s;
    }
}

/* ------------------------------------------------------------------ */
/* dequantizers: codes + scales -> exact values in binary64            */
/* ------------------------------------------------------------------ */

void oracle_dequant_fp8_tensor(const uint8_t *codes, int64_t rows, int64_t K, float scale,
                               double *out)
{
    for (int64_t i = 0; i < rows * K; i++)
        out[i] = oracle_dec_e4m3(codes[i]) * (double)scale;
}

void oracle_dequant_fp8_token(const uint8_t *codes, int64_t rows, int64_t K,
                              const float *scales, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = oracle_dec_e4m3(codes[i * K + k]) * (double)scales[i];
}

void oracle_dequant_fp8_group128(const uint8_t *codes, int64_t rows, int64_t K,
                                 const float *scales, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = oracle_dec_e4m3(codes[i * K + k]) * (double)scales[i * (K / 128) + k / 128];
}

void oracle_dequant_fp8_block128(const uint8_t *codes, int64_t rows, int64_t K,
                                 const float *scales, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = oracle_dec_e4m3(codes[i * K + k])
                             * (double)scales[(i / 128) * (K / 128) + k / 128];
}

void oracle_dequant_mxfp8(const uint8_t *codes, int64_t rows, int64_t K,
                          const uint8_t *scale_codes, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = oracle_dec_e4m3(codes[i * K + k])
                             * oracle_dec_e8m0(scale_codes[i * (K / 32) + k / 32]);
}

void oracle_dequant_mxfp4(const uint8_t *packed, int64_t rows, int64_t K,
                          const uint8_t *scale_codes, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++) {
            uint8_t byte = packed[i * (K / 2) + k / 2];
            uint8_t c = (k % 2) ? (byte >> 4) : (byte & 0xF);
            out[i * K + k] = oracle_dec_e2m1(c) * oracle_dec_e8m0(scale_codes[i * (K / 32) + k / 32]);
        }
}

void oracle_dequant_nvfp4(const uint8_t *packed, int64_t rows, int64_t K,
                          const uint8_t *scale_codes, float global, double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++) {
            uint8_t byte = packed[i * (K / 2) + k / 2];
            uint8_t c = (k % 2) ? (byte >> 4) : (byte & 0xF);
            out[i * K + k] = oracle_dec_e2m1(c) * oracle_dec_e4m3(scale_codes[i * (K / 16) + k / 16])
                             * (double)global;
        }
}

/* out: N x K, the dequantized weight (q - z) * s. */
void oracle_dequant_int4_g128(const int32_t *qweight, const uint16_t *scales,
                              const int32_t *qzeros, int64_t N, int64_t K, double *out)
{
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            int64_t g = k / 128;
            int q = (int)(((uint32_t)qweight[(k / 8) * N + n] >> (4 * (k % 8))) & 0xF);
            int z = (int)(((uint32_t)qzeros[g * (N / 8) + n / 8] >> (4 * (n % 8))) & 0xF);
            double s = (double)oracle_bf16_to_f32(scales[g * N + n]);
            out[n * K + k] = (double)(q - z) * s;
        }
}

void oracle_dequant_int8_row(const int8_t *codes, int64_t rows, int64_t K, const float *scales,
                             double *out)
{
    for (int64_t i = 0; i < rows; i++)
        for (int64_t k = 0; k < K; k++)
            out[i * K + k] = (double)codes[i * K + k] * (double)scales[i];
}
