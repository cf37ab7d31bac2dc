/*
 * A plain C99 consumer of include/qlin.h: it compiles without C++ or CUDA
 * headers, links libqlin.so, and checks the host-side part of the ABI that
 * needs no GPU: the version and status strings, the buffer-size queries, and
 * argument validation before any launch.  Exit status 0 on success; each
 * failed check prints one line.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "qlin.h"

static int failures = 0;

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            printf("FAILED line %d: %s\n", __LINE__, #cond);          \
            failures++;                                               \
        }                                                             \
    } while (0)

int main(void) {
    /* a non-null, 16-byte aligned address that no call below dereferences */
    void *const fake = (void *)(uintptr_t)(1u << 20);
    void *const misaligned = (void *)((uintptr_t)(1u << 20) + 2u);
    const int64_t big = (int64_t)1 << 31;
    int s;

    CHECK(strstr(qlin_version(), "sm_103a") != NULL);
    CHECK(qlin_last_cuda_error() == 0);
    for (s = QLIN_OK; s <= QLIN_ERR_DEVICE_TIMEOUT; s++) CHECK(strlen(qlin_status_string((qlin_status)s)) > 0);

    /* sizes (rows = M or N, K along the row) */
    CHECK(qlin_codes_bytes(QLIN_FP8_TOKEN, 4096, 3072) == (size_t)4096 * 3072);
    CHECK(qlin_scales_bytes(QLIN_FP8_TOKEN, QLIN_SCALE_CANONICAL, 4096, 3072) == (size_t)4096 * 4);
    CHECK(qlin_scales_bytes(QLIN_FP8_BLOCK128, QLIN_SCALE_CANONICAL, 12288, 3072) == (size_t)96 * 24 * 4);
    CHECK(qlin_codes_bytes(QLIN_NVFP4, 32768, 3072) == (size_t)32768 * 1536);
    CHECK(qlin_scales_bytes(QLIN_NVFP4, QLIN_SCALE_MMA, 20280, 3072) == (size_t)20352 * 192);
    CHECK(qlin_scales_bytes(QLIN_MXFP8, QLIN_SCALE_MMA, 20280, 5120) == (size_t)20352 * 160);
    CHECK(qlin_codes_bytes(QLIN_INT4_G128_ASYM, 4096, 4096) == (size_t)512 * 4096 * 4);
    CHECK(qlin_scales_bytes(QLIN_INT4_G128_ASYM, QLIN_SCALE_CANONICAL, 4096, 4096) == (size_t)32 * 4096 * 2);
    CHECK(qlin_zeros_bytes(QLIN_INT4_G128_ASYM, 4096, 4096) == (size_t)32 * 512 * 4);
    CHECK(qlin_codes_bytes(QLIN_BF16, 16, 16) == 0);
    CHECK(qlin_gemm_workspace_bytes(QLIN_INT4_G128_ASYM, QLIN_BF16, 16, 4096, 4096) == 0);
    CHECK(qlin_quant_workspace_bytes(QLIN_FP8_TENSOR, 128, 1024) >= sizeof(float));

    /* quantizers: validation happens before any launch */
    CHECK(qlin_quantize_act(QLIN_FP8_TOKEN, NULL, 128, 1024, 1024, fake, fake, NULL, QLIN_SCALE_CANONICAL, NULL, 0,
                            NULL, NULL) == QLIN_ERR_INVALID_ARG);
    CHECK(qlin_quantize_act(QLIN_FP8_TOKEN, misaligned, 128, 1024, 1024, fake, fake, NULL, QLIN_SCALE_CANONICAL, NULL,
                            0, NULL, NULL) == QLIN_ERR_ALIGNMENT);
    CHECK(qlin_quantize_act(QLIN_FP8_TENSOR, fake, 128, 1024, 1024, fake, fake, NULL, QLIN_SCALE_CANONICAL, NULL, 0,
                            NULL, NULL) == QLIN_ERR_WORKSPACE);
    CHECK(qlin_quantize_act(QLIN_INT4_G128_ASYM, fake, 128, 1024, 1024, fake, fake, NULL, QLIN_SCALE_CANONICAL, NULL,
                            0, NULL, NULL) == QLIN_ERR_UNSUPPORTED);
    CHECK(qlin_quantize_weight(QLIN_FP8_BLOCK128, fake, 200, 1024, 1024, fake, fake, NULL, NULL,
                               QLIN_SCALE_CANONICAL, NULL, 0, NULL, NULL) == QLIN_ERR_INVALID_ARG);
    CHECK(qlin_quantize_act(QLIN_FP8_TOKEN, fake, 1, big, big, fake, fake, NULL, QLIN_SCALE_CANONICAL, NULL, 0, NULL,
                            NULL) == QLIN_ERR_INVALID_ARG);

    /* GEMM pairs and shapes */
    CHECK(qlin_gemm(QLIN_NVFP4, QLIN_FP8_TOKEN, 128, 1024, 1024, fake, fake, fake, fake, fake, NULL, fake, NULL, fake,
                    1024, QLIN_SCALE_MMA, NULL, 0, NULL, NULL) == QLIN_ERR_UNSUPPORTED);
    CHECK(qlin_gemm(QLIN_FP8_TENSOR, QLIN_FP8_TENSOR, 0, 1024, 1024, fake, fake, NULL, fake, fake, NULL, NULL, NULL,
                    fake, 1024, QLIN_SCALE_CANONICAL, NULL, 0, NULL, NULL) == QLIN_ERR_INVALID_ARG);
    CHECK(qlin_gemm(QLIN_FP8_TENSOR, QLIN_FP8_TENSOR, 128, 1024, 1024, fake, fake, NULL, fake, fake, NULL, NULL, NULL,
                    misaligned, 1024, QLIN_SCALE_CANONICAL, NULL, 0, NULL, NULL) == QLIN_ERR_ALIGNMENT);
    CHECK(qlin_gemm(QLIN_MXFP8, QLIN_MXFP8, 128, 1024, 1024, fake, fake, NULL, fake, fake, NULL, NULL, NULL, fake,
                    1024, QLIN_SCALE_CANONICAL, NULL, 0, NULL, NULL) == QLIN_ERR_UNSUPPORTED);
    CHECK(qlin_gemm(QLIN_FP8_TENSOR, QLIN_BF16, 129, 1024, 1024, fake, NULL, NULL, fake, fake, NULL, NULL, NULL, fake,
                    1024, QLIN_SCALE_CANONICAL, NULL, 0, NULL, NULL) == QLIN_ERR_UNSUPPORTED);
    CHECK(qlin_gemm(QLIN_INT4_G128_ASYM, QLIN_BF16, 65535 * 64 + 1, 4096, 4096, fake, NULL, NULL, fake, fake, fake,
                    NULL, NULL, fake, 4096, QLIN_SCALE_CANONICAL, NULL, 0, NULL, NULL) == QLIN_ERR_INVALID_ARG);

    /* the other entry points */
    CHECK(qlin_quantize_fp8_tensor_noalloc(NULL, 8, 1024, 1024, fake, fake, NULL) == QLIN_ERR_INVALID_ARG);
    CHECK(qlin_quantize_fp8_tensor_noalloc(fake, QLIN_NOALLOC_MAX_ELEMENTS / 1024 + 1, 1024, 1024, fake, fake, NULL) ==
          QLIN_ERR_WORKSPACE);
    CHECK(qlin_debug_expire_wait(NULL, 10, NULL) == QLIN_ERR_INVALID_ARG);

    if (failures == 0) printf("c abi ok\n");
    return failures == 0 ? 0 : 1;
}
