// Internal launcher prototypes shared by the library's translation units.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "qlin.h"

namespace qlin {

constexpr int kNumSMs = 152;   // GB300: grids are sized in multiples of this

// ---------------------------------------------------------------- quantizers
// All take the bf16 source [rows, K] with leading dimension ld (elements).
cudaError_t launch_fp8_rowwise(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                               uint8_t* codes, float* scales, cudaStream_t st);
cudaError_t launch_int8_rowwise(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                                uint8_t* codes, float* scales, cudaStream_t st);
cudaError_t launch_fp8_tensor(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                              uint8_t* codes, float* scale, float* partials, int nparts,
                              cudaStream_t st);
cudaError_t launch_fp8_block128(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                                uint8_t* codes, float* scales, cudaStream_t st);
cudaError_t launch_fp8_group128(const uint16_t* x, int64_t rows, int64_t K, int64_t ld,
                                uint8_t* codes, float* scales, cudaStream_t st);
cudaError_t launch_mxfp8(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                         uint8_t* scales, bool mma_layout, cudaStream_t st);
cudaError_t launch_mxfp4(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                         uint8_t* scales, bool mma_layout, cudaStream_t st);
cudaError_t launch_mxfp4_dual(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                              uint8_t* scales, float* coarse, bool mma_layout, cudaStream_t st);
cudaError_t launch_nvfp4(const uint16_t* x, int64_t rows, int64_t K, int64_t ld, uint8_t* codes,
                         uint8_t* scales, float* global, bool mma_layout, float* partials,
                         int nparts, cudaStream_t st);
cudaError_t launch_int4_g128(const uint16_t* w, int64_t N, int64_t K, int64_t ld,
                             int32_t* qweight, uint16_t* scales, int32_t* qzeros, bool sym,
                             cudaStream_t st);

// Number of partial-amax slots the per-tensor reductions use for a tensor.
int amax_partials(int64_t rows, int64_t K);

// ---------------------------------------------------------------- GEMMs
struct GemmArgs {
    int64_t M, N, K, ldy;
    const void* x;            // codes (or bf16 activations for W4A16)
    const void* x_scales;
    const float* x_global;
    const void* w;            // codes / qweight
    const void* w_scales;
    const void* w_zeros;
    const float* w_global;
    const uint16_t* bias;     // bf16 [N] or null
    uint16_t* y;              // bf16 [M, ldy]
    void* workspace;
    size_t workspace_bytes;
    int* dev_status;
    bool x_group128;          // FP8 block GEMM: x_scales per (row, 128-K group) instead of per row
};

cudaError_t launch_gemm_fp8_tensor(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_fp8_block(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_mxfp8(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_nvfp4(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_mxfp4(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_mxfp4_dual(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_int8(const GemmArgs& a, cudaStream_t st);
// FP8 per-tensor weights x bf16 activations quantized per tensor inside the GEMM (M <= 128)
cudaError_t launch_gemm_fp8_tensor_fused_x(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_gemm_w4a16(const GemmArgs& a, cudaStream_t st);
size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K);

cudaError_t launch_debug_expire_wait(int* dev_status, uint32_t max_polls, cudaStream_t st);

}  // namespace qlin
