// W4A16 decode GEMM (int4 g128 weights x bf16 activations) -- placeholder
// until the tensor-core decode kernel lands.
#include "qlin_internal.h"

namespace qlin {
size_t w4a16_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }
cudaError_t launch_gemm_w4a16(const GemmArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace qlin
