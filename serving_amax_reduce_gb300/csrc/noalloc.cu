// Per-tensor FP8 quantization without any caller-provided or allocated
// workspace.
//
// Some callers cannot allocate device memory: a plugin running inside a
// serving engine that has already reserved the whole device memory budget
// for its own pool, or code that runs after start-up under a rule that the
// memory footprint must stay fixed.  They cannot pass the small workspace
// that qlin_quantize_act / qlin_quantize_weight use for the per-tensor amax
// partials either.  This entry point keeps those partials in a fixed device
// array that is part of the library image instead.
//
// The array is shared by every call on a device and keeps the last call's
// contents; each call overwrites exactly the slots it then reads, so nothing
// has to be cleared.  Two calls that overlap on the GPU (different streams
// without ordering) race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qlin_internal.h"

namespace {

// One partial maximum per reduction block of 16384 elements.
constexpr int64_t kElemsPerPartial = 16384;
static_assert(QLIN_NOALLOC_MAX_PARTIALS * kElemsPerPartial == QLIN_NOALLOC_MAX_ELEMENTS, "limits");

static __device__ __align__(256) float g_amax_partials[QLIN_NOALLOC_MAX_PARTIALS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
    unsigned long long ctx_id;   // the context the address belongs to (0: none yet)
    float* ptr;
};
Cached g_partials[kMaxDevices] = {};

// Unique id of the calling thread's current context, 0 if none is current or
// the driver does not say.  Ids are never reused within a process, so a
// context created after a device reset gets a new one.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    struct Entry {
        GetCurrent get_current = nullptr;
        GetId get_id = nullptr;
    };
    static const Entry e = [] {     // looked up once, thread-safe
        Entry r;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r.get_current = reinterpret_cast<GetCurrent>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r.get_id = reinterpret_cast<GetId>(p);
        return r;
    }();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!e.get_current || !e.get_id || e.get_current(&c) != CUDA_SUCCESS || !c || e.get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_amax_partials on the current device.  In host code the
// symbol is only a stand-in; its device address has to be asked for with that
// device current.  The answer is kept per device together with the id of the
// context it came from, and asked for again when the device's context has
// changed (after cudaDeviceReset the module is loaded anew, possibly
// elsewhere).
qlin_status partials_for_current_device(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return QLIN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return QLIN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = current_context_id();
    if (!g_partials[dev].ptr || id == 0 || g_partials[dev].ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_amax_partials) != cudaSuccess || !p) return QLIN_ERR_CUDA;
        g_partials[dev].ptr = static_cast<float*>(p);
        g_partials[dev].ctx_id = current_context_id();   // the lookup makes the device's context current
    }
    *out = g_partials[dev].ptr;
    return QLIN_OK;
}

}  // namespace

extern "C" qlin_status qlin_quantize_fp8_tensor_noalloc(const void* x_bf16_dev, int64_t rows, int64_t K, int64_t ld,
                                                        void* codes_dev, float* scale_dev, qlin_stream_t stream) {
    if (!x_bf16_dev || !codes_dev || !scale_dev || rows < 1 || K < 8 || (K & 7) || ld < K) return QLIN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x_bf16_dev) & 15u) || (ld * 2) % 16 || (reinterpret_cast<uintptr_t>(codes_dev) & 15u) ||
        (reinterpret_cast<uintptr_t>(scale_dev) & 3u))
        return QLIN_ERR_ALIGNMENT;
    if (rows > QLIN_NOALLOC_MAX_ELEMENTS / K) return QLIN_ERR_WORKSPACE;   // more partials than the fixed array holds
    const int64_t elems = rows * K;
    const int nparts = (int)((elems + kElemsPerPartial - 1) / kElemsPerPartial);
    float* partials = nullptr;
    qlin_status s = partials_for_current_device(&partials);
    if (s != QLIN_OK) return s;
    cudaError_t e = qlin::launch_fp8_tensor(static_cast<const uint16_t*>(x_bf16_dev), rows, K, ld,
                                            static_cast<uint8_t*>(codes_dev), scale_dev, partials, nparts,
                                            reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA;
}
