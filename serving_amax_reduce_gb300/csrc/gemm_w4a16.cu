// W4A16 decode GEMM: Y[M, N] = X[M, K] (bf16) . dequant(W)^T with W stored as
// int4 asymmetric codes, group 128 along K, GPTQ-style packing
// ("vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다", section "새로운 모델
// 양자화": bits 4, group_size 128, packing auto_round:auto_gptq).
//
//   Y[m, n] = sum_g s[g, n] * sum_{k in g} x[m, k] * (q[k, n] - z[g, n])
//
// Decode has few tokens, so the output channels take the MMA's M side
// ("swap AB"): a CTA owns 128 channels and MP tokens (MP = 16, 32 or 64,
// zero-filled past M by TMA; larger M runs as several token tiles).
// Per 128-K group:
//   warp 0    TMA: the packed int4 words (16 k-octets x 128 channels, 8 KB)
//             into a deep ring, so that enough HBM reads are in flight;
//   warp 14   TMA: the X tile (MP x 128 bf16, two 128-byte-swizzled boxes)
//             into its own ring (X is re-read by every CTA and sits in L2);
//   warps 2-9 dequantize each word into exact bf16 (q - z) values (small
//             integers, so no rounding) and store them in the 128-byte
//             swizzled K-major layout the MMA reads, three groups deep; the
//             zero points of 32 groups are staged in shared memory;
//   warp 1    one lane issues tcgen05.mma kind::f16 into one of four TMEM
//             partial buffers per 128-K group;
//   warps 10-13 multiply each group's partial by its bf16 scale (32 groups
//             staged in shared memory) and accumulate in registers (the
//             scale varies per group and channel, so it cannot be folded
//             into either operand exactly).
// Split-K: the CTAs of one thread-block cluster share an output tile and
// each take a contiguous range of groups; their fp32 partial tiles are summed
// through distributed shared memory, so the kernel needs no global scratch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qlin_internal.h"
#include "tc_ptx.cuh"

namespace qlin {
namespace {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int QW_BYTES = 16 * 128 * 4;     // one 128-K group: 16 k-octets x 128 channels int32
constexpr int A_BYTES = 2 * 128 * 128;     // one group dequantized: two 64-K sub-tiles of 128 x 64 bf16
constexpr int CHUNK = 32;                  // groups whose zero points / scales are staged at a time
constexpr int NP = 4;                      // TMEM partial buffers (groups the MMA may run ahead)
constexpr int THREADS = 480;               // 15 warps, see the role map in k_w4a16

template <int MP>
struct W4Cfg {
    static constexpr int XSUB = MP * 128;                           // one 64-K X sub-tile
    static constexpr int X_BYTES = 2 * XSUB;                        // one group of X
    static constexpr int SA = 3;                                    // dequantized groups in flight
    static constexpr int XS = (MP <= 32) ? 4 : 3;                   // X ring depth (groups)
    static constexpr int QS = (MP <= 32) ? 9 : 7;                   // weight ring depth (groups)
    static constexpr int OFF_A = 0;                                  // SA groups (reused for the reduction)
    static constexpr int OFF_X = OFF_A + SA * A_BYTES;
    static constexpr int OFF_QW = OFF_X + XS * X_BYTES;
    static constexpr int OFF_ZT = OFF_QW + QS * QW_BYTES;           // zero points [CHUNK][256] bytes
    static constexpr int OFF_ST = OFF_ZT + CHUNK * 256;             // scales [CHUNK][128] floats
    static constexpr int OFF_BAR = OFF_ST + CHUNK * 128 * 4;
    static constexpr int NBAR = 2 * QS + 2 * XS + 2 * SA + 2 * NP + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;
    static constexpr uint32_t TMEM_COLS = (NP * MP < 32) ? 32 : NP * MP;
    static constexpr int RED_BYTES = MP * 128 * 4;
    static_assert(RED_BYTES <= SA * A_BYTES, "reduction tile must fit in the A ring");
    static_assert(SMEM <= 232448, "shared memory budget");
    // kind::f16: D f32, A bf16, B bf16, K-major, N = MP, M = 128
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MP >> 3) << 17) |
                                      ((uint32_t)(128 >> 4) << 24);
};

struct W4Params {
    int M, N, K, groups;
    int64_t ldy;
    const uint16_t* scales;   // bf16 [K/128, N]
    const int32_t* qzeros;    // [K/128, N/8]
    uint16_t* y;
    int* status;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; i++)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

__device__ __forceinline__ void record_timeout(int* status, volatile uint32_t* abort_flag) {
    *abort_flag = 1u;
    if (status) atomicExch(status, (int)QLIN_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ float ld_peer_f32(uint32_t local_saddr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Eight 4-bit codes (k = 8o .. 8o+7 in bits [4j, 4j+4)) minus the zero point,
// as eight exact bf16 values: 0x4300 | q is the bf16 for 128 + q, and
// (128 + q) - (128 + z) is an exact small integer.
__device__ __forceinline__ uint4 dequant8(uint32_t w, __nv_bfloat162 bias2) {
    uint32_t h[4];
#pragma unroll
    for (int p = 0; p < 4; p++) {
        const uint32_t t = ((w >> (8 * p)) & 0xFu) | (((w >> (8 * p + 4)) & 0xFu) << 16) | 0x43004300u;
        __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&t);
        v = __hsub2(v, bias2);
        h[p] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

template <int MP>
__global__ void __launch_bounds__(THREADS, 1)
    k_w4a16(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmX, const W4Params p) {
    // Role map: warp 0 weight TMA, warp 1 MMA (and TMEM owner), warps 2-9
    // dequantize (thread d: channel d % 128, sub-tile d / 128 of each group),
    // warps 10-13 epilogue (TMEM lane quadrant = warp % 4), warp 14 X TMA.
    using C = W4Cfg<MP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* qempty = qfull + C::QS;
    uint64_t* xfull = qempty + C::QS;
    uint64_t* xempty = xfull + C::XS;
    uint64_t* afull = xempty + C::XS;
    uint64_t* aempty = afull + C::SA;
    uint64_t* pfull = aempty + C::SA;
    uint64_t* pempty = pfull + NP;
    uint64_t* drain = pempty + NP;
    // tmem, abort, MMA-consumed groups, weight groups issued, X groups issued, dequant-consumed groups
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cs = (int)gridDim.x;                 // cluster size = split-K ways
    const int rank = (int)cluster_rank();
    const int n0 = blockIdx.y * 128, m0 = blockIdx.z * MP;
    const int g0 = (int)((int64_t)p.groups * rank / cs), g1 = (int)((int64_t)p.groups * (rank + 1) / cs);
    const int ng_cta = g1 - g0;                    // 128-K groups of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::QS; s++) {
            mbar_init(qfull + s, 1);
            mbar_init(qempty + s, 8);             // the eight dequant warps
        }
        for (int s = 0; s < C::XS; s++) {
            mbar_init(xfull + s, 1);
            mbar_init(xempty + s, 1);             // the MMA commit
        }
        for (int s = 0; s < C::SA; s++) {
            mbar_init(afull + s, 8);
            mbar_init(aempty + s, 1);
        }
        for (int s = 0; s < NP; s++) {
            mbar_init(pfull + s, 1);
            mbar_init(pempty + s, 4);             // the four epilogue warps
        }
        mbar_init(drain, 1);
        fence_mbar_init();
        misc[1] = (p.status && *reinterpret_cast<volatile int*>(p.status) != 0) ? 1u : 0u;
        for (int i = 2; i < 6; i++) misc[i] = 0;
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) tmem_alloc(misc, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const bool skip = misc[1] != 0;

    float acc[MP];
#pragma unroll
    for (int i = 0; i < MP; i++) acc[i] = 0.0f;
    bool epi_ok = false;

    if (!skip && warp == 0 && lane == 0) {
        // ------------------------------------------------ weight producer (HBM stream)
        for (int t = 0; t < ng_cta; t++) {
            const int s = t % C::QS;
            if (!wait_or_abort(qempty + s, ((uint32_t)(t / C::QS) & 1u) ^ 1u, abort_flag)) {
                record_timeout(p.status, abort_flag);
                break;
            }
            mbar_arrive_expect_tx(qfull + s, QW_BYTES);
            tma_load_2d(smem + C::OFF_QW + s * QW_BYTES, &tmQ, n0, (g0 + t) * 16, qfull + s);
            misc[3] = (uint32_t)(t + 1);
        }
    } else if (!skip && warp == 14 && lane == 0) {
        // ------------------------------------------------ activation producer (L2)
        for (int t = 0; t < ng_cta; t++) {
            const int s = t % C::XS;
            if (!wait_or_abort(xempty + s, ((uint32_t)(t / C::XS) & 1u) ^ 1u, abort_flag)) {
                record_timeout(p.status, abort_flag);
                break;
            }
            const int k = (g0 + t) * 128;
            mbar_arrive_expect_tx(xfull + s, C::X_BYTES);
            tma_load_2d(smem + C::OFF_X + s * C::X_BYTES, &tmX, k, m0, xfull + s);
            tma_load_2d(smem + C::OFF_X + s * C::X_BYTES + C::XSUB, &tmX, k + 64, m0, xfull + s);
            misc[4] = (uint32_t)(t + 1);
        }
    } else if (!skip && warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        for (int t = 0; t < ng_cta; t++) {
            const int sx = t % C::XS, sa = t % C::SA, b = t % NP;
            if (!wait_or_abort(xfull + sx, (uint32_t)(t / C::XS) & 1u, abort_flag) ||
                !wait_or_abort(afull + sa, (uint32_t)(t / C::SA) & 1u, abort_flag) ||
                !wait_or_abort(pempty + b, ((uint32_t)(t / NP) & 1u) ^ 1u, abort_flag)) {
                record_timeout(p.status, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + C::OFF_A + sa * A_BYTES);
            const uint32_t x_base = smem_u32(smem + C::OFF_X + sx * C::X_BYTES);
            const uint32_t d = tmem + (uint32_t)(b * MP);
#pragma unroll
            for (int j = 0; j < 2; j++)
#pragma unroll
                for (int c = 0; c < 4; c++)
                    mma_f16(d, sdesc_sw128(a_base + j * (A_BYTES / 2) + c * 32),
                            sdesc_sw128(x_base + j * C::XSUB + c * 32), C::IDESC, (j > 0 || c > 0) ? 1u : 0u);
            tc_commit(aempty + sa);
            tc_commit(xempty + sx);
            tc_commit(pfull + b);
            misc[2] = (uint32_t)(t + 1);
        }
    } else if (!skip && warp >= 2 && warp < 10) {
        // ------------------------------------------------ dequantizers
        const int d = threadIdx.x - 64;            // 0..255
        const int n = d & 127, half = d >> 7;      // channel, 64-K sub-tile of each group
        const int ng = n0 + n;
        uint8_t* const zt = smem + C::OFF_ZT;      // this thread's column d of [CHUNK][256]
        uint8_t* const a_ring = smem + C::OFF_A;
        for (int t = 0; t < ng_cta; t++) {
            const int s = t % C::QS, sa = t % C::SA;
            if ((t % CHUNK) == 0) {
                for (int i = 0; i < CHUNK && t + i < ng_cta; i++) {
                    uint32_t z = 0;
                    if (ng < p.N)
                        z = ((uint32_t)__ldg(p.qzeros + (int64_t)(g0 + t + i) * (p.N >> 3) + (ng >> 3)) >> (4 * (ng & 7))) & 0xFu;
                    zt[i * 256 + d] = (uint8_t)z;
                }
            }
            if (!warp_wait(qfull + s, (uint32_t)(t / C::QS) & 1u, abort_flag) ||
                !warp_wait(aempty + sa, ((uint32_t)(t / C::SA) & 1u) ^ 1u, abort_flag)) {
                if (lane == 0) record_timeout(p.status, abort_flag);
                break;
            }
            const uint32_t zb = 0x4300u | zt[(t % CHUNK) * 256 + d];
            __nv_bfloat162 bias2;
            *reinterpret_cast<uint32_t*>(&bias2) = zb | (zb << 16);
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(smem + C::OFF_QW + s * QW_BYTES) + half * 8 * 128;
            uint8_t* arow = a_ring + sa * A_BYTES + half * (A_BYTES / 2) + n * 128;
            uint32_t w[8];
#pragma unroll
            for (int o = 0; o < 8; o++) w[o] = qw[o * 128 + n];
#pragma unroll
            for (int o = 0; o < 8; o++)
                *reinterpret_cast<uint4*>(arow + ((o ^ (n & 7)) << 4)) = dequant8(w[o], bias2);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull + sa);
                mbar_arrive(qempty + s);
            }
            if (threadIdx.x == 64) misc[5] = (uint32_t)(t + 1);
        }
    } else if (!skip && warp >= 10 && warp < 14) {
        // ------------------------------------------------ epilogue (scale promotion)
        const int q = warp & 3;
        const int n = q * 32 + lane;
        const int ng = n0 + n;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        float* const st = reinterpret_cast<float*>(smem + C::OFF_ST);   // this thread's column n of [CHUNK][128]
        epi_ok = true;
        for (int t = 0; t < ng_cta; t++) {
            const int b = t % NP;
            if ((t % CHUNK) == 0) {
                for (int i = 0; i < CHUNK && t + i < ng_cta; i++)
                    st[i * 128 + n] = (ng < p.N) ? __bfloat162float(__ushort_as_bfloat16(
                                                       __ldg(p.scales + (int64_t)(g0 + t + i) * p.N + ng)))
                                                 : 0.0f;
            }
            if (!warp_wait(pfull + b, (uint32_t)(t / NP) & 1u, abort_flag)) {
                if (lane == 0) record_timeout(p.status, abort_flag);
                epi_ok = false;
                break;
            }
            tc_fence_after();
            const float sc = st[(t % CHUNK) * 128 + n];
#pragma unroll
            for (int c = 0; c < MP / 16; c++) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(tmem + lane_addr + (uint32_t)(b * MP + c * 16), r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i++) acc[c * 16 + i] = fmaf(sc, __uint_as_float(r[i]), acc[c * 16 + i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty + b);
        }
    }

    // ---------------------------------------------------- drain after an abort
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        // every TMA copy this CTA issued must land before its shared memory goes
        for (uint32_t t = misc[5]; t < misc[3]; t++)
            mbar_wait(qfull + (t % C::QS), (t / C::QS) & 1u, kWaitLimitNs);
        for (uint32_t t = misc[2]; t < misc[4]; t++)
            mbar_wait(xfull + (t % C::XS), (t / C::XS) & 1u, kWaitLimitNs);
    }
    if (*abort_flag && warp == 1 && lane == 0) {
        tc_commit(drain);
        mbar_wait(drain, 0, kWaitLimitNs);
    }
    __syncthreads();

    // ---------------------------------------------------- output
    const bool ok = !*abort_flag;
    float* red = reinterpret_cast<float*>(smem + C::OFF_A);    // [MP][128] fp32, reuses the A ring
    if (cs == 1) {
        if (warp >= 10 && warp < 14 && epi_ok && ok) {
            const int ng = n0 + (warp & 3) * 32 + lane;
            if (ng < p.N) {
#pragma unroll
                for (int m = 0; m < MP; m++)
                    if (m0 + m < p.M)
                        p.y[(int64_t)(m0 + m) * p.ldy + ng] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
            }
        }
    } else {
        if (warp >= 10 && warp < 14) {
            const int n = (warp & 3) * 32 + lane;
#pragma unroll
            for (int m = 0; m < MP; m++) red[m * 128 + n] = (epi_ok && ok) ? acc[m] : 0.0f;
        }
        cluster_sync_all();
        // CTA `rank` sums columns [rank*128/cs, (rank+1)*128/cs) over the cluster.
        const int c0 = rank * 128 / cs, c1 = (rank + 1) * 128 / cs, width = c1 - c0;
        const uint32_t red_s = smem_u32(red);
        for (int idx = threadIdx.x; idx < MP * width; idx += blockDim.x) {
            const int m = idx / width, n = c0 + idx % width;
            float v = 0.0f;
            for (int r = 0; r < cs; r++) v += ld_peer_f32(red_s + (uint32_t)((m * 128 + n) * 4), (uint32_t)r);
            if (m0 + m < p.M && n0 + n < p.N && ok)
                p.y[(int64_t)(m0 + m) * p.ldy + n0 + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
        cluster_sync_all();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

int pick_mp(int64_t M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    return 64;                       // larger M runs as several 64-token tiles
}

// Split-K ways (cluster size) so that the grid is about one wave of SMs.
int pick_split(int64_t tiles, int64_t groups) {
    int cs = 1;
    while (cs < 8 && tiles * cs * 2 <= kNumSMs && groups >= 2 * cs * 2) cs *= 2;
    return cs;
}

template <int MP>
cudaError_t launch_mp(const GemmArgs& a, cudaStream_t st) {
    using C = W4Cfg<MP>;
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap tmQ, tmX;
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)(a.K / 8)};
        cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
        cuuint32_t box[2] = {128, 16};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&tmQ, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(a.w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)MP};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    W4Params p{};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.groups = (int)(a.K / 128);
    p.ldy = a.ldy;
    p.scales = static_cast<const uint16_t*>(a.w_scales);
    p.qzeros = static_cast<const int32_t*>(a.w_zeros);
    p.y = a.y;
    p.status = a.dev_status;

    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_w4a16<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t ntiles = (a.N + 127) / 128, mtiles = (a.M + MP - 1) / MP;
    const int cs = pick_split(ntiles * mtiles, p.groups);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)ntiles, (unsigned)mtiles);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_w4a16<MP>, tmQ, tmX, p);
}

}  // namespace

size_t w4a16_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_gemm_w4a16(const GemmArgs& a, cudaStream_t st) {
    switch (pick_mp(a.M)) {
        case 16: return launch_mp<16>(a, st);
        case 32: return launch_mp<32>(a, st);
        default: return launch_mp<64>(a, st);
    }
}

}  // namespace qlin
