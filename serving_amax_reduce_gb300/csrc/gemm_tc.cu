// Scaled low-precision GEMMs on the sm_103a tensor cores (tcgen05 + TMEM).
//
//   Y[m, n] = bf16( epilogue( sum_k Xq[m, k] * Wq[n, k] ) )
//
// The quantized matmul of "vLLM-Omni 在线量化（Online Quantization）完全指南"
// section "在线量化的底层工作原理" stage 3, for the formats of
// "[vLLM] 기타 양자화: FP8, ModelOpt, INC, TorchAO, Quark" section
// "FP8: vLLM의 핵심 양자화" (per-tensor; per-token x 128x128 block),
// stage 2 of the first page (MXFP8, E8M0 per 32 along K) and
// "vLLM-Omni 量化推理实践" Table 1 (NVFP4 attention projections of the mixed
// FP8/NVFP4 model).  The optional bias epilogue is the fused
// alpha * (A @ B) + bias the first page mentions for Blackwell FP8.
//
// Persistent CTAs (one per SM) walk 128 x 256 output tiles in a grouped
// raster; each CTA runs a warp-specialized pipeline:
//   warp 0   one lane issues TMA loads of the X and W tiles (128-byte
//            swizzle, zero fill past M) and the scale chunks into a
//            4-stage shared-memory ring;
//   warp 1   allocates TMEM; one lane issues tcgen05.mma into the TMEM
//            accumulator and tcgen05.commit to release each stage;
//   warps 2-3 NVFP4 / MXFP4: one lane each copies the stage's X / W scale
//            chunks smem -> TMEM with tcgen05.cp (12 / 6 copies per stage
//            would otherwise serialize with the MMAs on one issuing thread);
//   warps 4-11 (two warpgroups, raised to 232 registers with setmaxnreg)
//            copy the accumulator TMEM -> registers with tcgen05.ld,
//            release it to the next tile's MMAs at once, then apply the
//            scales and write bf16 while that tile's mainloop runs.
// Variants:
//   FP8 per-tensor  kind::f8f6f4, alpha = s_x * s_w in the epilogue.
//   FP8 block       kind::f8f6f4 into one of two TMEM partial buffers per
//                   128-wide K block; the eight epilogue warps promote each
//                   partial with its fp32 weight-block scale (one uniform
//                   load, a block ahead) into register accumulators (fp32
//                   block scales are not an MMA scale type), then multiply
//                   by the per-token scale (or, for 1 x 128 activation
//                   groups, fold each block's X scale into its multiplier).
//   MXFP8           kind::mxf8f6f4.block_scale.scale_vec::1X, UE8M0 scales
//                   copied smem -> TMEM with tcgen05.cp.
//   NVFP4           kind::mxf4nvf4.block_scale.scale_vec::4X, UE4M3 scales,
//                   alpha = g_x * g_w.
//   MXFP4 (W4A4)    kind::mxf4nvf4.block_scale.scale_vec::2X, UE8M0 scales
//                   (the online MXFP4 path of the same page).
//   INT8 (W8A8)     the online INT8 path of the same page, per-token X and
//                   per-channel W scales.  sm_103a has no integer MMA, so TMA
//                   stages the int8 tiles (64 K per stage) in a ring of their
//                   own and warps 12-19 (two more warpgroups) turn every code
//                   into the fp16 value of the same integer (q ^ 0x80 placed
//                   in the mantissa of 1024, minus 1152: exact) in the
//                   128-byte-swizzled layout the MMA reads; kind::f16 then
//                   multiplies exact integers with fp32 accumulation into one of
//                   two TMEM accumulators, and the epilogue applies
//                   s_x[m] * s_w[n].
//   FP8 per-tensor  with the activation quantization fused into the GEMM (the
//   fused X         producer quantizes the X tile): for M <= 128 (one row tile,
//                   the single-request shapes) X arrives in bf16.  The eight
//                   epilogue warps, idle during the mainloop, first take the
//                   tensor amax of X (every CTA's A tile is all of X), then turn
//                   each 128 x 128 bf16 block into E4M3 codes in the 128-byte-
//                   swizzled A stage while TMA brings the W tile, and drain the
//                   accumulator at the end of the tile.  Codes, s_x and the MMA
//                   sequence equal those of qlin_quantize_act + the per-tensor
//                   GEMM, so Y is the same bits; one launch instead of three.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qlin_internal.h"
#include "tc_ptx.cuh"

namespace qlin {
namespace {

using namespace ptx;

enum Kind { kFp8Tensor = 0, kFp8Block = 1, kMxfp8 = 2, kNvfp4 = 3, kMxfp4 = 4, kInt8 = 5, kFp8QX = 6, kMx4Dual = 7 };

constexpr int BM = 128;              // tile rows (X rows) = MMA M
constexpr int BKB = 128;             // K bytes per stage: 128 fp8 or 256 fp4 (one swizzle row)
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // bounded waits give up after 1 s

template <int KIND>
struct Cfg {
    // INT8: operands are converted on chip from an int8 staging ring
    static constexpr bool CVT = (KIND == kInt8);
    // FP8 per-tensor with bf16 X: the epilogue warps quantize the A stages
    static constexpr bool QX = (KIND == kFp8QX);
    static constexpr int BN = 256;
    static constexpr int STAGES = CVT ? 2 : 4;       // operand stages (converted fp16 for INT8)
    static constexpr int S8 = CVT ? 4 : 0;           // int8 staging stages
    static constexpr int EPI_WARPS = 8;              // two per TMEM lane quadrant, 128 columns each
    static constexpr int CVT_WARPS = CVT ? 8 : 0;    // warpgroups 3-4 (INT8 only): int8 -> fp16
    // warpgroup 0: TMA + MMA; warpgroups 1-2: epilogue; warpgroups 3-4: converters
    static constexpr int THREADS = 384 + 32 * CVT_WARPS;
    // setmaxnreg split, within the launch allocation (checked on the host
    // before launch): 128 x 40 + 256 x 232 = 64512 <= 384 x 168, and for INT8
    // 128 x 40 + 256 x 136 + 256 x 80 = 60416 <= 640 x 96.
    static constexpr int REGS_LAUNCH = CVT ? 96 : 168, REGS_CTRL = 40, REGS_EPI = CVT ? 136 : 232;
    static constexpr int REGS_CVT = 80;
    static_assert(128 * REGS_CTRL + 256 * REGS_EPI + 32 * CVT_WARPS * REGS_CVT <= THREADS * REGS_LAUNCH,
                  "register split");
    static constexpr int A_BYTES = BM * BKB;
    static constexpr int B_BYTES = BN * BKB;
    static constexpr int K8 = 64;                    // INT8: K per stage (64 fp16 = one 128-byte row)
    static constexpr int A8_BYTES = CVT ? BM * K8 : 0;
    static constexpr int B8_BYTES = CVT ? BN * K8 : 0;
    // 512-byte scale chunks (128 rows x 4 scales) per 128 rows per stage
    static constexpr bool DUAL = (KIND == kMx4Dual);  // MXFP4 dual-scale: per-512 partials promoted on chip
    static constexpr int SF_CHUNKS =
        (KIND == kMxfp8) ? 1 : (KIND == kNvfp4 ? 4 : ((KIND == kMxfp4 || KIND == kMx4Dual) ? 2 : 0));
    // NVFP4 has 12 scale-chunk copies per stage: two threads issue them off the
    // MMA thread; MXFP8's 3 copies stay with the MMA issuer
    static constexpr bool SPLIT_CP = (KIND == kNvfp4 || KIND == kMxfp4 || KIND == kMx4Dual);
    static constexpr int SFA_BYTES = SF_CHUNKS * 512;
    static constexpr int SFB_BYTES = SF_CHUNKS * 512 * (BN / 128);
    static constexpr int KSTEPS = BKB / 32;          // each MMA consumes 32 bytes of K
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int STG_BOX = 32 * 16 * 2;      // one 32 x 16 bf16 output box
    static constexpr int STG_BUFS = (KIND == kNvfp4) ? 1 : 2;   // staging boxes per epilogue warp
    static constexpr int STG_BYTES = STG_BOX * STG_BUFS;
    static constexpr int OFF_A8 = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr int OFF_B8 = OFF_A8 + S8 * A8_BYTES;
    static constexpr int OFF_STG = OFF_B8 + S8 * B8_BYTES;
    static constexpr int OFF_BAR = OFF_STG + EPI_WARPS * STG_BYTES;
    // full[S], empty[S], accf, acce, pfull[2], pempty[2], drain, sfready[S], s8full[S8], s8empty[S8]
    static constexpr int NBAR = 3 * STAGES + 7 + 2 * S8;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    // dual-scale: each epilogue warp stages its 128 columns' W coarse scales of a block
    static constexpr int OFF_SWS = OFF_MISC + 64;
    static constexpr int SWS_BYTES = DUAL ? EPI_WARPS * 128 * 4 : 0;
    static constexpr int SMEM = OFF_SWS + SWS_BYTES + 1024; // + slack for 1024-byte alignment
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int SFA_COL = 256;
    static constexpr int SFA_COLS = 4 * SF_CHUNKS;             // per stage
    static constexpr int SFB_COL = SFA_COL + STAGES * SFA_COLS;
    static constexpr int SFB_COLS = 4 * SF_CHUNKS * (BN / 128); // per stage
    static_assert(SFB_COL + STAGES * SFB_COLS <= 512, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// Instruction descriptors (M = 128, N = BN, both operands K-major).
template <int KIND>
__host__ __device__ constexpr uint32_t idesc_for() {
    constexpr uint32_t n = (uint32_t)(Cfg<KIND>::BN >> 3) << 17;
    constexpr uint32_t m = (uint32_t)(BM >> 4) << 24;
    if (KIND == kFp8Tensor || KIND == kFp8Block || KIND == kFp8QX)
        return (1u << 4) /* D f32 */ | (0u << 7) /* A e4m3 */ | (0u << 10) /* B e4m3 */ | n | m;
    if (KIND == kInt8)   // kind::f16
        return (1u << 4) /* D f32 */ | (0u << 7) /* A f16 */ | (0u << 10) /* B f16 */ | n | m;
    if (KIND == kMxfp8)
        return (0u << 7) | (0u << 10) | n | (1u << 23) /* UE8M0 scales */ | m;
    if (KIND == kMxfp4 || KIND == kMx4Dual)
        return (1u << 7) /* A e2m1 */ | (1u << 10) /* B e2m1 */ | n | (1u << 23) /* UE8M0 scales */ | m;
    return (1u << 7) /* A e2m1 */ | (1u << 10) /* B e2m1 */ | n | (0u << 23) /* UE4M3 scales */ | m;
}

struct TcParams {
    int M, N, K, nk;
    int64_t ldy;
    const float* x_scale;    // tensor: [1]; block: per-token [M]
    const float* w_scale;    // tensor: [1]; block: [N/128, K/128]
    const float* x_global;   // NVFP4
    const float* w_global;
    const uint8_t* sfa;      // MXFP8 / NVFP4 scales, tensor-core tiling
    const uint8_t* sfb;
    int64_t sf_chunks_per_row;
    const uint16_t* bias;
    uint16_t* y;
    int* status;
    int x_group;             // FP8 block: x_scale is [M, K/128] (1 x 128 groups) instead of [M]
    const uint16_t* xb;      // fused X (FP8 per-tensor): bf16 activations [M <= 128, K], row pitch K
};

__device__ __forceinline__ void record_timeout(int* status, volatile uint32_t* abort_flag) {
    *abort_flag = 1u;
    if (status) atomicExch(status, (int)QLIN_ERR_DEVICE_TIMEOUT);
}

// Wait with the wall-clock bound; also gives up early once another role of
// this CTA has aborted.
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

// Warp-uniform variant for the epilogue warps: lane 0 polls, the verdict is
// broadcast so that the following .sync.aligned TMEM loads stay converged.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag);
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// Four int8 codes (one word, lowest k in the low byte) -> the fp16 values of
// the same four integers as two f16x2 words (lower k in the low half).
// q ^ 0x80 = q + 128 in [0, 255]; as the low mantissa byte under 0x64 it
// reads as the fp16 value 1024 + q + 128, and subtracting 1152 (0x6480)
// leaves q exactly (every integer of magnitude below 2048 is an fp16 value).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = prmt(u, 0x64646464u, 0x5140u);   // bytes u0, 0x64, u1, 0x64
    const uint32_t b = prmt(u, 0x64646464u, 0x5342u);   // bytes u2, 0x64, u3, 0x64
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Write this warp's 32 rows x 32 columns (row = lane, values already scaled)
// at output (m, n) through the warp's shared-memory staging buffer: two
// 32 x 16 bf16 boxes stored by TMA.  Bias (if any) is added here; rows and
// columns outside Y are clipped by the tensor map.
template <int NBUF>
__device__ __forceinline__ void store_block32(const TcParams& p, const CUtensorMap* tmY, uint8_t* stg, int m, int n,
                                              const float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
        uint8_t* box = stg + (hh % NBUF) * (32 * 16 * 2);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            float a = v[hh * 16 + 2 * i], b = v[hh * 16 + 2 * i + 1];
            if (p.bias) {
                const int c = n + hh * 16 + 2 * i;
                if (c < p.N) a += __bfloat162float(__ushort_as_bfloat16(p.bias[c]));
                if (c + 1 < p.N) b += __bfloat162float(__ushort_as_bfloat16(p.bias[c + 1]));
            }
            w[i] = pack_bf16x2(a, b);
        }
        // the box stored NBUF boxes ago has left this staging buffer
        if (lane == 0) {
            if (NBUF == 1) bulk_wait_read_all();
            else asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        }
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(box + lane * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmY, n + hh * 16, m, box);
            bulk_commit_group();
        }
    }
}

// Grouped raster: bands of 16 row blocks; inside a band, consecutive tile
// indices walk down the rows first, so the CTAs running at the same time
// share A row blocks and B column blocks in L2.
template <int BN>
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& m0, int& n0) {
    constexpr int GM = 16;
    const int band = t / (GM * tiles_n);
    const int first_m = band * GM;
    const int gm = min(GM, tiles_m - first_m);
    const int idx = t - band * GM * tiles_n;
    m0 = (first_m + idx % gm) * BM;
    n0 = (idx / gm) * BN;
}

template <int KIND>
__global__ void __launch_bounds__(Cfg<KIND>::THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmY, const TcParams p) {
    using C = Cfg<KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + C::STAGES;
    uint64_t* accf = empty + C::STAGES;     // accumulator ready (non-block kinds)
    uint64_t* acce = accf + 1;              // accumulator drained into registers
    uint64_t* pfull = acce + 1;             // FP8 block: partial buffer b ready
    uint64_t* pempty = pfull + 2;           // FP8 block: partial buffer b drained
    uint64_t* drain = pempty + 2;
    uint64_t* sfready = drain + 1;          // MX / NVFP4: stage s's scale factors are in TMEM
    uint64_t* s8full = sfready + C::STAGES; // INT8: int8 staging slot landed (TMA)
    uint64_t* s8empty = s8full + C::S8;     // INT8: int8 staging slot read by the converters
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);   // tmem base, abort, consumed, issued
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + C::BN - 1) / C::BN;
    const int ntiles = tiles_m * tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            // TMA; or the converter warps (INT8); or TMA plus the epilogue warps (fused X)
            mbar_init(full + s, C::CVT ? C::CVT_WARPS : (C::QX ? 1 + C::EPI_WARPS : 1));
            mbar_init(empty + s, 1);
        }
        for (int s = 0; s < C::S8; s++) {
            mbar_init(s8full + s, 1);
            mbar_init(s8empty + s, C::CVT_WARPS);
        }
        mbar_init(accf, 1);
        mbar_init(acce, C::EPI_WARPS);
        mbar_init(pfull + 0, 1);
        mbar_init(pfull + 1, 1);
        mbar_init(pempty + 0, C::EPI_WARPS);
        mbar_init(pempty + 1, C::EPI_WARPS);
        mbar_init(drain, C::SPLIT_CP ? 3 : 1);   // the MMA issuer (+ the two scale-copy threads)
        for (int s = 0; s < C::STAGES; s++) mbar_init(sfready + s, 2);
        fence_mbar_init();
        // a launch that follows an expired wait does no work
        misc[1] = (p.status && *reinterpret_cast<volatile int*>(p.status) != 0) ? 1u : 0u;
        misc[2] = 0;
        misc[3] = 0;
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) tmem_alloc(misc, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const bool skip = misc[1] != 0;
    // Warpgroup 0 (TMA, MMA, two idle warps) gives registers to the two
    // epilogue warpgroups, which hold a 128-column fp32 tile row each.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CTRL));
    if (C::CVT && !skip && warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (INT8 staging ring)
        if constexpr (C::CVT) {
        uint32_t kg = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            int m0, n0;
            tile_coords<C::BN>(tile, tiles_m, tiles_n, m0, n0);
            for (int kb = 0; kb < p.nk; kb++, kg++) {
                const int j = (int)(kg % C::S8);
                if (!wait_or_abort(s8empty + j, ((kg / C::S8) & 1u) ^ 1u, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(s8full + j, C::A8_BYTES + C::B8_BYTES);
                tma_load_2d(smem + C::OFF_A8 + j * C::A8_BYTES, &tmA, kb * C::K8, m0, s8full + j);
                tma_load_2d(smem + C::OFF_B8 + j * C::B8_BYTES, &tmB, kb * C::K8, n0, s8full + j);
                misc[3] = kg + 1;
            }
        }
        }
    } else if (!C::CVT && !skip && warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t kg = 0;
        const int ntiles_b = (p.N + 127) / 128;
        const int64_t cpr = p.sf_chunks_per_row;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            int m0, n0;
            tile_coords<C::BN>(tile, tiles_m, tiles_n, m0, n0);
            uint32_t bytes = (C::QX ? 0 : C::A_BYTES) + C::B_BYTES;   // fused X: the A stage is written on chip
            if (C::SF_CHUNKS) {
                bytes += C::SFA_BYTES;
                for (int j = 0; j < C::BN / 128; j++)
                    if ((n0 >> 7) + j < ntiles_b) bytes += C::SF_CHUNKS * 512;
            }
            for (int kb = 0; kb < p.nk; kb++, kg++) {
                const int s = (int)(kg % C::STAGES);
                const uint32_t ph = (kg / C::STAGES) & 1u;
                if (!wait_or_abort(empty + s, ph ^ 1u, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full + s, bytes);
                if (!C::QX) tma_load_2d(smem + C::OFF_A + s * C::A_BYTES, &tmA, kb * BKB, m0, full + s);
                tma_load_2d(smem + C::OFF_B + s * C::B_BYTES, &tmB, kb * BKB, n0, full + s);
                if (C::SF_CHUNKS) {
                    bulk_load(smem + C::OFF_SFA + s * C::SFA_BYTES,
                              p.sfa + (((int64_t)(m0 >> 7) * cpr + (int64_t)kb * C::SF_CHUNKS) << 9), C::SFA_BYTES,
                              full + s);
                    for (int j = 0; j < C::BN / 128; j++) {
                        const int nt = (n0 >> 7) + j;
                        if (nt < ntiles_b)
                            bulk_load(smem + C::OFF_SFB + s * C::SFB_BYTES + j * C::SF_CHUNKS * 512,
                                      p.sfb + (((int64_t)nt * cpr + (int64_t)kb * C::SF_CHUNKS) << 9),
                                      C::SF_CHUNKS * 512, full + s);
                    }
                }
                misc[3] = kg + 1;
            }
        }
    } else if (!skip && warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_for<KIND>();
        uint32_t kg = 0, kbg = 0, it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, it++) {
            if (C::CVT) {
                // INT8: two accumulator buffers (2 x 256 columns); wait until the
                // epilogue has drained the one this tile reuses
                if (!wait_or_abort(pempty + (it & 1u), ((it >> 1) & 1u) ^ 1u, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
            } else if (KIND != kFp8Block && !C::DUAL) {
                if (!wait_or_abort(acce, (it & 1u) ^ 1u, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
            }
            for (int kb = 0; kb < p.nk; kb++, kg++) {
                const int s = (int)(kg % C::STAGES);
                const uint32_t ph = (kg / C::STAGES) & 1u;
                if (!wait_or_abort(full + s, ph, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok = false;
                    break;
                }
                uint32_t d = C::CVT ? tmem + (it & 1u) * (uint32_t)C::BN : tmem;
                if (KIND == kFp8Block) {
                    const int b = (int)(kbg & 1u);
                    if (!wait_or_abort(pempty + b, ((kbg >> 1) & 1u) ^ 1u, abort_flag)) {
                        record_timeout(p.status, abort_flag);
                        ok = false;
                        break;
                    }
                    d = tmem + (uint32_t)(b * C::BN);
                }
                if (C::DUAL && (kb & 1) == 0) {
                    // one 512-K partial (two stages) at a time in columns [0, BN): wait until
                    // the epilogue has read the previous one
                    if (!wait_or_abort(pempty, (kbg & 1u) ^ 1u, abort_flag)) {
                        record_timeout(p.status, abort_flag);
                        ok = false;
                        break;
                    }
                }
                if (C::SPLIT_CP && !wait_or_abort(sfready + s, ph, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + C::OFF_A + s * C::A_BYTES);
                const uint32_t b_base = smem_u32(smem + C::OFF_B + s * C::B_BYTES);
                if (KIND == kMxfp8) {
                    const uint32_t sfa_base = smem_u32(smem + C::OFF_SFA + s * C::SFA_BYTES);
                    const uint32_t sfb_base = smem_u32(smem + C::OFF_SFB + s * C::SFB_BYTES);
                    tmem_cp_32x128b_x4(tmem + C::SFA_COL + s * C::SFA_COLS, sdesc_sf(sfa_base));
#pragma unroll
                    for (int j = 0; j < C::BN / 128; j++)
                        tmem_cp_32x128b_x4(tmem + C::SFB_COL + s * C::SFB_COLS + j * 4, sdesc_sf(sfb_base + j * 512));
                }
#pragma unroll
                for (int c = 0; c < C::KSTEPS; c++) {
                    const uint64_t ad = sdesc_sw128(a_base + c * 32);
                    const uint64_t bd = sdesc_sw128(b_base + c * 32);
                    const uint32_t acc =
                        (KIND == kFp8Block) ? (c > 0) : (C::DUAL ? ((kb & 1) || c > 0) : (kb > 0 || c > 0));
                    if (KIND == kFp8Tensor || KIND == kFp8Block || KIND == kFp8QX) {
                        mma_f8f6f4(d, ad, bd, idesc, acc);
                    } else if (KIND == kInt8) {
                        mma_f16(d, ad, bd, idesc, acc);
                    } else if (KIND == kMxfp8) {
                        const uint32_t id = idesc | ((uint32_t)c << 4) | ((uint32_t)c << 29);
                        mma_mxf8(d, ad, bd, id, tmem + C::SFA_COL + s * C::SFA_COLS,
                                 tmem + C::SFB_COL + s * C::SFB_COLS, acc);
                    } else if (KIND == kMxfp4 || KIND == kMx4Dual) {
                        // chunk c/2 holds the scales of two MMAs; the ids 0 / 2 select the pair
                        const uint32_t sf = (uint32_t)(c & 1) * 2u;
                        const uint32_t id = idesc | (sf << 4) | (sf << 29);
                        mma_mxf4(d, ad, bd, id, tmem + C::SFA_COL + s * C::SFA_COLS + (c >> 1) * 4,
                                 tmem + C::SFB_COL + s * C::SFB_COLS + (c >> 1) * 4 * (C::BN / 128), acc);
                    } else {
                        mma_nvf4(d, ad, bd, idesc, tmem + C::SFA_COL + s * C::SFA_COLS + c * 4,
                                 tmem + C::SFB_COL + s * C::SFB_COLS + c * 4 * (C::BN / 128), acc);
                    }
                }
                tc_commit(empty + s);
                if (KIND == kFp8Block) {
                    tc_commit(pfull + (kbg & 1u));
                    kbg++;
                }
                if (C::DUAL && (kb & 1) == 1) {
                    tc_commit(pfull);
                    kbg++;
                }
                misc[2] = kg + 1;
            }
            if (ok && C::CVT) tc_commit(pfull + (it & 1u));
            else if (ok && KIND != kFp8Block && !C::DUAL) tc_commit(accf);
        }
    } else if (!skip && C::SPLIT_CP && (warp == 2 || warp == 3) && lane == 0) {
        // ------------------------------------------------ scale-factor copies (NVFP4)
        // smem -> TMEM with tcgen05.cp, off the MMA thread: warp 2 copies the
        // X scales, warp 3 the W scales, into the stage's TMEM slot; the MMA
        // thread waits for both commits.  A slot is rewritten only after the
        // stage's TMA has landed again, i.e. after the MMAs that read it ended.
        uint32_t kg = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            for (int kb = 0; kb < p.nk; kb++, kg++) {
                const int s = (int)(kg % C::STAGES);
                const uint32_t ph = (kg / C::STAGES) & 1u;
                if (!wait_or_abort(full + s, ph, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok = false;
                    break;
                }
                const uint32_t sfa_base = smem_u32(smem + C::OFF_SFA + s * C::SFA_BYTES);
                const uint32_t sfb_base = smem_u32(smem + C::OFF_SFB + s * C::SFB_BYTES);
                if (warp == 2) {
#pragma unroll
                    for (int c = 0; c < C::SF_CHUNKS; c++)
                        tmem_cp_32x128b_x4(tmem + C::SFA_COL + s * C::SFA_COLS + c * 4, sdesc_sf(sfa_base + c * 512));
                } else {
#pragma unroll
                    for (int c = 0; c < C::SF_CHUNKS; c++)
#pragma unroll
                        for (int j = 0; j < C::BN / 128; j++)
                            tmem_cp_32x128b_x4(tmem + C::SFB_COL + s * C::SFB_COLS + c * 4 * (C::BN / 128) + j * 4,
                                               sdesc_sf(sfb_base + (j * C::SF_CHUNKS + c) * 512));
                }
                tc_commit(sfready + s);
            }
        }
    }
    } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_EPI));
    if (!skip) {
        // ------------------------------------------------ epilogue (8 warps)
        const int q = warp & 3;                 // TMEM lane quadrant this warp may read
        const int h = (warp - 4) >> 2;          // which 128-column half of the tile
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        float alpha = 1.0f;
        if (KIND == kFp8Tensor) alpha = __fmul_rn(__ldg(p.x_scale), __ldg(p.w_scale));
        if (KIND == kNvfp4) alpha = __fmul_rn(__ldg(p.x_global), __ldg(p.w_global));
        const int et = (warp - 4) * 32 + lane;  // fused X: this thread among the 256 epilogue threads
        float rx = 1.0f;                        // fused X: the code multiplier 448 / amax
        if constexpr (C::QX) {
            // Tensor amax of X (M <= 128 rows, all of them in this CTA's A tile),
            // 32 vectors in flight per thread, then over the eight warps.
            const uint32_t nvr = (uint32_t)(p.K >> 3), nvec = (uint32_t)p.M * nvr;
            float a = 0.0f;
            for (uint32_t v0 = (uint32_t)et; v0 < nvec; v0 += 256u * 32u) {
                uint4 t[32];
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const uint32_t v = v0 + (uint32_t)j * 256u;
                    if (v < nvec) {
                        const uint32_t r = v / nvr;
                        t[j] = __ldg(reinterpret_cast<const uint4*>(p.xb + (int64_t)r * p.K + (int64_t)(v - r * nvr) * 8));
                    } else {
                        t[j] = make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const uint32_t w[4] = {t[j].x, t[j].y, t[j].z, t[j].w};
#pragma unroll
                    for (int e = 0; e < 4; e++)
                        a = fmaxf(a, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            if (lane == 0) misc[4 + (warp - 4)] = __float_as_uint(a);
            asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight epilogue warps
#pragma unroll
            for (int w = 0; w < C::EPI_WARPS; w++) a = fmaxf(a, __uint_as_float(misc[4 + w]));
            // the per-tensor FP8 granule: s = amax / 448, codes E4M3(x * (448 / amax))
            float sx = 1.0f;
            if (a != 0.0f) {
                sx = __fdiv_rn(a, 448.0f);
                rx = __fdiv_rn(448.0f, a);
            }
            alpha = __fmul_rn(sx, __ldg(p.w_scale));
        }
        uint32_t it = 0, kbg = 0, kq = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, it++) {
            int m0, n0;
            tile_coords<C::BN>(tile, tiles_m, tiles_n, m0, n0);
            const int row = m0 + q * 32 + lane;
            const int ncol = n0 + h * 128;
            bool ok = true;
            if constexpr (C::QX) {
                // Quantize this tile's X blocks (128 rows x 128 K bf16 -> E4M3) into
                // the A stages: thread et takes 16-code chunk et & 7 of rows
                // et / 8 + 32 i, i = 0..3, stored at chunk position c ^ (row & 7)
                // (the 128-byte swizzle); the loads run two blocks ahead.
                const int c = et & 7, sw = (et >> 3) & 7;
                auto load_x = [&](int kb, uint4 (&d)[8]) {
                    const int k = kb * 128 + c * 16;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int r = m0 + i * 32 + (et >> 3);
                        const bool in = r < p.M && k < p.K;
                        const uint16_t* src = p.xb + (int64_t)r * p.K + k;
                        d[2 * i] = in ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
                        d[2 * i + 1] = in ? __ldg(reinterpret_cast<const uint4*>(src + 8)) : make_uint4(0, 0, 0, 0);
                    }
                };
                uint4 nv[8], nv2[8];
                load_x(0, nv);
                if (p.nk > 1) load_x(1, nv2);
                for (int kb = 0; kb < p.nk; kb++, kq++) {
                    uint4 cv[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        cv[i] = nv[i];
                        nv[i] = nv2[i];
                    }
                    if (kb + 2 < p.nk) load_x(kb + 2, nv2);
                    const int s = (int)(kq % C::STAGES);
                    if (!warp_wait_or_abort(empty + s, ((kq / C::STAGES) & 1u) ^ 1u, abort_flag)) {
                        if (lane == 0) record_timeout(p.status, abort_flag);
                        ok = false;
                        break;
                    }
                    uint8_t* a_st = smem + C::OFF_A + s * C::A_BYTES;
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const uint32_t w[8] = {cv[2 * i].x, cv[2 * i].y, cv[2 * i].z, cv[2 * i].w,
                                               cv[2 * i + 1].x, cv[2 * i + 1].y, cv[2 * i + 1].z, cv[2 * i + 1].w};
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            const uint32_t lo = cvt_e4m3x2(__fmul_rn(__uint_as_float(w[2 * j] << 16), rx),
                                                           __fmul_rn(__uint_as_float(w[2 * j] & 0xFFFF0000u), rx));
                            const uint32_t hi = cvt_e4m3x2(__fmul_rn(__uint_as_float(w[2 * j + 1] << 16), rx),
                                                           __fmul_rn(__uint_as_float(w[2 * j + 1] & 0xFFFF0000u), rx));
                            o[j] = lo | (hi << 16);
                        }
                        const int r = i * 32 + (et >> 3);
                        *reinterpret_cast<uint4*>(a_st + r * 128 + ((c ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    fence_proxy_async_smem();         // generic-proxy writes -> the MMA's async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full + s);
                }
                if (!ok) break;
            }
            if constexpr (C::CVT) {
                // INT8: accumulator buffer it & 1, read in two 64-column halves
                // (fewer registers) and released after the second
                const uint32_t b = it & 1u;
                if (!warp_wait_or_abort(pfull + b, (it >> 1) & 1u, abort_flag)) {
                    if (lane == 0) record_timeout(p.status, abort_flag);
                    break;
                }
                tc_fence_after();
                uint8_t* stg = smem + C::OFF_STG + (warp - 4) * C::STG_BYTES;
                const float sxr = row < p.M ? __ldg(p.x_scale + row) : 0.0f;
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t r[2][32];
#pragma unroll
                    for (int c = 0; c < 2; c++)
                        tmem_ld_32x32b_x32(tmem + lane_addr + b * (uint32_t)C::BN + (uint32_t)(h * 128 + (2 * hh + c) * 32),
                                           r[c]);
                    tmem_ld_wait();
                    if (hh == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(pempty + b);   // the MMA may reuse this buffer
                    }
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        const int col0 = ncol + (2 * hh + c) * 32;
                        if (col0 < p.N) {
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; i++) {
                                const int col = col0 + i;
                                v[i] = __uint_as_float(r[c][i]) * sxr * (col < p.N ? __ldg(p.w_scale + col) : 0.0f);
                            }
                            store_block32<C::STG_BUFS>(p, &tmY, stg, m0 + q * 32, col0, v);
                        }
                    }
                }
            } else if (KIND != kFp8Block && !C::DUAL) {
                if (!warp_wait_or_abort(accf, it & 1u, abort_flag)) {
                    if (lane == 0) record_timeout(p.status, abort_flag);
                    break;
                }
                tc_fence_after();
                uint32_t r[4][32];
#pragma unroll
                for (int c = 0; c < 4; c++)
                    tmem_ld_32x32b_x32(tmem + lane_addr + (uint32_t)(h * 128 + c * 32), r[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce);     // the MMA may start the next tile
                uint8_t* stg = smem + C::OFF_STG + (warp - 4) * C::STG_BYTES;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    if (ncol + c * 32 < p.N) {
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[c][i]) * alpha;
                        store_block32<C::STG_BUFS>(p, &tmY, stg, m0 + q * 32, ncol + c * 32, v);
                    }
                }
            } else if constexpr (C::DUAL) {
                // MXFP4 dual-scale: each 512-K partial (two stages), scaled by the row's and
                // the column's coarse scales of that block.  The warp stages its 128 columns'
                // W coarse scales of the block in its own shared slot (4 per lane, loaded a
                // block ahead), so the multipliers come from broadcast reads.
                const int nblk = p.K >> 9;
                const bool row_ok = row < p.M;
                const float* const sxrow = p.x_scale + (int64_t)(row_ok ? row : 0) * nblk;
                float* const sws = reinterpret_cast<float*>(smem + C::OFF_SWS) + (warp - 4) * 128;
                float sx_next = row_ok ? __ldg(sxrow) : 0.0f;
                float swn[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int col = ncol + lane + 32 * i;
                    swn[i] = col < p.N ? __ldg(p.w_scale + (int64_t)col * nblk) : 0.0f;
                }
                uint64_t acc2[64];                  // 128 fp32 accumulators as (lo, hi) pairs
#pragma unroll
                for (int i = 0; i < 64; i++) acc2[i] = 0ull;
                for (int b = 0; b < nblk; b++, kbg++) {
                    const float sx = sx_next;
                    __syncwarp();                   // every lane is done with the previous block's slot
#pragma unroll
                    for (int i = 0; i < 4; i++) sws[lane + 32 * i] = swn[i];
                    __syncwarp();
                    if (b + 1 < nblk) {
                        sx_next = row_ok ? __ldg(sxrow + b + 1) : 0.0f;
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int col = ncol + lane + 32 * i;
                            swn[i] = col < p.N ? __ldg(p.w_scale + (int64_t)col * nblk + b + 1) : 0.0f;
                        }
                    }
                    if (!warp_wait_or_abort(pfull, kbg & 1u, abort_flag)) {
                        if (lane == 0) record_timeout(p.status, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // two 64-column loads; the partial's columns are released after the second
                    const uint32_t pbase = tmem + lane_addr + (uint32_t)(h * 128);
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        uint32_t r[64];
                        tmem_ld_32x32b_x64(pbase + (uint32_t)(c * 64), r);
                        tmem_ld_wait();
                        if (c == 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(pempty);
                        }
#pragma unroll
                        for (int i = 0; i < 32; i++) {
                            const float m0 = sx * sws[c * 64 + 2 * i], m1 = sx * sws[c * 64 + 2 * i + 1];
                            acc2[c * 32 + i] = ffma2(pack_f32x2(__float_as_uint(m0), __float_as_uint(m1)),
                                                     pack_f32x2(r[2 * i], r[2 * i + 1]), acc2[c * 32 + i]);
                        }
                    }
                }
                if (!ok) break;
                uint8_t* stg = smem + C::OFF_STG + (warp - 4) * C::STG_BYTES;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    if (ncol + c * 32 < p.N) {
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 16; i++) unpack_f32x2(acc2[c * 16 + i], v[2 * i], v[2 * i + 1]);
                        store_block32<C::STG_BUFS>(p, &tmY, stg, m0 + q * 32, ncol + c * 32, v);
                    }
                }
            } else {
                const int nt = ncol >> 7;
                const bool col_ok = ncol < p.N;
                const int kblocks = p.K >> 7;
                // per-token X scale (applied once at the end), or with 1 x 128 groups
                // one X scale per block, folded into that block's multiplier
                const bool xg = p.x_group != 0, row_ok = row < p.M;
                const float sx = xg ? 1.0f : (row_ok ? __ldg(p.x_scale + row) : 0.0f);
                const float* const sxrow = p.x_scale + (int64_t)(row_ok ? row : 0) * kblocks;
                float sxg_next = xg ? (row_ok ? __ldg(sxrow) : 0.0f) : 1.0f;
                // this half-tile's weight-block scales: one uniform load per block,
                // issued a block ahead so that its latency is hidden
                const float* const swrow = p.w_scale + (int64_t)(col_ok ? nt : 0) * kblocks;
                float sw_next = col_ok ? __ldg(swrow) : 0.0f;
                uint64_t acc2[64];                  // 128 fp32 accumulators as (lo, hi) pairs
#pragma unroll
                for (int i = 0; i < 64; i++) acc2[i] = 0ull;
                for (int kb = 0; kb < p.nk; kb++, kbg++) {
                    const float sw = sw_next * sxg_next;
                    if (col_ok && kb + 1 < kblocks) sw_next = __ldg(swrow + kb + 1);
                    if (xg && row_ok && kb + 1 < kblocks) sxg_next = __ldg(sxrow + kb + 1);
                    const int b = (int)(kbg & 1u);
                    if (!warp_wait_or_abort(pfull + b, (kbg >> 1) & 1u, abort_flag)) {
                        if (lane == 0) record_timeout(p.status, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // two 64-column loads; the buffer is released after the second
                    const uint32_t pbase = tmem + lane_addr + (uint32_t)(b * C::BN + h * 128);
                    const uint64_t swp = pack_f32x2(__float_as_uint(sw), __float_as_uint(sw));
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        uint32_t r[64];
                        tmem_ld_32x32b_x64(pbase + (uint32_t)(c * 64), r);
                        tmem_ld_wait();
                        if (c == 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(pempty + b);
                        }
#pragma unroll
                        for (int i = 0; i < 32; i++)
                            acc2[c * 32 + i] = ffma2(swp, pack_f32x2(r[2 * i], r[2 * i + 1]), acc2[c * 32 + i]);
                    }
                }
                if (!ok) break;
                uint8_t* stg = smem + C::OFF_STG + (warp - 4) * C::STG_BYTES;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    if (ncol + c * 32 < p.N) {
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 16; i++) {
                            unpack_f32x2(acc2[c * 16 + i], v[2 * i], v[2 * i + 1]);
                            v[2 * i] *= sx;
                            v[2 * i + 1] *= sx;
                        }
                        store_block32<C::STG_BUFS>(p, &tmY, stg, m0 + q * 32, ncol + c * 32, v);
                    }
                }
            }
        }
    }

    if (lane == 0) bulk_wait_all();              // this warp's output stores have completed
    } else {
        if constexpr (C::CVT) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CVT));
        if (!skip) {
            // ------------------------------------------------ int8 -> fp16 converters (8 warps)
            // A stage holds 384 rows (128 of X, 256 of W) of 64 int8 = 4 chunks
            // of 16 codes; thread ct (0..255) takes chunk ct & 3 of rows
            // ct / 4 + 64 i, i = 0..5 (8 rows per warp per round: 128 contiguous
            // staging bytes per quarter warp).
            // Chunk c of row r becomes 16-byte fp16 chunks 2c and 2c + 1 of the
            // row's 128 bytes, stored at chunk position (2c [+1]) ^ (r & 7):
            // the 128-byte swizzle the MMA descriptors expect (8-row atoms).
            const int ct = (warp - 12) * 32 + lane;
            uint32_t kg = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < p.nk; kb++, kg++) {
                    const int j = (int)(kg % C::S8), s = (int)(kg % C::STAGES);
                    if (!warp_wait_or_abort(s8full + j, (kg / C::S8) & 1u, abort_flag) ||
                        !warp_wait_or_abort(empty + s, ((kg / C::STAGES) & 1u) ^ 1u, abort_flag)) {
                        if (lane == 0) record_timeout(p.status, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint8_t* a8 = smem + C::OFF_A8 + j * C::A8_BYTES;
                    const uint8_t* b8 = smem + C::OFF_B8 + j * C::B8_BYTES;
                    uint8_t* a16 = smem + C::OFF_A + s * C::A_BYTES;
                    uint8_t* b16 = smem + C::OFF_B + s * C::B_BYTES;
                    // a batch of chunks is read before any is stored: stores may not
                    // be ordered before loads the compiler cannot prove disjoint,
                    // which would serialize load -> convert -> store chunk by chunk
                    constexpr int TPR = 32 * C::CVT_WARPS / 4;   // rows per round
                    constexpr int ROUNDS = (BM + C::BN) / TPR, BATCH = ROUNDS / 2;
                    const int c = ct & 3, sw = (ct >> 2) & 7;   // same chunk and swizzle row every round
#pragma unroll
                    for (int i0 = 0; i0 < ROUNDS; i0 += BATCH) {
                        uint4 qv[BATCH];
#pragma unroll
                        for (int i = 0; i < BATCH; i++) {
                            const int r = (i0 + i) * TPR + (ct >> 2);  // rows < BM come from X
                            const uint8_t* src = r < BM ? a8 + r * C::K8 : b8 + (r - BM) * C::K8;
                            qv[i] = *reinterpret_cast<const uint4*>(src + c * 16);
                        }
#pragma unroll
                        for (int i = 0; i < BATCH; i++) {
                            const int r = (i0 + i) * TPR + (ct >> 2);
                            uint8_t* row = r < BM ? a16 + r * 128 : b16 + (r - BM) * 128;
                            uint4 h0, h1;
                            i8x4_to_f16x4(qv[i].x, h0.x, h0.y);
                            i8x4_to_f16x4(qv[i].y, h0.z, h0.w);
                            i8x4_to_f16x4(qv[i].z, h1.x, h1.y);
                            i8x4_to_f16x4(qv[i].w, h1.z, h1.w);
                            *reinterpret_cast<uint4*>(row + (((2 * c) ^ sw) << 4)) = h0;
                            *reinterpret_cast<uint4*>(row + (((2 * c + 1) ^ sw) << 4)) = h1;
                        }
                    }
                    fence_proxy_async_smem();         // generic-proxy writes -> the MMA's async proxy
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(s8empty + j);
                        mbar_arrive(full + s);
                    }
                }
            }
        }
        }
    }

    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        // Let every TMA copy this CTA issued land before its shared memory is
        // released: wait (bounded) on the stages issued but not consumed.
        const uint32_t issued = misc[3];
        if constexpr (C::CVT) {
            // at most the last S8 staging loads can still be in flight; a
            // load whose phase already completed passes at once
            for (uint32_t kg = issued > (uint32_t)C::S8 ? issued - C::S8 : 0u; kg < issued; kg++)
                mbar_wait(s8full + (kg % C::S8), (kg / C::S8) & 1u, kWaitLimitNs);
        } else {
            for (uint32_t kg = misc[2]; kg < issued; kg++)
                mbar_wait(full + (kg % C::STAGES), (kg / C::STAGES) & 1u, kWaitLimitNs);
        }
    }
    if (*abort_flag && lane == 0 && (warp == 1 || (C::SPLIT_CP && (warp == 2 || warp == 3)))) {
        // ... and every MMA / scale copy issued has finished reading shared
        // memory (a commit with nothing outstanding arrives at once)
        tc_commit(drain);
        if (warp == 1) mbar_wait(drain, 0, kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
int num_sms() {
    static const int n = [] {     // initialised once, thread-safe
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            return v;
        return kNumSMs;
    }();
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {     // looked up once, thread-safe
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// Byte matrix [rows, inner_bytes] with row pitch `pitch` bytes, box of
// box_rows x box_inner bytes (128-byte swizzle for the MMA operand tiles, none
// for the INT8 staging tiles), zero fill outside the matrix.
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint64_t pitch,
                  uint32_t box_rows, uint32_t box_inner = BKB, bool swizzle = true) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner_bytes, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t launch_tc(const GemmArgs& a, cudaStream_t st) {
    using C = Cfg<KIND>;
    const uint64_t kbytes = (KIND == kNvfp4 || KIND == kMxfp4 || KIND == kMx4Dual) ? (uint64_t)a.K / 2 : (uint64_t)a.K;
    CUtensorMap tmA, tmB;
    if (C::CVT) {
        if (!make_tmap_u8(&tmA, a.x, kbytes, (uint64_t)a.M, kbytes, BM, C::K8, false) ||
            !make_tmap_u8(&tmB, a.w, kbytes, (uint64_t)a.N, kbytes, C::BN, C::K8, false))
            return cudaErrorInvalidValue;
    } else if (C::QX) {
        // fused X: no A tiles are loaded; tmA is a valid copy of the W map (only prefetched)
        if (!make_tmap_u8(&tmB, a.w, kbytes, (uint64_t)a.N, kbytes, C::BN)) return cudaErrorInvalidValue;
        tmA = tmB;
    } else {
        if (!make_tmap_u8(&tmA, a.x, kbytes, (uint64_t)a.M, kbytes, BM)) return cudaErrorInvalidValue;
        if (!make_tmap_u8(&tmB, a.w, kbytes, (uint64_t)a.N, kbytes, C::BN)) return cudaErrorInvalidValue;
    }
    CUtensorMap tmY;
    {
        auto fn = encode_fn();
        cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.M};
        cuuint64_t strides[1] = {(cuuint64_t)a.ldy * 2};
        cuuint32_t box[2] = {16, 32};
        cuuint32_t estr[2] = {1, 1};
        if (!fn || fn(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.y, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    TcParams p{};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.nk = C::CVT ? (int)((a.K + C::K8 - 1) / C::K8) : (int)((kbytes + BKB - 1) / BKB);
    p.ldy = a.ldy;
    p.x_scale = static_cast<const float*>(a.x_scales);
    p.w_scale = static_cast<const float*>(a.w_scales);
    p.x_global = a.x_global;
    p.w_global = a.w_global;
    p.sfa = static_cast<const uint8_t*>(a.x_scales);
    p.sfb = static_cast<const uint8_t*>(a.w_scales);
    p.sf_chunks_per_row = (KIND == kMxfp8 || KIND == kMxfp4 || KIND == kMx4Dual) ? a.K / 128 : a.K / 64;
    if (KIND == kMx4Dual) {      // the coarse scales: [M, K/512] and [N, K/512]
        p.x_scale = a.x_global;
        p.w_scale = a.w_global;
    }
    p.bias = a.bias;
    p.y = a.y;
    p.status = a.dev_status;
    p.x_group = a.x_group128 ? 1 : 0;
    p.xb = static_cast<const uint16_t*>(a.x);
    // Several threads may run this setup at once; it is idempotent.
    static std::atomic<bool> attr_set{false};
    if (!attr_set.load(std::memory_order_acquire)) {
        // The in-kernel setmaxnreg split assumes the launch allocation of
        // REGS_LAUNCH registers per thread; refuse to launch otherwise.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k_gemm_tc<KIND>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != C::REGS_LAUNCH) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(k_gemm_tc<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set.store(true, std::memory_order_release);
    }
    const int64_t ntiles = ((a.N + C::BN - 1) / C::BN) * ((a.M + BM - 1) / BM);
    const int grid = (int)(ntiles < num_sms() ? ntiles : num_sms());   // persistent: one CTA per SM
    k_gemm_tc<KIND><<<grid, C::THREADS, C::SMEM, st>>>(tmA, tmB, tmY, p);
    return cudaGetLastError();
}

__global__ void k_expire_wait(int* status, uint32_t max_polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        bool done = false;
        for (uint32_t i = 0; i < max_polls && !done; i++) done = mbar_try_wait(&bar, 0);
        if (!done) atomicExch(status, (int)QLIN_ERR_DEVICE_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_gemm_fp8_tensor(const GemmArgs& a, cudaStream_t st) { return launch_tc<kFp8Tensor>(a, st); }
cudaError_t launch_gemm_fp8_block(const GemmArgs& a, cudaStream_t st) { return launch_tc<kFp8Block>(a, st); }
cudaError_t launch_gemm_mxfp8(const GemmArgs& a, cudaStream_t st) { return launch_tc<kMxfp8>(a, st); }
cudaError_t launch_gemm_nvfp4(const GemmArgs& a, cudaStream_t st) { return launch_tc<kNvfp4>(a, st); }
cudaError_t launch_gemm_mxfp4(const GemmArgs& a, cudaStream_t st) { return launch_tc<kMxfp4>(a, st); }
cudaError_t launch_gemm_mxfp4_dual(const GemmArgs& a, cudaStream_t st) { return launch_tc<kMx4Dual>(a, st); }
cudaError_t launch_gemm_int8(const GemmArgs& a, cudaStream_t st) { return launch_tc<kInt8>(a, st); }
cudaError_t launch_gemm_fp8_tensor_fused_x(const GemmArgs& a, cudaStream_t st) { return launch_tc<kFp8QX>(a, st); }

cudaError_t launch_debug_expire_wait(int* dev_status, uint32_t max_polls, cudaStream_t st) {
    k_expire_wait<<<1, 32, 0, st>>>(dev_status, max_polls);
    return cudaGetLastError();
}

}  // namespace qlin
