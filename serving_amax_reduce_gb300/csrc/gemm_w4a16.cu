// W4A16 decode GEMM: Y[M, N] = X[M, K] (bf16) . dequant(W)^T (+ bias) with W
// stored as int4 asymmetric codes, group 128 along K, GPTQ-style packing
// ("vLLM-Omni는 AutoRound 양자화로 추론을 가속화합니다", section "새로운 모델
// 양자화": bits 4, group_size 128, packing auto_round:auto_gptq).
//
//   Y[m, n] = sum_g s[g, n] * sum_{k in g} x[m, k] * (q[k, n] - z[g, n])
//
// Two kernels.  For M <= 16, k_w4a16_mma (further down) dequantizes in
// registers and feeds warp-level mma.sync: at 16 tokens a tcgen05 MMA has
// N = 16 and the tensor pipe is bound by its per-instruction cost.  For larger
// M, k_w4a16 below runs tcgen05 with the output channels on the MMA's M side
// ("swap AB"): a CTA owns 128 channels and MP = 64 tokens (zero-filled past M
// by TMA; larger M runs as several token tiles).
// Per 128-K group:
//   warp 0    TMA: the packed int4 words (16 k-octets x 128 channels, 8 KB)
//             into a deep ring, so that enough HBM reads are in flight;
//   warp 14   TMA: the X tile (MP x 128 bf16, two 128-byte-swizzled boxes)
//             into its own ring (X is re-read by every CTA and sits in L2);
//   warps 2-9 dequantize, in two sets of four warps that take alternate
//             groups: each thread owns one channel, turns its 16 words into
//             128 exact bf16 (q - z) values (small integers, so no rounding)
//             and writes them with one tcgen05.st into the group's tensor
//             memory stage, which the MMA reads as its A operand; the set
//             also permutes the group's X tile within 8-element K chunks to
//             the order in which the dequantized pairs come out;
//   warps 1, 15 one lane each issues the group's tcgen05.mma kind::f16 (A from
//             tensor memory, X from shared memory) into the group's TMEM
//             partial buffer; the two issuers take alternate groups, which
//             doubles the rate at which small MMAs enter the tensor pipe;
//   warps 10-13 multiply each group's partial by its bf16 scale (staged in
//             shared memory) and accumulate in registers: the scale varies per
//             group and channel, so it cannot be folded into either operand
//             exactly.
// Split-K: the CTAs of one thread-block cluster share an output tile and
// each take a contiguous range of groups; their fp32 partial tiles are summed
// through distributed shared memory, so the kernel needs no global scratch.
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

constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int QW_BYTES = 16 * 128 * 4;     // one 128-K group: 16 k-octets x 128 channels int32
constexpr int A_COLS = 64;                 // TMEM columns per dequantized group (128 K as bf16 pairs)
constexpr int ZCH = 16;                    // groups of one dequant set whose zero points are staged at a time
constexpr int SCH = 16;                    // groups whose scales are staged at a time (epilogue)
constexpr uint32_t TMEM_COLS = 512;

template <int MP>
struct W4Cfg {
    // Dequant sets of four warps take groups in turn.  (Four sets measured no
    // faster than two: the tensor pipe's small-MMA rate and the handoffs bound
    // a group, not the dequant arithmetic.)
    static constexpr int NSETS = 2;
    static constexpr int E0 = 2 + 4 * NSETS;                        // first epilogue warp
    static constexpr int THREADS = 32 * (E0 + 6);                   // + 4 epilogue, X producer, odd MMA issuer
    static constexpr int XSUB = MP * 128;                           // one 64-K X sub-tile
    static constexpr int X_BYTES = 2 * XSUB;                        // one group of X
    // One ring of R group slots: a TMEM A stage, an X slot in shared memory and
    // a TMEM partial buffer move together, so that one commit per group frees
    // the A stage and the X slot and announces the partial (the tensor pipe
    // takes a commit about as slowly as a small MMA).  R is even, so that each
    // slot always belongs to the same one of the two MMA issuers.
    static constexpr int R = 4;
    static constexpr int RA = R, RP = R, XS = R;
    static constexpr int QS = (MP <= 32) ? 16 : 12;                 // weight ring depth (groups)
    static constexpr int OFF_QW = 0;                                // weight ring
    static constexpr int OFF_X = OFF_QW + QS * QW_BYTES;
    static constexpr int OFF_ZT = OFF_X + XS * X_BYTES;             // zero points [2 sets][ZCH][128] bytes
    static constexpr int OFF_ST = OFF_ZT + NSETS * ZCH * 128;       // scales [SCH][128] floats
    static constexpr int OFF_RED = OFF_ST + SCH * 128 * 4;          // split-K partial tile [MP][128] fp32
    static constexpr int OFF_BAR = OFF_RED + MP * 128 * 4;
    static constexpr int NBAR = 2 * QS + 4 * R + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;
    static constexpr uint32_t P_COL = RA * A_COLS;                  // partial buffers follow the A stages
    static_assert(P_COL + RP * MP <= TMEM_COLS, "tensor memory budget");
    static_assert(RA % 2 == 0 && RP % 2 == 0, "stages alternate between the two issuers");
    static_assert(X_BYTES % 1024 == 0 && OFF_X % 1024 == 0, "128-byte-swizzled tiles need 1 KB alignment");
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
    const uint16_t* bias;     // bf16 [N] or null
    uint16_t* y;
    int* status;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
    if (mbar_test_wait(bar, parity)) return true;          // usually complete already: no suspend
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

// Load from the shared memory of CTA `rank` of this cluster (ordered by the
// cluster barrier that precedes the reduction, so independent loads may overlap).
__device__ __forceinline__ float ld_peer_f32(uint32_t local_saddr, uint32_t rank) {
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
    return v;
}

// Eight 4-bit codes (k = 8o .. 8o+7 in bits [4j, 4j+4)) minus the zero point,
// as eight exact bf16 values: 0x4300 | q is the bf16 for 128 + q, and
// (128 + q) - (128 + z) is an exact small integer.  The codes are taken two at
// a time from bits [4j, 4j+4) and [4j+16, 4j+20), so the pairs come out as
// (k0, k4), (k1, k5), (k2, k6), (k3, k7): every 8-element K chunk of the A
// operand is in the order 0 4 1 5 2 6 3 7, and the X tile is permuted the
// same way (permute_x_chunk), which leaves each dot product unchanged.
__device__ __forceinline__ void dequant8(uint32_t w, __nv_bfloat162 bias2, uint32_t* out) {
    constexpr uint32_t kMask = 0x000F000Fu, kMagic = 0x43004300u;
    uint32_t v[4];
    v[0] = lop3_and_or(w, kMask, kMagic);
    v[1] = lop3_and_or(w >> 4, kMask, kMagic);
    v[2] = lop3_and_or(w >> 8, kMask, kMagic);
    v[3] = lop3_and_or(w >> 12, kMask, kMagic);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        __nv_bfloat162 h = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v[i]), bias2);
        out[i] = *reinterpret_cast<uint32_t*>(&h);
    }
}

// One 16-byte chunk of X (k0 .. k7, bf16) into the order 0 4 1 5 2 6 3 7.
__device__ __forceinline__ uint4 permute_x_chunk(uint4 c) {
    return make_uint4(prmt(c.x, c.z, 0x5410u), prmt(c.x, c.z, 0x7632u), prmt(c.y, c.w, 0x5410u),
                      prmt(c.y, c.w, 0x7632u));
}

template <int MP>
__global__ void __launch_bounds__(W4Cfg<MP>::THREADS, 1)
    k_w4a16(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmX, const W4Params p) {
    // Role map: warp 0 weight TMA, warp 1 MMA for even groups (and TMEM owner),
    // warps 2 .. E0-1 dequantize in NSETS sets of four (set s takes the groups
    // t % NSETS == s; TMEM lane quadrant = warp % 4), warps E0 .. E0+3 epilogue
    // (quadrant = warp % 4), warp E0+4 X TMA, warp E0+5 MMA for odd groups.
    using C = W4Cfg<MP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* qempty = qfull + C::QS;
    uint64_t* xfull = qempty + C::QS;    // slot r: X loaded (TMA)
    uint64_t* afull = xfull + C::R;      // slot r: A stage written and X permuted
    uint64_t* done = afull + C::R;       // slot r: its MMAs finished (A stage, X slot free; partial ready)
    uint64_t* pempty = done + C::R;      // slot r: the epilogue has read the partial
    uint64_t* drain = pempty + C::R;
    // tmem, abort, -, weight groups issued, X groups issued
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cs = (int)gridDim.x;                 // cluster size = split-K ways
    const int rank = (int)cluster_ctarank();
    const int n0 = blockIdx.y * 128, m0 = blockIdx.z * MP;
    const int g0 = (int)((int64_t)p.groups * rank / cs), g1 = (int)((int64_t)p.groups * (rank + 1) / cs);
    const int ng_cta = g1 - g0;                    // 128-K groups of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::QS; s++) {
            mbar_init(qfull + s, 1);
            mbar_init(qempty + s, 4);             // the four warps of one dequant set
        }
        for (int s = 0; s < C::R; s++) {
            mbar_init(xfull + s, 1);
            mbar_init(afull + s, 4);              // the four warps of one dequant set
            mbar_init(done + s, 1);               // one MMA commit per group
            mbar_init(pempty + s, 4);             // the four epilogue warps
        }
        mbar_init(drain, 2);                      // both MMA issuers
        fence_mbar_init();
        misc[1] = (p.status && *reinterpret_cast<volatile int*>(p.status) != 0) ? 1u : 0u;
        for (int i = 2; i < 6; i++) misc[i] = 0;
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) tmem_alloc(misc, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const bool skip = misc[1] != 0;

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
    } else if (!skip && warp == C::E0 + 4 && lane == 0) {
        // ------------------------------------------------ activation producer (L2)
        for (int t = 0; t < ng_cta; t++) {
            const int s = t % C::R;
            if (!wait_or_abort(done + s, ((uint32_t)(t / C::R) & 1u) ^ 1u, abort_flag)) {
                record_timeout(p.status, abort_flag);
                break;
            }
            const int k = (g0 + t) * 128;
            mbar_arrive_expect_tx(xfull + s, C::X_BYTES);
            tma_load_2d(smem + C::OFF_X + s * C::X_BYTES, &tmX, k, m0, xfull + s);
            tma_load_2d(smem + C::OFF_X + s * C::X_BYTES + C::XSUB, &tmX, k + 64, m0, xfull + s);
            misc[4] = (uint32_t)(t + 1);
        }
    } else if (!skip && (warp == 1 || warp == C::E0 + 5) && lane == 0) {
        // ------------------------------------------------ MMA issuers (even / odd groups)
        for (int t = (warp == 1) ? 0 : 1; t < ng_cta; t += 2) {
            const int a = t % C::RA, pb = t % C::RP, sx = t % C::XS;
            // afull: the dequant set has written A and permuted this group's X tile
            if (!wait_or_abort(afull + a, (uint32_t)(t / C::RA) & 1u, abort_flag) ||
                !wait_or_abort(pempty + pb, ((uint32_t)(t / C::RP) & 1u) ^ 1u, abort_flag)) {
                record_timeout(p.status, abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t a_t = tmem + (uint32_t)(a * A_COLS);
            const uint32_t x_base = smem_u32(smem + C::OFF_X + sx * C::X_BYTES);
            const uint32_t d = tmem + C::P_COL + (uint32_t)(pb * MP);
#pragma unroll
            for (int j = 0; j < 2; j++)
#pragma unroll
                for (int c = 0; c < 4; c++)
                    mma_f16_ta(d, a_t + (uint32_t)((j * 4 + c) * 8), sdesc_sw128(x_base + j * C::XSUB + c * 32),
                               C::IDESC, (j > 0 || c > 0) ? 1u : 0u);
            tc_commit(done + a);
        }
    } else if (!skip && warp >= 2 && warp < C::E0) {
        // ------------------------------------------------ dequantizers
        const int set = (warp - 2) >> 2;           // takes groups t with t % NSETS == set
        const int quad = warp & 3;                 // the TMEM lanes this warp may write
        const int n = quad * 32 + lane;            // channel of the tile = TMEM lane = row of A
        const int ng = n0 + n;
        uint8_t* const zt = smem + C::OFF_ZT + set * (ZCH * 128);   // column n of [ZCH][128]
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        int u = 0;                                 // index of t among this set's groups
        for (int t = set; t < ng_cta; t += C::NSETS, u++) {
            if ((u % ZCH) == 0) {
                // the zero points of this set's next ZCH groups, all loads in flight at once
                uint32_t zw[ZCH];
#pragma unroll
                for (int i = 0; i < ZCH; i++)
                    zw[i] = (ng < p.N && t + C::NSETS * i < ng_cta)
                                ? (uint32_t)__ldg(p.qzeros + (int64_t)(g0 + t + C::NSETS * i) * (p.N >> 3) + (ng >> 3))
                                : 0u;
#pragma unroll
                for (int i = 0; i < ZCH; i++) zt[i * 128 + n] = (uint8_t)((zw[i] >> (4 * (ng & 7))) & 0xFu);
            }
            const int s = t % C::QS, a = t % C::RA, sx = t % C::XS;
            if (!warp_wait(xfull + sx, (uint32_t)(t / C::XS) & 1u, abort_flag) ||
                !warp_wait(qfull + s, (uint32_t)(t / C::QS) & 1u, abort_flag)) {
                if (lane == 0) record_timeout(p.status, abort_flag);
                break;
            }
            {
                // this group's X tile (MP x 128 bf16 = MP * 16 chunks), permuted in place
                uint4* xc = reinterpret_cast<uint4*>(smem + C::OFF_X + sx * C::X_BYTES);
#pragma unroll
                for (int i = 0; i < MP / 8; i++) xc[i * 128 + n] = permute_x_chunk(xc[i * 128 + n]);
                fence_proxy_async_smem();            // the MMA reads X through the async proxy
            }
            const uint32_t zb = 0x4300u | zt[(u % ZCH) * 128 + n];
            __nv_bfloat162 bias2;
            *reinterpret_cast<uint32_t*>(&bias2) = zb | (zb << 16);
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(smem + C::OFF_QW + s * QW_BYTES);
            uint32_t w[16];
#pragma unroll
            for (int o = 0; o < 16; o++) w[o] = qw[o * 128 + n];
            __syncwarp();
            if (lane == 0) mbar_arrive(qempty + s);   // the words are in registers: the slot may refill
            uint32_t av[64];
#pragma unroll
            for (int o = 0; o < 16; o++) dequant8(w[o], bias2, av + 4 * o);
            // only the TMEM write waits for the slot's previous MMAs, so the
            // loads and the arithmetic above overlap them
            if (!warp_wait(done + a, ((uint32_t)(t / C::RA) & 1u) ^ 1u, abort_flag)) {
                if (lane == 0) record_timeout(p.status, abort_flag);
                break;
            }
            tc_fence_after();
            tmem_st_32x32b_x64(tmem + lane_addr + (uint32_t)(a * A_COLS), av);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull + a);
        }
    } else if (!skip && warp >= C::E0 && warp < C::E0 + 4) {
        // ------------------------------------------------ epilogue (scale promotion)
        const int q = warp & 3;
        const int n = q * 32 + lane;
        const int ng = n0 + n;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        float* const st = reinterpret_cast<float*>(smem + C::OFF_ST);   // this thread's column n of [SCH][128]
        float acc[MP];
#pragma unroll
        for (int i = 0; i < MP; i++) acc[i] = 0.0f;
        bool epi_ok = true;
        for (int t = 0; t < ng_cta; t++) {
            const int pb = t % C::RP;
            if ((t % SCH) == 0) {
                // batches of loads in flight at once (smaller batches where acc is large)
                constexpr int SB = (MP >= 64) ? 8 : SCH;
#pragma unroll
                for (int i0 = 0; i0 < SCH; i0 += SB) {
                    uint16_t sw[SB];
#pragma unroll
                    for (int i = 0; i < SB; i++)
                        sw[i] = (ng < p.N && t + i0 + i < ng_cta)
                                    ? __ldg(p.scales + (int64_t)(g0 + t + i0 + i) * p.N + ng)
                                    : (uint16_t)0;
#pragma unroll
                    for (int i = 0; i < SB; i++)
                        st[(i0 + i) * 128 + n] = __bfloat162float(__ushort_as_bfloat16(sw[i]));
                }
            }
            if (!warp_wait(done + pb, (uint32_t)(t / C::RP) & 1u, abort_flag)) {
                if (lane == 0) record_timeout(p.status, abort_flag);
                epi_ok = false;
                break;
            }
            tc_fence_after();
            const float sc = st[(t % SCH) * 128 + n];
#pragma unroll
            for (int c = 0; c < MP / 16; c++) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + lane_addr + C::P_COL + (uint32_t)(pb * MP + c * 16), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i++) acc[c * 16 + i] = fmaf(sc, __uint_as_float(v[i]), acc[c * 16 + i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty + pb);
        }
        // every group of this CTA is in acc once the loop ran to the end
        if (cs == 1) {
            if (epi_ok && ng < p.N) {
                const float b = p.bias ? __bfloat162float(__ushort_as_bfloat16(p.bias[ng])) : 0.0f;
#pragma unroll
                for (int m = 0; m < MP; m++)
                    if (m0 + m < p.M)
                        p.y[(int64_t)(m0 + m) * p.ldy + ng] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m] + b));
            }
        } else {
            float* const red = reinterpret_cast<float*>(smem + C::OFF_RED);
#pragma unroll
            for (int m = 0; m < MP; m++) red[m * 128 + n] = epi_ok ? acc[m] : 0.0f;
        }
    }

    // ---------------------------------------------------- drain after an abort
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        // every TMA copy this CTA issued must land before its shared memory goes;
        // a ring slot's latest phase covers every earlier copy into it
        const int wq = (int)misc[3], wx = (int)misc[4];
        for (int t = (wq > C::QS ? wq - C::QS : 0); t < wq; t++)
            mbar_wait(qfull + (t % C::QS), (uint32_t)(t / C::QS) & 1u, kWaitLimitNs);
        for (int t = (wx > C::XS ? wx - C::XS : 0); t < wx; t++)
            mbar_wait(xfull + (t % C::XS), (uint32_t)(t / C::XS) & 1u, kWaitLimitNs);
    }
    if (*abort_flag && (warp == 1 || warp == C::E0 + 5) && lane == 0) {
        tc_commit(drain);                          // each issuer's own MMAs
        mbar_wait(drain, 0, kWaitLimitNs);
    }
    __syncthreads();

    // ---------------------------------------------------- split-K reduction over the cluster
    const bool ok = !*abort_flag;
    if (cs > 1) {
        const float* red = reinterpret_cast<const float*>(smem + C::OFF_RED);
        cluster_sync_all();
        // CTA `rank` sums columns [rank*128/cs, (rank+1)*128/cs) over the cluster.
        const int c0 = rank * 128 / cs, c1 = (rank + 1) * 128 / cs, width = c1 - c0;
        const uint32_t red_s = smem_u32(red);
        for (int idx = threadIdx.x; idx < MP * width; idx += blockDim.x) {
            const int m = idx / width, n = c0 + idx % width;
            const uint32_t off = red_s + (uint32_t)((m * 128 + n) * 4);
            float part[8];
#pragma unroll
            for (int r = 0; r < 8; r++) part[r] = (r < cs) ? ld_peer_f32(off, (uint32_t)r) : 0.0f;
            float v = 0.0f;
#pragma unroll
            for (int r = 0; r < 8; r++) v += part[r];
            if (m0 + m < p.M && n0 + n < p.N && ok) {
                const float b = p.bias ? __bfloat162float(__ushort_as_bfloat16(p.bias[n0 + n])) : 0.0f;
                p.y[(int64_t)(m0 + m) * p.ldy + n0 + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + b));
            }
        }
        cluster_sync_all();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- M <= 16: warp-level MMA
// At 16 tokens each tcgen05 MMA of the kernel above has N = 16 and the tensor
// pipe is bound by its per-instruction cost.  This variant dequantizes in
// registers: the packed words stream through a cp.async ring in shared memory
// (three pairs of groups ahead), each lane turns its int4 codes into exact
// bf16 (q - z) values (the same 0x4300 trick) and feeds them straight to
// mma.sync.m16n8k16 (tokens = the MMA's 16 rows, 8 channels per instruction).
//
// CTA = 128 channels x this cluster rank's 128-K groups; 8 warps: warp w takes
// the 32 channels (w & 3) * 32 and the groups of parity w >> 2.  In a warp,
// lane group c4 = lane / 4 owns the 4 consecutive channels 4 c4 + t, one per
// n8 tile t (MMA column c4 of tile t), so its weights come as one 16-byte
// shared-memory read per 8-K octet.  For a 16-K step the B fragment of lane q = lane % 4
// needs 4 codes: they are taken from octet q / 2 as the pairs (j, j + 4) and
// (j + 1, j + 5), j = 2 (q % 2); X is staged with every 8-K octet in the order
// 0 4 1 5 2 6 3 7, which puts the four matching A values of a row at positions
// 4q .. 4q + 3 (one 8-byte load), the same logical K order on both sides.
// Split-K runs over the cluster exactly as above.
constexpr int kXRow = 144;          // bf16 per staged X row: 128 + 16 (8-byte A loads hit 32 banks)
constexpr int kWRow = 136;          // 32-bit words per staged weight octet row: 128 + 8 (conflict-free 16-byte reads)
constexpr int kWPairs = 3;          // weight ring depth, in pairs of groups
constexpr int kMmaSmem = (2 * 2 * 16 * kXRow) * 2 + 16 * 128 * 4 + (2 * kWPairs) * 16 * kWRow * 4;

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 bytes global -> shared, bypassing L1; src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Codes in bits [sh, sh + 4) and [sh + 16, sh + 20) minus the zero point: an
// exact bf16 pair.
__device__ __forceinline__ uint32_t dq_pair(uint32_t w, int sh, __nv_bfloat162 bias2) {
    const uint32_t v = lop3_and_or(w >> sh, 0x000F000Fu, 0x43004300u);
    __nv_bfloat162 h = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), bias2);
    return *reinterpret_cast<uint32_t*>(&h);
}

struct W4MmaParams {
    int M, N, K, groups;
    int64_t ldy;
    const int32_t* qweight;   // [K/8, N]
    const uint16_t* x;        // bf16 [M, K]
    const uint16_t* scales;   // bf16 [K/128, N]
    const int32_t* qzeros;    // [K/128, N/8]
    const uint16_t* bias;
    uint16_t* y;
};

__global__ void __launch_bounds__(256, 2) k_w4a16_mma(const W4MmaParams p) {
    extern __shared__ __align__(16) uint8_t smem_mma[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_mma);                         // [2 buf][2 parity][16][kXRow]
    float* red = reinterpret_cast<float*>(smem_mma + 2 * 2 * 16 * kXRow * 2);      // [16][128]
    uint32_t* wsm = reinterpret_cast<uint32_t*>(smem_mma + 2 * 2 * 16 * kXRow * 2 + 16 * 128 * 4);  // [slot][16][kWRow]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int slice = warp & 3, par = warp >> 2, c4 = lane >> 2, q = lane & 3;
    const int cs = (int)gridDim.x, rank = (int)cluster_ctarank();
    const int n0 = (int)blockIdx.y * 128, m0 = (int)blockIdx.z * 16;
    const int g0 = rank * p.groups / cs, g1 = (rank + 1) * p.groups / cs;
    const int npairs = (g1 - g0 + 1) / 2;
    const int chb = n0 + slice * 32 + 4 * c4;           // this lane's 4 B-fragment channels
    const bool bok = chb < p.N;                          // N % 8 == 0: all 4 or none
    const int chs = n0 + slice * 32 + 8 * q;             // the 8 channels of this lane's C columns
    const int sh0 = 8 * (q & 1);                         // pair (j, j + 4), j = 2 (q % 2)

    // X of a pair of groups (16 rows x 16 octets each), two octets per thread
    auto load_x = [&](int pr, uint4 (&xv)[2]) {
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int idx = tid + 256 * j, pa = idx >> 8, row = (idx >> 4) & 15, oct = idx & 15;
            const int g = g0 + 2 * pr + pa;
            const bool in = g < g1 && m0 + row < p.M;
            xv[j] = in ? __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)(m0 + row) * p.K + g * 128 + oct * 8))
                       : make_uint4(0, 0, 0, 0);
        }
    };
    auto store_x = [&](int buf, const uint4 (&xv)[2]) {
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int idx = tid + 256 * j, pa = idx >> 8, row = (idx >> 4) & 15, oct = idx & 15;
            *reinterpret_cast<uint4*>(xs + ((buf * 2 + pa) * 16 + row) * kXRow + oct * 8) = permute_x_chunk(xv[j]);
        }
    };
    // weights of a pair of groups into ring slots: 2 x 16 octet rows x 32 chunks of 16 bytes
    auto issue_w = [&](int pp) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = tid + 256 * j, pa = c >> 9, row = (c >> 5) & 15, cc = c & 31;
            const int g = g0 + 2 * pp + pa, slot = 2 * (pp % kWPairs) + pa;
            const bool in = g < g1 && n0 + cc * 4 < p.N;
            const int32_t* src = p.qweight + (int64_t)(in ? g * 16 + row : 0) * p.N + (in ? n0 + cc * 4 : 0);
            cp_async16(wsm + (slot * 16 + row) * kWRow + cc * 4, src, in ? 16u : 0u);
        }
        cp_async_commit();
    };

    float acc[4][4];
#pragma unroll
    for (int t = 0; t < 4; t++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[t][i] = 0.0f;

#pragma unroll
    for (int pp = 0; pp < kWPairs; pp++) issue_w(pp);   // empty pairs still commit, keeping the count
    uint4 xv[2];
    load_x(0, xv);
    store_x(0, xv);
    if (npairs > 1) load_x(1, xv);
    for (int pr = 0; pr < npairs; pr++) {
        const int g = g0 + 2 * pr + par;
        const int buf = pr & 1;
        cp_async_wait<kWPairs - 1>();                     // this pair's weights have landed
        __syncthreads();
        // this group's zero points (B channels) and scales (C columns)
        __nv_bfloat162 zb[4];
        float sc[8];
        {
            const bool gin = g < g1;
            const uint32_t zw = (bok && gin) ? (uint32_t)__ldg(p.qzeros + (int64_t)g * (p.N / 8) + chb / 8) : 0u;
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const uint16_t zbits = (uint16_t)(0x4300u | ((zw >> (4 * ((chb & 7) + t))) & 0xFu));
                zb[t] = __halves2bfloat162(__ushort_as_bfloat16(zbits), __ushort_as_bfloat16(zbits));
            }
            const uint4 sv = (gin && chs < p.N) ? __ldg(reinterpret_cast<const uint4*>(p.scales + (int64_t)g * p.N + chs))
                                                : make_uint4(0, 0, 0, 0);
            const uint32_t s2[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                sc[2 * i] = __uint_as_float(s2[i] << 16);
                sc[2 * i + 1] = __uint_as_float(s2[i] & 0xFFFF0000u);
            }
        }
        float cg[4][4];
#pragma unroll
        for (int t = 0; t < 4; t++)
#pragma unroll
            for (int i = 0; i < 4; i++) cg[t][i] = 0.0f;
        const uint16_t* xr = xs + (buf * 2 + par) * 16 * kXRow;
        const uint32_t* wr = wsm + (2 * (pr % kWPairs) + par) * 16 * kWRow + (slice * 32 + 4 * c4);
#pragma unroll
        for (int st = 0; st < 8; st++) {
            const uint2 ar0 = *reinterpret_cast<const uint2*>(xr + c4 * kXRow + 16 * st + 4 * q);
            const uint2 ar1 = *reinterpret_cast<const uint2*>(xr + (c4 + 8) * kXRow + 16 * st + 4 * q);
            const uint4 wv = *reinterpret_cast<const uint4*>(wr + (2 * st + (q >> 1)) * kWRow);
            const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const uint32_t b0 = dq_pair(w4[t], sh0, zb[t]);
                const uint32_t b1 = dq_pair(w4[t], sh0 + 4, zb[t]);
                mma_16816(cg[t], ar0.x, ar1.x, ar0.y, ar1.y, b0, b1);
            }
        }
        // C columns 2q, 2q + 1 of tile t are channels chs + t and chs + 4 + t
#pragma unroll
        for (int t = 0; t < 4; t++) {
            acc[t][0] += cg[t][0] * sc[t];
            acc[t][1] += cg[t][1] * sc[4 + t];
            acc[t][2] += cg[t][2] * sc[t];
            acc[t][3] += cg[t][3] * sc[4 + t];
        }
        // stage the next pair's X (the buffer read two pairs ago is free since the barrier above)
        if (pr + 1 < npairs) store_x(buf ^ 1, xv);
        if (pr + 2 < npairs) load_x(pr + 2, xv);
        __syncthreads();                                  // this pair's weight slots are free
        issue_w(pr + kWPairs);
    }
    cp_async_wait<0>();

    // the two group parities into one partial tile: rows c4 and c4 + 8
    const int cb = slice * 32 + 8 * q;
    if (par == 0) {
#pragma unroll
        for (int t = 0; t < 4; t++) {
            red[c4 * 128 + cb + t] = acc[t][0];
            red[c4 * 128 + cb + 4 + t] = acc[t][1];
            red[(c4 + 8) * 128 + cb + t] = acc[t][2];
            red[(c4 + 8) * 128 + cb + 4 + t] = acc[t][3];
        }
    }
    __syncthreads();
    if (par == 1) {
#pragma unroll
        for (int t = 0; t < 4; t++) {
            red[c4 * 128 + cb + t] += acc[t][0];
            red[c4 * 128 + cb + 4 + t] += acc[t][1];
            red[(c4 + 8) * 128 + cb + t] += acc[t][2];
            red[(c4 + 8) * 128 + cb + 4 + t] += acc[t][3];
        }
    }
    __syncthreads();
    // split-K over the cluster: CTA `rank` sums columns [rank*128/cs, (rank+1)*128/cs)
    if (cs > 1) cluster_sync_all();
    const int col0 = rank * 128 / cs, col1 = (rank + 1) * 128 / cs, width = col1 - col0;
    const uint32_t red_s = smem_u32(red);
    for (int idx = tid; idx < 16 * width; idx += 256) {
        const int m = idx / width, n = col0 + idx % width;
        float v = 0.0f;
        if (cs > 1) {
            const uint32_t off = red_s + (uint32_t)((m * 128 + n) * 4);
            float part[8];
#pragma unroll
            for (int r = 0; r < 8; r++) part[r] = (r < cs) ? ld_peer_f32(off, (uint32_t)r) : 0.0f;
#pragma unroll
            for (int r = 0; r < 8; r++) v += part[r];
        } else {
            v = red[m * 128 + n];
        }
        if (m0 + m < p.M && n0 + n < p.N) {
            const float b = p.bias ? __bfloat162float(__ushort_as_bfloat16(p.bias[n0 + n])) : 0.0f;
            p.y[(int64_t)(m0 + m) * p.ldy + n0 + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + b));
        }
    }
    if (cs > 1) cluster_sync_all();
}

// M <= 8: the same ring and staging with the roles of the MMA operands swapped.
// The weights are the A operand (16 channels per instruction, rows c4 and
// c4 + 8 of two 16-channel m-tiles per warp) and the tokens the B operand (8
// per instruction), so a 16-K step costs two MMAs per warp instead of four.
// The K order is the one above: lane q's A values of a step are the pairs
// (j, j + 4) and (j + 1, j + 5), j = 2 (q % 2), of octet q / 2, and its B values
// the staged X positions 4q .. 4q + 3 of token c4 (one 8-byte read).
__global__ void __launch_bounds__(256, 2) k_w4a16_mma8(const W4MmaParams p) {
    extern __shared__ __align__(16) uint8_t smem_mma[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_mma);                         // [2 buf][2 parity][16][kXRow]
    float* red = reinterpret_cast<float*>(smem_mma + 2 * 2 * 16 * kXRow * 2);      // [16][128]
    uint32_t* wsm = reinterpret_cast<uint32_t*>(smem_mma + 2 * 2 * 16 * kXRow * 2 + 16 * 128 * 4);  // [slot][16][kWRow]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int slice = warp & 3, par = warp >> 2, c4 = lane >> 2, q = lane & 3;
    const int cs = (int)gridDim.x, rank = (int)cluster_ctarank();
    const int n0 = (int)blockIdx.y * 128, m0 = 0;
    const int g0 = rank * p.groups / cs, g1 = (rank + 1) * p.groups / cs;
    const int npairs = (g1 - g0 + 1) / 2;
    // this lane's 4 A-fragment channels (rows c4 and c4 + 8 of m-tiles 0 and 1), CTA-local
    int chl[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; mt++)
#pragma unroll
        for (int r = 0; r < 2; r++) chl[mt][r] = slice * 32 + mt * 16 + c4 + 8 * r;
    const int sh0 = 8 * (q & 1);                         // pair (j, j + 4), j = 2 (q % 2)

    // X of a pair of groups (16 rows x 16 octets each), two octets per thread
    auto load_x = [&](int pr, uint4 (&xv)[2]) {
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int idx = tid + 256 * j, pa = idx >> 8, row = (idx >> 4) & 15, oct = idx & 15;
            const int g = g0 + 2 * pr + pa;
            const bool in = g < g1 && m0 + row < p.M;
            xv[j] = in ? __ldg(reinterpret_cast<const uint4*>(p.x + (int64_t)(m0 + row) * p.K + g * 128 + oct * 8))
                       : make_uint4(0, 0, 0, 0);
        }
    };
    auto store_x = [&](int buf, const uint4 (&xv)[2]) {
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int idx = tid + 256 * j, pa = idx >> 8, row = (idx >> 4) & 15, oct = idx & 15;
            *reinterpret_cast<uint4*>(xs + ((buf * 2 + pa) * 16 + row) * kXRow + oct * 8) = permute_x_chunk(xv[j]);
        }
    };
    // weights of a pair of groups into ring slots: 2 x 16 octet rows x 32 chunks of 16 bytes
    auto issue_w = [&](int pp) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = tid + 256 * j, pa = c >> 9, row = (c >> 5) & 15, cc = c & 31;
            const int g = g0 + 2 * pp + pa, slot = 2 * (pp % kWPairs) + pa;
            const bool in = g < g1 && n0 + cc * 4 < p.N;
            const int32_t* src = p.qweight + (int64_t)(in ? g * 16 + row : 0) * p.N + (in ? n0 + cc * 4 : 0);
            cp_async16(wsm + (slot * 16 + row) * kWRow + cc * 4, src, in ? 16u : 0u);
        }
        cp_async_commit();
    };

    float acc[2][4];
#pragma unroll
    for (int t = 0; t < 2; t++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[t][i] = 0.0f;

#pragma unroll
    for (int pp = 0; pp < kWPairs; pp++) issue_w(pp);   // empty pairs still commit, keeping the count
    uint4 xv[2];
    load_x(0, xv);
    store_x(0, xv);
    if (npairs > 1) load_x(1, xv);
    for (int pr = 0; pr < npairs; pr++) {
        const int g = g0 + 2 * pr + par;
        const int buf = pr & 1;
        cp_async_wait<kWPairs - 1>();                     // this pair's weights have landed
        __syncthreads();
        // this group's zero points and scales for the lane's 4 A rows (channels)
        __nv_bfloat162 zb[2][2];
        float sc[2][2];
        {
            const bool gin = g < g1;
#pragma unroll
            for (int mt = 0; mt < 2; mt++)
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    const int ch = n0 + chl[mt][r];
                    const bool ok = gin && ch < p.N;
                    const uint32_t zw = ok ? (uint32_t)__ldg(p.qzeros + (int64_t)g * (p.N / 8) + ch / 8) : 0u;
                    const uint16_t zbits = (uint16_t)(0x4300u | ((zw >> (4 * (ch & 7))) & 0xFu));
                    zb[mt][r] = __halves2bfloat162(__ushort_as_bfloat16(zbits), __ushort_as_bfloat16(zbits));
                    sc[mt][r] = ok ? __uint_as_float((uint32_t)__ldg(p.scales + (int64_t)g * p.N + ch) << 16) : 0.0f;
                }
        }
        float cg[2][4];
#pragma unroll
        for (int t = 0; t < 2; t++)
#pragma unroll
            for (int i = 0; i < 4; i++) cg[t][i] = 0.0f;
        const uint16_t* xr = xs + (buf * 2 + par) * 16 * kXRow;
        const uint32_t* wr = wsm + (2 * (pr % kWPairs) + par) * 16 * kWRow;
#pragma unroll
        for (int st = 0; st < 8; st++) {
            // B: token c4, the staged positions 4q .. 4q + 3 of this 16-K step
            const uint2 bx = *reinterpret_cast<const uint2*>(xr + c4 * kXRow + 16 * st + 4 * q);
            const uint32_t* wo = wr + (2 * st + (q >> 1)) * kWRow;
#pragma unroll
            for (int mt = 0; mt < 2; mt++) {
                const uint32_t wa = wo[chl[mt][0]], wb = wo[chl[mt][1]];
                const uint32_t a0 = dq_pair(wa, sh0, zb[mt][0]), a2 = dq_pair(wa, sh0 + 4, zb[mt][0]);
                const uint32_t a1 = dq_pair(wb, sh0, zb[mt][1]), a3 = dq_pair(wb, sh0 + 4, zb[mt][1]);
                mma_16816(cg[mt], a0, a1, a2, a3, bx.x, bx.y);
            }
        }
        // C rows c4, c4 + 8 are channels chl[mt][0], chl[mt][1]; columns 2q, 2q + 1 are tokens
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
            acc[mt][0] += cg[mt][0] * sc[mt][0];
            acc[mt][1] += cg[mt][1] * sc[mt][0];
            acc[mt][2] += cg[mt][2] * sc[mt][1];
            acc[mt][3] += cg[mt][3] * sc[mt][1];
        }
        // stage the next pair's X (the buffer read two pairs ago is free since the barrier above)
        if (pr + 1 < npairs) store_x(buf ^ 1, xv);
        if (pr + 2 < npairs) load_x(pr + 2, xv);
        __syncthreads();                                  // this pair's weight slots are free
        issue_w(pr + kWPairs);
    }
    cp_async_wait<0>();

    // the two group parities into one partial tile red[token][channel], tokens 2q and 2q + 1
    if (par == 0) {
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
            red[(2 * q) * 128 + chl[mt][0]] = acc[mt][0];
            red[(2 * q + 1) * 128 + chl[mt][0]] = acc[mt][1];
            red[(2 * q) * 128 + chl[mt][1]] = acc[mt][2];
            red[(2 * q + 1) * 128 + chl[mt][1]] = acc[mt][3];
        }
    }
    __syncthreads();
    if (par == 1) {
#pragma unroll
        for (int mt = 0; mt < 2; mt++) {
            red[(2 * q) * 128 + chl[mt][0]] += acc[mt][0];
            red[(2 * q + 1) * 128 + chl[mt][0]] += acc[mt][1];
            red[(2 * q) * 128 + chl[mt][1]] += acc[mt][2];
            red[(2 * q + 1) * 128 + chl[mt][1]] += acc[mt][3];
        }
    }
    __syncthreads();
    // split-K over the cluster: CTA `rank` sums columns [rank*128/cs, (rank+1)*128/cs)
    if (cs > 1) cluster_sync_all();
    const int col0 = rank * 128 / cs, col1 = (rank + 1) * 128 / cs, width = col1 - col0;
    const uint32_t red_s = smem_u32(red);
    for (int idx = tid; idx < 8 * width; idx += 256) {
        const int m = idx / width, n = col0 + idx % width;
        float v = 0.0f;
        if (cs > 1) {
            const uint32_t off = red_s + (uint32_t)((m * 128 + n) * 4);
            float part[8];
#pragma unroll
            for (int r = 0; r < 8; r++) part[r] = (r < cs) ? ld_peer_f32(off, (uint32_t)r) : 0.0f;
#pragma unroll
            for (int r = 0; r < 8; r++) v += part[r];
        } else {
            v = red[m * 128 + n];
        }
        if (m0 + m < p.M && n0 + n < p.N) {
            const float b = p.bias ? __bfloat162float(__ushort_as_bfloat16(p.bias[n0 + n])) : 0.0f;
            p.y[(int64_t)(m0 + m) * p.ldy + n0 + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + b));
        }
    }
    if (cs > 1) cluster_sync_all();
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

// Split-K ways (cluster size) so that the grid is about one wave of SMs.  At
// most 4: each CTA holds most of an SM's shared memory, and clusters of up to
// 4 such CTAs are the sizes this kernel has been run and checked with.
int pick_split(int64_t tiles, int64_t groups) {
    int cs = 1;
    while (cs < 4 && tiles * cs * 2 <= kNumSMs && groups >= 2 * cs * 2) cs *= 2;
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
    p.bias = a.bias;
    p.y = a.y;
    p.status = a.dev_status;

    // Several threads may run this setup at once; it is idempotent.
    static std::atomic<bool> attr_set{false};
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(k_w4a16<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set.store(true, std::memory_order_release);
    }
    const int64_t ntiles = (a.N + 127) / 128, mtiles = (a.M + MP - 1) / MP;
    const int cs = pick_split(ntiles * mtiles, p.groups);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)ntiles, (unsigned)mtiles);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_w4a16<MP>, tmQ, tmX, p);
    if (e != cudaSuccess) (void)cudaGetLastError();   // a refused launch leaves no error for the next call
    return e;
}

}  // namespace

size_t w4a16_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

// Split-K ways (cluster size, 1..8, not only powers of two) for the warp-level
// kernel: as many as fit one wave of two CTAs per SM, with at least two
// 128-K groups per CTA.
int pick_split_mma(int64_t tiles, int64_t groups) {
    int cs = 1;
    while (cs < 8 && tiles * (cs + 1) <= 2 * kNumSMs && groups >= 2 * (cs + 1)) cs++;
    return cs;
}

cudaError_t launch_w4a16_mma(const GemmArgs& a, cudaStream_t st) {
    const bool m8 = a.M <= 8;
    W4MmaParams p{};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.groups = (int)(a.K / 128);
    p.ldy = a.ldy;
    p.qweight = static_cast<const int32_t*>(a.w);
    p.x = static_cast<const uint16_t*>(a.x);
    p.scales = static_cast<const uint16_t*>(a.w_scales);
    p.qzeros = static_cast<const int32_t*>(a.w_zeros);
    p.bias = a.bias;
    p.y = a.y;
    const int64_t ntiles = (a.N + 127) / 128, mtiles = (a.M + 15) / 16;
    const int cs = pick_split_mma(ntiles * mtiles, p.groups);
    // Several threads may run this setup at once; it is idempotent.
    static std::atomic<bool> attr_set{false};
    if (!attr_set.load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(k_w4a16_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_w4a16_mma8, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
        if (e != cudaSuccess) return e;
        attr_set.store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)ntiles, (unsigned)mtiles);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = kMmaSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = m8 ? cudaLaunchKernelEx(&cfg, k_w4a16_mma8, p) : cudaLaunchKernelEx(&cfg, k_w4a16_mma, p);
    if (e != cudaSuccess) (void)cudaGetLastError();   // a refused launch leaves no error for the next call
    return e;
}

cudaError_t launch_gemm_w4a16(const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 16) return launch_w4a16_mma(a, st);
    return launch_mp<64>(a, st);     // 64-token tiles, zero-filled past M; larger M runs several
}

}  // namespace qlin
