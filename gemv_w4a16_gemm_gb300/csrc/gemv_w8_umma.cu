// gemv_w8_umma.cu -- int8 weight-only linear layer for 5 <= M <= 64 (and
// for K beyond the CUDA-core kernel's range) on the tcgen05 tensor core.
//
//   out[m,n] = bf16_RN( fp32( sum_k x[m,k] * W[n,k] ) * scales[n] )
//
// ("gpt-fast issue #114": WeightOnlyInt8Linear.forward, F.linear(x,
// W.to(bf16)) * scales, and its open question of batch sizes above one;
// this is a new GB300 design with the same arithmetic.)
//
// The contraction runs in fp16 on the 5th-generation tensor core with fp32
// accumulation, exactly as far as the operands go:
//   * A (weights): every int8 weight b is the fp16 number b exactly.  The
//     dequant warps read the weight's bytes straight from the row-major int8
//     matrix (2-D TMA boxes of 128 rows x 128 bytes, 128-byte swizzle) and
//     build the fp16 pairs with one byte permute per two weights, placing b
//     ^ 0x80 = b + 128 in the mantissa of 1024 (0x6400 | u = 1024 + u), then
//     one fp16x2 subtraction of 1152; (1024 + b + 128) - 1152 = b exactly.
//     They store A to tensor memory with 16-lane x 256-bit stores in natural
//     K order: thread t's register pair of repetition i holds row t/4 (and
//     t/4 + 8), K = 16i + 4(t % 4) .. + 3, the four bytes one 32-bit shared
//     load returns.
//   * B (activations): act_prep_w8 scales each row m of x by a power of two
//     2^sigma_m chosen from the row's max |x| (max |x| 2^sigma in [2^14,
//     2^15)), so every bf16 value at or above 2^-28 of the row's max is an
//     fp16 number exactly, and writes x' = x 2^sigma in fp16 in the
//     128-byte-swizzle K-major layout the MMA's descriptor reads.
//   * D (fp32, tensor memory) accumulates sum_k b x' over the CTA's K range;
//     the epilogue writes bf16_RN((D 2^-sigma_m) * scale_n), or the fp32
//     partial when the pair's K is split between CTAs (a third launch sums
//     the partials in CTA order and applies the same epilogue).
//
// The pipeline is that of gemv_w4_umma.cu (one CTA per SM; a weight
// producer, an activation producer, two MMA issuers (one per 128-row group
// of a 256-row pair), four epilogue warps and eight dequant warps; stream-K
// over (pair, 256-K super-block) units; every wait bounded by one second of
// %globaltimer).  A unit's weights are 64 KB (four boxes), so the weight
// ring holds two or three units; the dequant warps release a unit after
// they have stored it.
//
// Bounds (derived for every launch the plan makes): TMA boxes start at K
// byte offsets 256 b + 128 h < 256 KB and rows 128 g with g < G (the box's
// rows and columns outside the matrix read zeros); shared rings inside
// [SX x (NP x 512)][SW x 65536] of a 1024-aligned base; TMEM columns below
// 512 (D [0, 256), A slot k sub-block h at 256 + 64 (2k + h) + 32 gi + 8 i,
// + 8 <= 512); partials below P * 2 * M * 256; outputs only for n < N,
// m < M.
#include <cstring>

#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace w4q {

namespace {

constexpr int W8_PAIR_ROWS = 256;
constexpr int W8_BOX = 128 * 128;               // one TMA box: 128 rows x 128 K bytes
constexpr int W8_UNIT_BYTES = 4 * W8_BOX;       // [group][K half] boxes of a unit
constexpr int W8_EPI_WARPS = 4;
constexpr int W8_DQ_WARPS = 8;
constexpr int W8_FIRST_EPI = 2;
constexpr int W8_FIRST_DQ = W8_FIRST_EPI + W8_EPI_WARPS;
constexpr int W8_MMA1 = W8_FIRST_DQ + W8_DQ_WARPS;
constexpr int W8_XPROD = W8_MMA1 + 1;
constexpr int W8_THREADS = (W8_XPROD + 1) * 32;
constexpr uint32_t W8_TMEM_COLS = 512;
constexpr uint32_t W8_DCOL = 128;               // columns per accumulator buffer
constexpr uint32_t W8_ACOL = 2 * W8_DCOL;       // first A column (two accumulator buffers)
constexpr int W8_NA = 2;                        // A slots of two 64-K sub-blocks
constexpr int W8_SMEM_LIMIT = 227 * 1024;

struct W8UParams {
    CUtensorMap tmap;          // W int8 [N][K]: boxes of 128 K x 128 rows, 128-byte swizzle
    const uint8_t *xs;         // [KB][4][NP][128 B]: x' fp16, swizzled K-major (act_prep_w8)
    const float *xf;           // [NP]: 2^-sigma_m
    const __nv_bfloat16 *scales;
    __nv_bfloat16 *out;        // bf16 [M][N]
    float *partial;            // fp32 [P][2][M][256]
    unsigned *err;
    int M, N, K, KB, G, G2, P, split;
    long long U;
};

template <int NP>
__host__ __device__ constexpr int w8_xstages()
{
    return NP <= 16 ? 3 : 2;
}

template <int NP>
__host__ __device__ constexpr int w8_wstages()
{
    int s = 3;
    while (s > 2 && s * W8_UNIT_BYTES + w8_xstages<NP>() * NP * 512 + 2048 > W8_SMEM_LIMIT)
        --s;
    return s;
}

template <int NP>
__host__ __device__ constexpr int w8_smem()
{
    return w8_xstages<NP>() * NP * 512 + w8_wstages<NP>() * W8_UNIT_BYTES + 1024;
}

__host__ __device__ __forceinline__ long long w8_range_begin(const W8UParams &p, int c)
{
    if (p.split == 0)
        return (long long)c * p.U / p.P;
    const int g = c / p.split, j = c % p.split;
    return (long long)g * p.KB + (long long)j * p.KB / p.split;
}

__host__ __device__ __forceinline__ int w8_range_owner(const W8UParams &p, long long u)
{
    if (p.split == 0)
        return (int)(((u + 1) * p.P - 1) / p.U);
    const int g = (int)(u / p.KB), b = (int)(u % p.KB);
    return g * p.split + (int)(((long long)(b + 1) * p.split - 1) / p.KB);
}

__device__ __forceinline__ uint32_t w8_lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Four int8 weights (one 32-bit word, K order) -> two fp16 pairs, exactly.
__device__ __forceinline__ void w8_word_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;                       // b + 128 per byte
    lo = f16x2_sub(prmt(u, 0x64646464u, 0x5140u), 0x64806480u);  // bytes 0, 1
    hi = f16x2_sub(prmt(u, 0x64646464u, 0x7362u), 0x64806480u);  // bytes 2, 3
}

template <int NP>
__global__ void __launch_bounds__(W8_THREADS, 1) w8_umma_kernel(const __grid_constant__ W8UParams p)
{
    constexpr int SW = w8_wstages<NP>();
    constexpr int SX = w8_xstages<NP>();
    constexpr uint32_t IDESC = idesc_f16_f32(128, NP);
    constexpr int XB = NP * 512;

    extern __shared__ uint8_t w8_dsmem[];
    __shared__ __align__(8) uint64_t bars[2 * SW + 2 * SX + 2 * W8_NA + 5];
    __shared__ uint32_t tmem_slot;
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(w8_dsmem) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const long long u0 = w8_range_begin(p, c);
    const long long u1 = (c + 1 < p.P) ? w8_range_begin(p, c + 1) : p.U;
    const int n_iter = (int)(u1 - u0);
    const int gp_first = (int)(u0 / p.KB), b_first = (int)(u0 % p.KB);

    constexpr int B0 = 2 * SW + 2 * SX;
    const uint32_t wfull0 = smem_addr(&bars[0]);
    const uint32_t wempty0 = smem_addr(&bars[SW]);
    const uint32_t xfull0 = smem_addr(&bars[2 * SW]);
    const uint32_t xempty0 = smem_addr(&bars[2 * SW + SX]);
    const uint32_t afull0 = smem_addr(&bars[B0]);
    const uint32_t aempty0 = smem_addr(&bars[B0 + W8_NA]);
    const uint32_t dfull0 = smem_addr(&bars[B0 + 2 * W8_NA]);       // [2]
    const uint32_t dempty0 = smem_addr(&bars[B0 + 2 * W8_NA + 2]);  // [2]
    const uint32_t mdone = smem_addr(&bars[B0 + 2 * W8_NA + 4]);
    uint8_t *const xring = smem;              // SX x (NP x 512 B), 1024-aligned
    uint8_t *const wring = smem + SX * XB;    // SW x 65536 B, 1024-aligned

    if (threadIdx.x == 0) {
        for (int s = 0; s < SW; ++s) {
            mbar_init(wfull0 + 8 * s, 1);
            mbar_init(wempty0 + 8 * s, W8_DQ_WARPS);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull0 + 8 * s, 1);
            mbar_init(xempty0 + 8 * s, 2);
        }
        for (int k = 0; k < W8_NA; ++k) {
            mbar_init(afull0 + 8 * k, W8_DQ_WARPS);
            mbar_init(aempty0 + 8 * k, 2);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(dfull0 + 8 * d, 2);
            mbar_init(dempty0 + 8 * d, W8_EPI_WARPS);
        }
        mbar_init(mdone, 2);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&tmem_slot), W8_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------- producer of the weights
        if (lane == 0 && n_iter > 0) {
            const uint64_t pol_w = policy_evict_first();
            int gp = gp_first, b = b_first, issued = 0;
            for (int i = 0; i < n_iter; ++i) {
                const int slot = i % SW;
                if (i >= SW && !mbar_wait_sleep(wempty0 + 8 * slot, (uint32_t)((i / SW) - 1) & 1u)) {
                    report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                const uint32_t bar = wfull0 + 8 * slot;
                const int ng = (2 * gp + 1 < p.G) ? 2 : 1;
                mbar_arrive_expect_tx(bar, (uint32_t)(ng * 2 * W8_BOX));
                const uint32_t dst = smem_addr(wring + slot * W8_UNIT_BYTES);
                for (int gi = 0; gi < ng; ++gi)
                    for (int h = 0; h < 2; ++h)
                        tma_load_2d(dst + (uint32_t)((2 * gi + h) * W8_BOX), &p.tmap, 256 * b + 128 * h,
                                    128 * (2 * gp + gi), bar, pol_w);
                issued = i + 1;
                if (++b == p.KB) {
                    b = 0;
                    ++gp;
                }
            }
            for (int i = (issued > SW ? issued - SW : 0); i < issued; ++i)
                if (!mbar_wait_sleep(wfull0 + 8 * (i % SW), (uint32_t)(i / SW) & 1u)) {
                    report_error(p.err, ERR_DRAIN_WAIT);
                    break;
                }
        }
    } else if (warp == W8_XPROD) {
        // ------------------------------------------- producer of the x stages
        if (lane == 0 && n_iter > 0) {
            const uint64_t pol_x = policy_evict_last();
            pdl_wait();  // x' comes from act_prep_w8, launched just before
            int b = b_first, issued = 0;
            for (int i = 0; i < n_iter; ++i) {
                const int slot = i % SX;
                if (i >= SX && !mbar_wait_sleep(xempty0 + 8 * slot, (uint32_t)((i / SX) - 1) & 1u)) {
                    report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                const uint32_t bar = xfull0 + 8 * slot;
                mbar_arrive_expect_tx(bar, (uint32_t)XB);
                bulk_g2s(smem_addr(xring + slot * XB), p.xs + (size_t)b * XB, XB, bar, pol_x);
                issued = i + 1;
                if (++b == p.KB)
                    b = 0;
            }
            for (int i = (issued > SX ? issued - SX : 0); i < issued; ++i)
                if (!mbar_wait_sleep(xfull0 + 8 * (i % SX), (uint32_t)(i / SX) & 1u)) {
                    report_error(p.err, ERR_DRAIN_WAIT);
                    break;
                }
        }
    } else if (warp == 1 || warp == W8_MMA1) {
        // ------------------------------------------------------ MMA issuers
        const int gi = warp == 1 ? 0 : 1;
        if (lane == 0 && n_iter > 0) {
            int a_it = 0, d_it = 0, gp = gp_first, b = b_first;
            bool first = true, ok = true;
            for (int i = 0; i < n_iter && ok; ++i) {
                const int slot = i % SX;
                if (!mbar_wait_sleep(xfull0 + 8 * slot, (uint32_t)(i / SX) & 1u) ||
                    (first && !mbar_wait_sleep(dempty0 + 8 * (d_it & 1), (uint32_t)((d_it >> 1) & 1) ^ 1u))) {
                    report_error(p.err, ERR_FULL_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const bool live = gi == 0 || 2 * gp + 1 < p.G;
                const uint32_t d_tmem = tmem + W8_DCOL * (uint32_t)(d_it & 1) + (uint32_t)(gi * NP);
                const uint64_t bdesc = sdesc_sw128_kmajor(smem_addr(xring + slot * XB));
                for (int s0 = 0; s0 < 4; s0 += 2) {  // one A slot: two 64-K sub-blocks
                    const int k = a_it % W8_NA;
                    if (!mbar_wait_sleep(afull0 + 8 * k, (uint32_t)(a_it / W8_NA) & 1u)) {
                        report_error(p.err, ERR_FULL_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (live) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int sbk = s0 + h;
                            const uint32_t a_tmem = tmem + W8_ACOL + (uint32_t)(64 * (2 * k + h) + 32 * gi);
                            const uint64_t bd = bdesc + (uint64_t)((sbk * NP * 128) >> 4);
                            umma_ts(d_tmem, a_tmem, bd, IDESC, (first && sbk == 0) ? 0u : 1u);
                            umma_ts(d_tmem, a_tmem + 8, bd + 2, IDESC, 1u);
                            umma_ts(d_tmem, a_tmem + 16, bd + 4, IDESC, 1u);
                            umma_ts(d_tmem, a_tmem + 24, bd + 6, IDESC, 1u);
                        }
                    }
                    umma_commit(aempty0 + 8 * k);
                    ++a_it;
                }
                if (!ok)
                    break;
                umma_commit(xempty0 + 8 * slot);
                first = false;
                if (++b == p.KB || i == n_iter - 1) {
                    umma_commit(dfull0 + 8 * (d_it & 1));
                    ++d_it;
                    first = true;
                    b = 0;
                    ++gp;
                }
            }
            umma_commit(mdone);
            if (!mbar_wait_sleep(mdone, 0u))
                report_error(p.err, ERR_DRAIN_WAIT);
        }
    } else if (warp < W8_FIRST_DQ) {
        // --------------------------------------------------------- epilogue
        pdl_wait();  // xf (act_prep_w8) and the outputs / partials of earlier kernels
        const int q = warp & 3;
        const int L = 32 * q + lane;  // TMEM lane = row within the tile group
        const size_t seg = (size_t)p.M * W8_PAIR_ROWS;
        const int gp_last = n_iter > 0 ? (int)((u1 - 1) / p.KB) : gp_first - 1;
        for (int gp = gp_first, d = 0; gp <= gp_last; ++gp, ++d) {
            if (!mbar_wait_sleep(dfull0 + 8 * (d & 1), (uint32_t)(d >> 1) & 1u)) {
                report_error(p.err, ERR_FULL_WAIT);
                break;
            }
            tc_fence_after_sync();
            const int ng = (2 * gp + 1 < p.G) ? 2 : 1;
            const long long gb = (long long)gp * p.KB, ge = gb + p.KB;
            const bool whole = gb >= u0 && ge <= u1;
            const int slot = (gp == gp_first) ? 0 : 1;
            for (int gi = 0; gi < ng; ++gi) {
                const int n = (2 * gp + gi) * 128 + L;
                const float sn = (whole && n < p.N) ? __bfloat162float(p.scales[n]) : 0.f;
                float *dst = p.partial + (size_t)(c * 2 + slot) * seg + (size_t)gi * 128 + L;
                constexpr int CC = NP < 32 ? NP : 32;
#pragma unroll
                for (int c0 = 0; c0 < NP; c0 += CC) {
                    uint32_t r[CC / 8][8];
#pragma unroll
                    for (int ch = 0; ch < CC / 8; ++ch)
                        tmem_ld_32x32b_x8(tmem + ((uint32_t)(32 * q) << 16) + W8_DCOL * (uint32_t)(d & 1) +
                                              (uint32_t)(gi * NP + c0 + 8 * ch),
                                          r[ch]);
                    tmem_wait_ld();
                    if (c0 >= p.M)
                        continue;
                    if (whole) {
                        if (n < p.N) {
#pragma unroll
                            for (int m = 0; m < CC; ++m)
                                if (c0 + m < p.M)
                                    p.out[(size_t)(c0 + m) * p.N + n] = __float2bfloat16_rn(
                                        (__uint_as_float(r[m / 8][m % 8]) * p.xf[c0 + m]) * sn);
                        }
                    } else {
#pragma unroll
                        for (int m = 0; m < CC; ++m)
                            if (c0 + m < p.M)
                                dst[(size_t)(c0 + m) * W8_PAIR_ROWS] = __uint_as_float(r[m / 8][m % 8]);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(dempty0 + 8 * (d & 1));
        }
    } else {
        // ---------------------------------------------------------- dequant
        // A warp may access only its quarter (warp id % 4) of the TMEM
        // lanes: warp w converts row tile 2 (w % 4) + half of both groups.
        const int dw = warp - W8_FIRST_DQ;
        const int tl = 2 * (warp & 3) + ((dw >> 2) & 1);
        const int r = lane >> 2, tq = lane & 3;
        const uint32_t tlane = (uint32_t)(16 * tl) << 16;  // its 16 TMEM lanes
        const int R = 16 * tl + r;                         // row within the group (and R + 8)
        int a_it = 0, gp = gp_first, b = b_first, pend = -1;
        bool ok = true;
        for (int i = 0; i < n_iter && ok; ++i) {
            const int slot = i % SW;
            if (!mbar_wait_sleep(wfull0 + 8 * slot, (uint32_t)(i / SW) & 1u)) {
                report_error(p.err, ERR_FULL_WAIT);
                break;
            }
            const int ng = (2 * gp + 1 < p.G) ? 2 : 1;
            const uint32_t ubase = smem_addr(wring + slot * W8_UNIT_BYTES);
#pragma unroll
            for (int sbk = 0; sbk < 4; ++sbk) {
                const int hk = sbk >> 1, cb = 4 * (sbk & 1);  // K half, its first 16-byte chunk
                uint32_t v[2][16];
#pragma unroll
                for (int gg = 0; gg < 2; ++gg)
                    if (gg < ng) {
                        const uint32_t box = ubase + (uint32_t)((2 * gg + hk) * W8_BOX);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            // row R: 16-byte chunk cb + j at (cb + j) ^ (R % 8), word tq
                            const uint32_t off = (uint32_t)((((cb + j) ^ (R & 7)) << 4) + 4 * tq);
                            const uint32_t w0 = w8_lds32(box + (uint32_t)R * 128u + off);
                            const uint32_t w1 = w8_lds32(box + (uint32_t)(R + 8) * 128u + off);
                            w8_word_to_f16(w0, v[gg][4 * j], v[gg][4 * j + 1]);
                            w8_word_to_f16(w1, v[gg][4 * j + 2], v[gg][4 * j + 3]);
                        }
                    }
                const int k = a_it % W8_NA;
                if ((sbk & 1) == 0) {  // the first sub-block of a slot
                    if (pend >= 0) {   // the previous slot's stores: complete, then publish
                        tmem_wait_st();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(afull0 + 8 * pend);
                        pend = -1;
                    }
                    if (!mbar_wait_sleep(aempty0 + 8 * k, ((uint32_t)(a_it / W8_NA) & 1u) ^ 1u)) {
                        report_error(p.err, ERR_EMPTY_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
#pragma unroll
                for (int gg = 0; gg < 2; ++gg)
                    if (gg < ng)
                        tmem_st_16x256b_x4(tmem + tlane + W8_ACOL +
                                               (uint32_t)(64 * (2 * k + (sbk & 1)) + 32 * gg),
                                           v[gg]);
                if (sbk & 1) {
                    pend = k;
                    ++a_it;
                }
            }
            __syncwarp();  // every lane's shared loads of the unit are done
            if (lane == 0)
                mbar_arrive(wempty0 + 8 * slot);
            if (++b == p.KB) {
                b = 0;
                ++gp;
            }
        }
        if (pend >= 0) {
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(afull0 + 8 * pend);
        }
    }

    pdl_launch_dependents();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, W8_TMEM_COLS);
    }
}

// x -> x' = fp16(x 2^sigma_m) in the B layout: block (row m < NP, 2048-column
// chunk), eight columns (one 16-byte chunk of a 128-byte line) per thread.
// sigma_m from max |x[m]| (every block of the row finds it): max |x| 2^sigma
// in [2^14, 2^15), 0 for an all-zero row; xf[m] = 2^-sigma_m.  Rows m >= M
// and columns k >= K are written as zeros.
__global__ void __launch_bounds__(256) act_prep_w8_kernel(const __nv_bfloat16 *__restrict__ x, int M,
                                                          int K, int KB, int NP,
                                                          uint8_t *__restrict__ xs,
                                                          float *__restrict__ xf)
{
    pdl_launch_dependents();  // the main kernel may start streaming weights
    pdl_wait();               // x (and this workspace) may belong to the previous kernel
    __shared__ uint32_t wmax[8];
    const int m = blockIdx.x;
    const int k0 = blockIdx.y * 2048 + threadIdx.x * 8;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
    const bool live = m < M && k0 < K;
    const uint4 raw = live ? row[k0 / 8] : make_uint4(0u, 0u, 0u, 0u);
    uint32_t h = 0u;
    if (m < M) {
#pragma unroll 4
        for (int j = threadIdx.x; j < K / 8; j += 256) {
            const uint4 v = row[j];
            h = __vmaxu2(h, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                     __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
        }
    }
    h = max(h & 0xFFFFu, h >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = h;
    __syncthreads();
    uint32_t a = 0u;
    for (int w = 0; w < 8; ++w)
        a = max(a, wmax[w]);
    // e with max |x| in [2^e, 2^(e+1)), from the bf16 bits
    int sigma = 0;
    if (a != 0u) {
        const int e = a >= 0x80u ? (int)(a >> 7) - 127 : (31 - __clz((int)a)) - 133;
        sigma = 14 - e;
    }
    if (blockIdx.y == 0 && threadIdx.x == 0)
        xf[m] = m < M ? ldexpf(1.0f, -sigma) : 0.f;
    if (k0 >= KB * 256)
        return;
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half lo = __float2half_rn(ldexpf(bf16lo_to_f32(w[j]), sigma));
        const __half hi = __float2half_rn(ldexpf(bf16hi_to_f32(w[j]), sigma));
        o[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
    }
    // element k0: super-block k0 / 256, sub-block (k0 % 256) / 64, chunk (k0 % 64) / 8
    const int bs = k0 / 64, ch = (k0 % 64) / 8;
    uint8_t *line = xs + ((size_t)bs * NP + m) * 128;
    *reinterpret_cast<uint4 *>(line + ((ch ^ (m & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Sum of the fp32 partials of the pairs that several CTAs share, in CTA
// order, then the epilogue of the main kernel.  Block (pair, ROWS rows of
// x); CHUNK contributors' loads go out together.
template <int ROWS, int CHUNK>
__global__ void __launch_bounds__(W8_PAIR_ROWS) w8_umma_fixup_kernel(const __grid_constant__ W8UParams p)
{
    constexpr int W8_FIX_ROWS = ROWS;
    // The next call's preparation may launch and wait beside these blocks
    // (measured on 6656 x 19968 at M = 16: 31.1 -> 29.4 us per call).
    pdl_launch_dependents();
    pdl_wait();
    const int gp = blockIdx.x, m0 = blockIdx.y * W8_FIX_ROWS, row = threadIdx.x;
    const long long gb = (long long)gp * p.KB, ge = gb + p.KB;
    const int cf = w8_range_owner(p, gb), cl = w8_range_owner(p, ge - 1);
    const int n = gp * W8_PAIR_ROWS + row;
    if (cf == cl || n >= p.N)
        return;  // a whole pair: written by the main kernel
    const size_t seg = (size_t)p.M * W8_PAIR_ROWS;
    const int slot0 = (w8_range_begin(p, cf) == gb) ? 0 : 1;
    const float *first = p.partial + (size_t)(cf * 2 + slot0) * seg + (size_t)m0 * W8_PAIR_ROWS + row;
    const float *rest = p.partial + (size_t)(cf * 2 + 2) * seg + (size_t)m0 * W8_PAIR_ROWS + row;
    const int nc = cl - cf;
    float v[W8_FIX_ROWS];
#pragma unroll
    for (int r = 0; r < W8_FIX_ROWS; ++r)
        v[r] = (m0 + r < p.M) ? __ldcg(first + (size_t)r * W8_PAIR_ROWS) : 0.f;
    for (int j = 0; j < nc; j += CHUNK) {
        float t[W8_FIX_ROWS][CHUNK];
#pragma unroll
        for (int r = 0; r < W8_FIX_ROWS; ++r)
#pragma unroll
            for (int u = 0; u < CHUNK; ++u)
                t[r][u] = (m0 + r < p.M && j + u < nc)
                              ? __ldcg(rest + (size_t)(j + u) * 2 * seg + (size_t)r * W8_PAIR_ROWS)
                              : 0.f;
#pragma unroll
        for (int r = 0; r < W8_FIX_ROWS; ++r)
#pragma unroll
            for (int u = 0; u < CHUNK; ++u)
                if (j + u < nc)
                    v[r] += t[r][u];
    }
    const float sn = __bfloat162float(p.scales[n]);
#pragma unroll
    for (int r = 0; r < W8_FIX_ROWS; ++r)
        if (m0 + r < p.M)
            p.out[(size_t)(m0 + r) * p.N + n] = __float2bfloat16_rn((v[r] * p.xf[m0 + r]) * sn);
}

// ------------------------------------------------------------------ host

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled()
{
    static const EncodeTiled fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                                &q) == cudaSuccess && q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<EncodeTiled>(f)
                   : nullptr;
    }();
    return fn;
}

size_t w8_align(size_t v) { return (v + 255) / 256 * 256; }

struct W8Plan {
    int M, N, K, KB, G, G2, NP, P, split;
    bool fixup;
};

W8Plan w8_plan(int M, int N, int K, int sm_count)
{
    W8Plan pl;
    pl.M = M;
    pl.N = N;
    pl.K = K;
    pl.KB = (K + 255) / 256;
    pl.G = (N + 127) / 128;
    pl.G2 = (pl.G + 1) / 2;
    pl.NP = (M + 15) / 16 * 16;
    const long long U = (long long)pl.G2 * pl.KB;
    const int sms = sm_count > 0 ? sm_count : 1;
    if (pl.KB <= 4 && pl.G2 <= sms) {  // a pair's whole K per CTA: no partial-sum launch
        pl.split = 1;
        pl.P = pl.G2;
        pl.fixup = false;
    } else {
        pl.split = 0;
        pl.P = (int)(U < sms ? U : sms);
        pl.fixup = !(U % pl.P == 0 && (U / pl.P) % pl.KB == 0);
    }
    return pl;
}

// Workspace: [x' (K/256) * NP * 512][xf NP fp32][partials P * 2 * M * 256 fp32].
struct W8Layout {
    size_t xs, xf, partial, total;
};

W8Layout w8_layout(const W8Plan &pl)
{
    W8Layout L;
    size_t o = 0;
    L.xs = o;
    o += w8_align((size_t)pl.KB * pl.NP * 512);
    L.xf = o;
    o += w8_align((size_t)pl.NP * 4);
    L.partial = o;
    o += pl.fixup ? (size_t)pl.P * 2 * pl.M * W8_PAIR_ROWS * sizeof(float) : 0;
    L.total = o;
    return L;
}

cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int NP>
cudaError_t launch_w8_umma_np(const W8UParams &p, cudaStream_t stream)
{
    auto fn = w8_umma_kernel<NP>;
    static std::atomic<unsigned long long> opted_in{0};
    cudaError_t e = smem_opt_in_once(opted_in, fn, w8_smem<NP>());
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)p.P), dim3(W8_THREADS), w8_smem<NP>(), stream, attr);
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace

size_t w8_tc_workspace(int M, int N, int K, int sm_count)
{
    return w8_layout(w8_plan(M, N, K, sm_count)).total;
}

int w8_tc_launches(int M, int N, int K, int sm_count)
{
    return w8_plan(M, N, K, sm_count).fixup ? 3 : 2;
}

cudaError_t launch_w8_tc(const void *x, const int8_t *W, const void *scales, void *out, int M, int N,
                         int K, int sm_count, void *workspace, unsigned *err, cudaStream_t stream)
{
    const W8Plan pl = w8_plan(M, N, K, sm_count);
    const W8Layout L = w8_layout(pl);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    W8UParams p;
    memset(&p, 0, sizeof p);
    const EncodeTiled enc = encode_tiled();
    if (enc == nullptr)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&p.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.xs = ws + L.xs;
    p.xf = reinterpret_cast<const float *>(ws + L.xf);
    p.scales = static_cast<const __nv_bfloat16 *>(scales);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.partial = reinterpret_cast<float *>(ws + L.partial);
    p.err = err;
    p.M = M;
    p.N = N;
    p.K = K;
    p.KB = pl.KB;
    p.G = pl.G;
    p.G2 = pl.G2;
    p.P = pl.P;
    p.split = pl.split;
    p.U = (long long)pl.G2 * pl.KB;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3((unsigned)pl.NP, (unsigned)((pl.KB * 256 + 2047) / 2048)),
                                        dim3(256), 0, stream, attr);
    cudaError_t e = cudaLaunchKernelEx(&cfg, act_prep_w8_kernel, static_cast<const __nv_bfloat16 *>(x), M,
                                       K, pl.KB, pl.NP, ws + L.xs, reinterpret_cast<float *>(ws + L.xf));
    if (e != cudaSuccess)
        return e;
    switch (pl.NP) {
    case 16: e = launch_w8_umma_np<16>(p, stream); break;
    case 32: e = launch_w8_umma_np<32>(p, stream); break;
    case 48: e = launch_w8_umma_np<48>(p, stream); break;
    default: e = launch_w8_umma_np<64>(p, stream); break;
    }
    if (e != cudaSuccess || !pl.fixup)
        return e;
    const FixShape fs = fix_shape(pl.G2, M, pl.KB, p.U, pl.P, pl.split, sm_count);
    auto fn = fs.rows == 4 ? (fs.chunk == 4 ? w8_umma_fixup_kernel<4, 4> : w8_umma_fixup_kernel<4, 8>)
                           : (fs.chunk == 4 ? w8_umma_fixup_kernel<8, 4> : w8_umma_fixup_kernel<8, 8>);
    cudaLaunchConfig_t fcfg = pdl_config(dim3((unsigned)pl.G2, (unsigned)((M + fs.rows - 1) / fs.rows)),
                                         dim3(W8_PAIR_ROWS), 0, stream, attr);
    return cudaLaunchKernelEx(&fcfg, fn, p);
}

}  // namespace w4q
