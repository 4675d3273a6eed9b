// gemv_w4_umma.cu -- W4A16 linear layer for 9 <= M <= 64 on the tcgen05
// tensor core (sm_103a).
//
//   out[M,N] = x[M,K] . dequant(Wq)[N,K]^T,   dequant(q) = (q - z) * s
//
// ("test_int4_quantized_gemm.py": the dequant + F.linear reference and the
// W4A16 tile kernels, which dequantize a weight tile to bf16 and run it
// through the tensor core; this is a new design for GB300, not their code.)
//
// At these M the call is a real contraction (2 * M * N * K flops on N*K/2
// bytes of codes), so the weight is dequantized once and multiplied on the
// 5th-generation tensor core, with the operands where that core wants them:
//
//   * A (weights, 128 rows of a tile group x 16 K per instruction) lives in
//     tensor memory: dequant warps write (q - z) * s, rounded once to bf16,
//     straight from registers with 16-lane x 256-bit TMEM stores.  The packed
//     layout's per-lane words (built for the m16n8k16 fragment) map onto that
//     store shape one to one, so no shuffles or shared-memory round trip.
//   * B (activations, M rows padded to NP = 16..64, K-major) lives in shared
//     memory in the 128-byte-swizzle layout the MMA reads through a matrix
//     descriptor.  act_prep writes x in exactly that byte order (rows >= M
//     zero), with the K order inside every 16-column step permuted to match
//     the column order of the TMEM stores, so one bulk copy per stage lands it.
//   * D (fp32, 128 lanes x NP columns per tile group) accumulates in tensor
//     memory over the CTA's whole K range and is read once by the epilogue.
//
// One CTA per SM, 16 warps: two producers (bulk copies of the codes, and of
// the activation stages), two MMA issuers (one thread per tile group of the
// pair; warp 1 also owns the TMEM allocation), four epilogue warps (one per
// TMEM lane quarter) and eight dequant warps.  A work unit is a pair of tile
// groups (256 rows) x one 256-K super-block: both groups share one copy of
// the activation stage.  Units are split into P contiguous ranges (stream-K,
// or a fixed split of each pair's K); a pair that one CTA covers entirely is
// written directly, the others through fp32 partials that a third launch
// (umma_fixup_kernel, started by programmatic dependent launch as the main
// kernel's CTAs finish) sums in CTA order: a last-arriver sum inside the main
// kernel would leave M x (contributors) dependent L2 round trips per thread
// at the tail of the kernel.
//
// Bounds (derived for every launch the plan can make): packed sources stay
// below ceil(N/128) * 8 * KB * 2432 bytes (group 2gp + 1 of a pair is
// copied only when 2gp + 1 < G); activation sources below KB * NP * 512;
// shared-memory rings inside [SX x (NP x 512)][SW x 38912] of a 1024-aligned base; TMEM
// columns below 512 (accumulators [0, 256), A slot k sub-block h at
// 256 + 64 (SPS k + h) + 32g + 8j, + 8 <= 512); partial indices below P * 2 * M * 256; outputs only for
// n < N and m < M.
//
// Pipelines (every wait sleeps in mbarrier.try_wait and gives up after one
// second of %globaltimer):
//   codes producer --wfull[s]--> dequant     (packed codes of both groups, unit i)
//   dequant        --wempty[s]-> producer    (codes read into registers)
//   x producer     --xfull[t]--> MMA         (the activation stage of unit i)
//   MMA            --xempty[t]-> x producer  (tcgen05.commit: x no longer read)
//   dequant  --afull[k]-> MMA                (A slot k written to TMEM)
//   MMA      --aempty[k]-> dequant           (tcgen05.commit: slot k consumed)
//   MMA      --dfull[d]-> epilogue           (the pair's accumulators final)
//   epilogue --dempty[d]> MMA                (accumulators read out)
// The accumulators are double-buffered (d = pair parity), so the MMAs of
// the next pair do not wait for the epilogue of the last one.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"
#include "timeline.cuh"

namespace w4q {

namespace {

constexpr int UT_TILE_BYTES = 2432;               // 16 rows x 256 K: codes, scales, zeros
constexpr int UT_GROUP_BYTES = 8 * UT_TILE_BYTES; // one tile group at one super-block
constexpr int UT_PAIR_ROWS = 256;
constexpr int UT_EPI_WARPS = 4;
#ifndef W4Q_UMMA_DQ_WARPS
#define W4Q_UMMA_DQ_WARPS 8
#endif
constexpr int UT_DQ_WARPS = W4Q_UMMA_DQ_WARPS;   // 8: two groups per warp, 16: one
constexpr int UT_GPW = 16 / UT_DQ_WARPS;         // tile groups per dequant warp
constexpr int UT_FIRST_EPI = 2;
constexpr int UT_FIRST_DQ = UT_FIRST_EPI + UT_EPI_WARPS;
constexpr int UT_MMA1 = UT_FIRST_DQ + UT_DQ_WARPS;             // MMA issuer of group 1
constexpr int UT_XPROD = UT_MMA1 + 1;                           // producer of the x ring
constexpr int UT_THREADS = (UT_XPROD + 1) * 32;
#ifndef W4Q_UMMA_NDB
#define W4Q_UMMA_NDB 2
#endif
constexpr int UT_NDB = W4Q_UMMA_NDB;  // accumulator buffers (pairs in flight)
constexpr uint32_t UT_TMEM_COLS = 512;
constexpr uint32_t UT_DCOL = 128;    // columns per accumulator buffer (2 groups x NP <= 128)
constexpr uint32_t UT_ACOL = UT_DCOL * UT_NDB;              // first A column
#ifndef W4Q_UMMA_SPS
#define W4Q_UMMA_SPS 2
#endif
// An A slot holds SPS 64-K sub-blocks of both groups: the dequant warps
// synchronise with the MMA issuers once per slot.
constexpr int UT_SPS = W4Q_UMMA_SPS;
constexpr int UT_NA = (int)((UT_TMEM_COLS - UT_ACOL) / (64 * UT_SPS));  // A slots
constexpr int UT_SMEM_LIMIT = 227 * 1024;

struct UParams {
    const uint8_t *packed;
    const uint8_t *xs;       // [K/256][4][NP][128 B]: swizzled, K-permuted x (act_prep)
    __nv_bfloat16 *out;      // bf16 [M][N]
    float *partial;          // fp32 [P][2][M][256]
    unsigned *err;
    int M, N, K, KB, G, G2, P, split;
    long long U;
};

// Two rings: the codes of a unit (both groups, 38912 B) are released as soon
// as the dequant warps hold them in registers, so that ring can run several
// units ahead and keep HBM busy; the activation stage (NP x 512 B, from L2)
// is released by the MMAs' commit.
constexpr int UT_CODE_BYTES = 2 * UT_GROUP_BYTES;

template <int NP>
__host__ __device__ constexpr int ut_xstages()
{
    return NP <= 16 ? 3 : 2;
}

template <int NP>
__host__ __device__ constexpr int ut_wstages()
{
    int s = 6;
    while (s > 2 && s * UT_CODE_BYTES + ut_xstages<NP>() * NP * 512 + 2048 > UT_SMEM_LIMIT)
        --s;
    return s;
}

template <int NP>
__host__ __device__ constexpr int ut_smem()
{
    // [x ring][codes ring] + alignment slack
    return ut_xstages<NP>() * NP * 512 + ut_wstages<NP>() * UT_CODE_BYTES + 1024;
}

__host__ __device__ __forceinline__ long long ut_range_begin(const UParams &p, int c)
{
    if (p.split == 0)
        return (long long)c * p.U / p.P;
    const int g = c / p.split, j = c % p.split;
    return (long long)g * p.KB + (long long)j * p.KB / p.split;
}

// The CTA whose range holds unit u (the largest c with begin(c) <= u).
__host__ __device__ __forceinline__ int ut_range_owner(const UParams &p, long long u)
{
    if (p.split == 0)
        return (int)(((u + 1) * p.P - 1) / p.U);
    const int g = (int)(u / p.KB), b = (int)(u % p.KB);
    return g * p.split + (int)(((long long)(b + 1) * p.split - 1) / p.KB);
}

// Eight codes of one word -> four bf16x2 A values (q - z) * s of the 16x256b
// store order: (row r, K pair i), (row r, pair i + 4), (row r + 8, pair i),
// (row r + 8, pair i + 4), where the word holds rows r, r + 8 and columns
// 2i, 2i + 1, 2i + 8, 2i + 9 of a 16-column step (nibble of row r + 8a,
// column 2i + 8e + h at bit 8a + 4e + 16h).
__device__ __forceinline__ void ut_dequant_word(uint32_t w, uint32_t zr, uint32_t zr8,
                                                uint32_t s2r, uint32_t s2r8, uint32_t *v)
{
    v[0] = bf16x2_mul(bf16x2_sub(and_or(w, 0x000F000Fu, 0x43004300u), zr), s2r);
    v[1] = bf16x2_mul(bf16x2_sub(and_or(w >> 4, 0x000F000Fu, 0x43004300u), zr), s2r);
    v[2] = bf16x2_mul(bf16x2_sub(and_or(w >> 8, 0x000F000Fu, 0x43004300u), zr8), s2r8);
    v[3] = bf16x2_mul(bf16x2_sub(and_or(w >> 12, 0x000F000Fu, 0x43004300u), zr8), s2r8);
}

template <int NP>
__global__ void __launch_bounds__(UT_THREADS, 1) w4_umma_kernel(const UParams p)
{
    constexpr int SW = ut_wstages<NP>();  // codes ring
    constexpr int SX = ut_xstages<NP>();  // activation ring
    constexpr uint32_t IDESC = idesc_bf16_f32(128, NP);
    constexpr int XB = NP * 512;  // activation bytes of one stage

    extern __shared__ uint8_t ut_dsmem[];
    __shared__ __align__(8) uint64_t bars[2 * SW + 2 * SX + 2 * UT_NA + 5];
    __shared__ uint32_t tmem_slot;
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(ut_dsmem) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const long long u0 = ut_range_begin(p, c);
    const long long u1 = (c + 1 < p.P) ? ut_range_begin(p, c + 1) : p.U;
    const int n_iter = (int)(u1 - u0);
    const int gp_first = (int)(u0 / p.KB), b_first = (int)(u0 % p.KB);

    constexpr int B0 = 2 * SW + 2 * SX;
    const uint32_t wfull0 = smem_addr(&bars[0]);
    const uint32_t wempty0 = smem_addr(&bars[SW]);
    const uint32_t xfull0 = smem_addr(&bars[2 * SW]);
    const uint32_t xempty0 = smem_addr(&bars[2 * SW + SX]);
    const uint32_t afull0 = smem_addr(&bars[B0]);
    const uint32_t aempty0 = smem_addr(&bars[B0 + UT_NA]);
    const uint32_t dfull0 = smem_addr(&bars[B0 + 2 * UT_NA]);       // [2]
    const uint32_t dempty0 = smem_addr(&bars[B0 + 2 * UT_NA + 2]);  // [2]
    const uint32_t mdone = smem_addr(&bars[B0 + 2 * UT_NA + 4]);
    uint8_t *const xring = smem;                // SX x (NP x 512 B), 1024-aligned
    uint8_t *const wring = smem + SX * XB;      // SW x 38912 B

    if (threadIdx.x == 0) {
        for (int s = 0; s < SW; ++s) {
            mbar_init(wfull0 + 8 * s, 1);
            mbar_init(wempty0 + 8 * s, UT_DQ_WARPS);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull0 + 8 * s, 1);
            mbar_init(xempty0 + 8 * s, 2);
        }
        for (int k = 0; k < UT_NA; ++k) {
            mbar_init(afull0 + 8 * k, UT_DQ_WARPS);
            mbar_init(aempty0 + 8 * k, 2);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(dfull0 + 8 * d, 2);
            mbar_init(dempty0 + 8 * d, UT_EPI_WARPS);
        }
        mbar_init(mdone, 2);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&tmem_slot), UT_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_slot;
    if (threadIdx.x == 0)
        W4Q_STAMP(40);

    if (warp == 0) {
        // ----------------------------------------------- producer of the codes
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
                const uint32_t dst = smem_addr(wring + slot * UT_CODE_BYTES);
                const bool g1 = 2 * gp + 1 < p.G;
                mbar_arrive_expect_tx(bar, (uint32_t)((g1 ? 2 : 1) * UT_GROUP_BYTES));
                bulk_g2s(dst, p.packed + ((size_t)(2 * gp) * p.KB + b) * UT_GROUP_BYTES,
                         UT_GROUP_BYTES, bar, pol_w);
                if (g1)
                    bulk_g2s(dst + UT_GROUP_BYTES,
                             p.packed + ((size_t)(2 * gp + 1) * p.KB + b) * UT_GROUP_BYTES,
                             UT_GROUP_BYTES, bar, pol_w);
                issued = i + 1;
                if (++b == p.KB) {
                    b = 0;
                    ++gp;
                }
            }
            // drain: every issued copy has landed before the CTA exits
            for (int i = (issued > SW ? issued - SW : 0); i < issued; ++i)
                if (!mbar_wait_sleep(wfull0 + 8 * (i % SW), (uint32_t)(i / SW) & 1u)) {
                    report_error(p.err, ERR_DRAIN_WAIT);
                    break;
                }
        }
    } else if (warp == UT_XPROD) {
        // ------------------------------------------- producer of the x stages
        if (lane == 0 && n_iter > 0) {
            const uint64_t pol_x = policy_evict_last();
            pdl_wait();  // x comes from act_prep, launched just before
            W4Q_STAMP(41);
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
    } else if (warp == 1 || warp == UT_MMA1) {
        // ------------------------------------------------------ MMA issuers
        // One thread per tile group of the pair: a single issuing thread
        // tops out near 47 cycles per N = 64 instruction, two keep the
        // tensor core at its 32.  Group 1's thread commits (with nothing to
        // wait for) even when the pair has no group 1, so every barrier
        // still receives both arrivals.
        const int gi = warp == 1 ? 0 : 1;
        if (lane == 0 && n_iter > 0) {
            int a_it = 0, d_it = 0, gp = gp_first, b = b_first;
            bool first = true, ok = true;
            for (int i = 0; i < n_iter && ok; ++i) {
                const int slot = i % SX;
                if (!mbar_wait_sleep(xfull0 + 8 * slot, (uint32_t)(i / SX) & 1u) ||
                    (first && !mbar_wait_sleep(dempty0 + 8 * (d_it % UT_NDB),
                                                 (uint32_t)((d_it / UT_NDB) & 1) ^ 1u))) {
                    report_error(p.err, ERR_FULL_WAIT);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const bool live = gi == 0 || 2 * gp + 1 < p.G;
                const uint32_t d_tmem = tmem + UT_DCOL * (uint32_t)(d_it % UT_NDB) + (uint32_t)(gi * NP);
                const uint64_t bdesc = sdesc_sw128_kmajor(smem_addr(xring + slot * XB));
                for (int s0 = 0; s0 < 4; s0 += UT_SPS) {  // one A slot: UT_SPS sub-blocks
                    const int k = a_it % UT_NA;
                    if (!mbar_wait_sleep(afull0 + 8 * k, (uint32_t)(a_it / UT_NA) & 1u)) {
                        report_error(p.err, ERR_FULL_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (live) {
#pragma unroll
                        for (int h = 0; h < UT_SPS; ++h) {
                            const int sbk = s0 + h;
                            const uint32_t a_tmem =
                                tmem + UT_ACOL + (uint32_t)(64 * (UT_SPS * k + h) + 32 * gi);
                            // the start-address field (bits 0..13, bytes / 16) advances
                            // by one sub-block of rows, then by 32 bytes per K step
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
                umma_commit(xempty0 + 8 * slot);  // the x stage is no longer read
                first = false;
                if (++b == p.KB || i == n_iter - 1) {  // the pair's last unit in this range
                    umma_commit(dfull0 + 8 * (d_it % UT_NDB));
                    ++d_it;
                    first = true;
                    b = 0;
                    ++gp;
                }
            }
            // every MMA this CTA issued has completed before TMEM is freed
            umma_commit(mdone);
            if (!mbar_wait_sleep(mdone, 0u))
                report_error(p.err, ERR_DRAIN_WAIT);
        }
    } else if (warp < UT_FIRST_DQ) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int L = 32 * q + lane;  // TMEM lane = row within the tile group
        const size_t seg = (size_t)p.M * UT_PAIR_ROWS;
        const int gp_last = n_iter > 0 ? (int)((u1 - 1) / p.KB) : gp_first - 1;
        for (int gp = gp_first, d = 0; gp <= gp_last; ++gp, ++d) {
            if (!mbar_wait_sleep(dfull0 + 8 * (d % UT_NDB), (uint32_t)(d / UT_NDB) & 1u)) {
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
                float *dst = p.partial + (size_t)(c * 2 + slot) * seg + (size_t)gi * 128 + L;
                // 32 accumulator columns (rows of x) at a time
                constexpr int CC = NP < 32 ? NP : 32;
#pragma unroll
                for (int c0 = 0; c0 < NP; c0 += CC) {
                    uint32_t r[CC / 8][8];
#pragma unroll
                    for (int ch = 0; ch < CC / 8; ++ch)
                        tmem_ld_32x32b_x8(tmem + ((uint32_t)(32 * q) << 16) +
                                              UT_DCOL * (uint32_t)(d % UT_NDB) +
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
                                    p.out[(size_t)(c0 + m) * p.N + n] =
                                        __float2bfloat16_rn(__uint_as_float(r[m / 8][m % 8]));
                        }
                    } else {
#pragma unroll
                        for (int m = 0; m < CC; ++m)
                            if (c0 + m < p.M)
                                dst[(size_t)(c0 + m) * UT_PAIR_ROWS] = __uint_as_float(r[m / 8][m % 8]);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(dempty0 + 8 * (d % UT_NDB));
        }
    } else {
        // ---------------------------------------------------------- dequant
        const int dw = warp - UT_FIRST_DQ;
        const int q = warp & 3, half = (dw >> 2) & 1;
        const int g0 = UT_GPW == 1 ? (dw >> 3) : 0;          // first group of the pair
        const int tl = 2 * q + half;                          // tile of the group
        const uint32_t tlane = (uint32_t)(16 * tl) << 16;    // its 16 TMEM lanes
        const int r = lane >> 2;
        // The stores of a sub-block complete while the next one is dequantized:
        // slot `pend` is published (wait::st, then afull) one step later.
        int a_it = 0, gp = gp_first, b = b_first, pend = -1;
        bool ok = true;
        for (int i = 0; i < n_iter && ok; ++i) {
            const int slot = i % SW;
            if (!mbar_wait_sleep(wfull0 + 8 * slot, (uint32_t)(i / SW) & 1u)) {
                report_error(p.err, ERR_FULL_WAIT);
                break;
            }
            const int ng = (2 * gp + 1 < p.G) ? 2 : 1;
            const uint32_t tbase = smem_addr(wring + slot * UT_CODE_BYTES + tl * UT_TILE_BYTES);
            uint4 wq[UT_GPW][4], sc0[UT_GPW], sc1[UT_GPW], zz[UT_GPW];
#pragma unroll
            for (int gg = 0; gg < UT_GPW; ++gg)
                if (g0 + gg < ng) {
                    const uint32_t tb = tbase + (uint32_t)((g0 + gg) * UT_GROUP_BYTES);
#pragma unroll
                    for (int sbk = 0; sbk < 4; ++sbk)
                        wq[gg][sbk] = lds128(tb + 512 * sbk + 16 * lane);
                    sc0[gg] = lds128(tb + 2048 + 16 * r);
                    sc1[gg] = lds128(tb + 2048 + 128 + 16 * r);
                    zz[gg] = lds128(tb + 2304 + 16 * r);
                }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(wempty0 + 8 * slot);  // the unit's codes are in registers
#pragma unroll
            for (int sbk = 0; sbk < 4; ++sbk) {
                uint32_t v[UT_GPW][16];
#pragma unroll
                for (int gg = 0; gg < UT_GPW; ++gg)
                    if (g0 + gg < ng) {
                        const uint32_t scw[8] = {sc0[gg].x, sc0[gg].y, sc0[gg].z, sc0[gg].w,
                                                 sc1[gg].x, sc1[gg].y, sc1[gg].z, sc1[gg].w};
                        const uint32_t zw[4] = {zz[gg].x, zz[gg].y, zz[gg].z, zz[gg].w};
                        const uint32_t wv[4] = {wq[gg][sbk].x, wq[gg][sbk].y, wq[gg][sbk].z,
                                                wq[gg][sbk].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int g = 2 * sbk + (j >> 1);     // group of 32 within the stage
                            const uint32_t zsrc = zw[g >> 1];
                            const uint32_t zb = (uint32_t)((2 * g) & 3);  // z[r][g]; z[r+8][g] next
                            const uint32_t sp = scw[g];
                            // (128 + z) in both bf16 halves, rows r and r + 8; (s, s) likewise
                            const uint32_t zr = prmt(zsrc, 0x43u, 0x4040u + 0x0101u * zb);
                            const uint32_t zr8 = prmt(zsrc, 0x43u, 0x4040u + 0x0101u * (zb + 1));
                            const uint32_t s2r = prmt(sp, sp, 0x1010u), s2r8 = prmt(sp, sp, 0x3232u);
                            ut_dequant_word(wv[j], zr, zr8, s2r, s2r8, &v[gg][4 * j]);
                        }
                    }
                const int k = a_it % UT_NA;
                if (sbk % UT_SPS == 0) {  // the first sub-block of a slot
                    if (pend >= 0) {      // the previous slot's stores: complete, then publish
                        tmem_wait_st();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(afull0 + 8 * pend);
                        pend = -1;
                    }
                    if (!mbar_wait_sleep(aempty0 + 8 * k, ((uint32_t)(a_it / UT_NA) & 1u) ^ 1u)) {
                        report_error(p.err, ERR_EMPTY_WAIT);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
#pragma unroll
                for (int gg = 0; gg < UT_GPW; ++gg)
                    if (g0 + gg < ng)
                        tmem_st_16x256b_x4(tmem + tlane + UT_ACOL +
                                               (uint32_t)(64 * (UT_SPS * k + sbk % UT_SPS) +
                                                          32 * (g0 + gg)),
                                           v[gg]);
                if (sbk % UT_SPS == UT_SPS - 1) {
                    pend = k;
                    ++a_it;
                }
            }
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

    // The fixup launch may start once every CTA is here (it waits for the
    // grid's completion before reading partials); triggering any earlier
    // would park its blocks, waiting, beside the dequant warps.
    pdl_launch_dependents();
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0)
        W4Q_STAMP(42);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, UT_TMEM_COLS);
    }
}

// x -> the B operand layout.  One thread per (super-block b, sub-block, row < NP, 16-column step j): the
// step's eight column pairs w0..w7 are stored in the order
// w0 w4 w1 w5 | w2 w6 w3 w7 (the column order of the 16x256b TMEM stores of
// A) as two 16-byte chunks 2j, 2j + 1 of the row's 128-byte line, each at
// chunk position (chunk ^ row % 8).  Rows >= M are written as zeros.
__global__ void __launch_bounds__(256) act_prep_umma_kernel(const __nv_bfloat16 *__restrict__ x,
                                                            int M, int K, int NP,
                                                            uint8_t *__restrict__ xs)
{
    if (threadIdx.x == 0 && blockIdx.x == 0)
        W4Q_STAMP(44);
    pdl_launch_dependents();  // the main kernel may start streaming weights
    pdl_wait();               // x (and this workspace) may belong to the previous kernel
    if (threadIdx.x == 0 && blockIdx.x == 0)
        W4Q_STAMP(45);
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    const long long pieces = (long long)(K / 64) * NP * 4;
    if (tid >= pieces)
        return;
    const int j = tid & 3;
    const int row = (tid >> 2) % NP;
    const int bs = (tid >> 2) / NP;  // b * 4 + sub-block
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    if (row < M) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)row * K + bs * 64 + j * 16);
        const uint4 a = src[0], b = src[1];
        lo = make_uint4(a.x, b.x, a.y, b.y);
        hi = make_uint4(a.z, b.z, a.w, b.w);
    }
    uint8_t *line = xs + ((size_t)bs * NP + row) * 128;
    const int r8 = row & 7;
    *reinterpret_cast<uint4 *>(line + ((2 * j) ^ r8) * 16) = lo;
    *reinterpret_cast<uint4 *>(line + ((2 * j + 1) ^ r8) * 16) = hi;
}

// Sum of the fp32 partials of the pairs that several CTAs share, in CTA
// order (deterministic).  Block (pair, ROWS rows of x), one thread per pair
// row: the loads of CHUNK contributors go out together before their
// in-order sum, so the launch is about one wave of a few L2 round trips
// (fix_shape picks ROWS and CHUNK).  Launched behind the main kernel with
// programmatic dependent launch; griddepcontrol.wait holds it until the
// main kernel has finished.
template <int ROWS, int CHUNK>
__global__ void __launch_bounds__(UT_PAIR_ROWS) umma_fixup_kernel(const UParams p)
{
    constexpr int UT_FIX_ROWS = ROWS, UT_FIX_CHUNK = CHUNK;
    // The next call's preparation may launch and wait beside these blocks
    // (measured on 6656 x 19968 at M = 16: 31.1 -> 29.4 us per call).
    pdl_launch_dependents();
    pdl_wait();
    if (threadIdx.x == 0)
        W4Q_STAMP(47);
    const int gp = blockIdx.x, m0 = blockIdx.y * UT_FIX_ROWS, row = threadIdx.x;
    const long long gb = (long long)gp * p.KB, ge = gb + p.KB;
    const int cf = ut_range_owner(p, gb), cl = ut_range_owner(p, ge - 1);
    const int n = gp * UT_PAIR_ROWS + row;
    if (cf == cl || n >= p.N)
        return;  // a whole pair: written by the main kernel
    const size_t seg = (size_t)p.M * UT_PAIR_ROWS;
    const int slot0 = (ut_range_begin(p, cf) == gb) ? 0 : 1;
    const float *first = p.partial + (size_t)(cf * 2 + slot0) * seg + (size_t)m0 * UT_PAIR_ROWS + row;
    const float *rest = p.partial + (size_t)(cf * 2 + 2) * seg + (size_t)m0 * UT_PAIR_ROWS + row;
    const int nc = cl - cf;  // contributors after cf (slot 0 of cf + 1 ..)
    float v[UT_FIX_ROWS];
#pragma unroll
    for (int r = 0; r < UT_FIX_ROWS; ++r)
        v[r] = (m0 + r < p.M) ? __ldcg(first + (size_t)r * UT_PAIR_ROWS) : 0.f;
    for (int j = 0; j < nc; j += UT_FIX_CHUNK) {
        float t[UT_FIX_ROWS][UT_FIX_CHUNK];
#pragma unroll
        for (int r = 0; r < UT_FIX_ROWS; ++r)
#pragma unroll
            for (int u = 0; u < UT_FIX_CHUNK; ++u)
                t[r][u] = (m0 + r < p.M && j + u < nc)
                              ? __ldcg(rest + (size_t)(j + u) * 2 * seg + (size_t)r * UT_PAIR_ROWS)
                              : 0.f;
#pragma unroll
        for (int r = 0; r < UT_FIX_ROWS; ++r)
#pragma unroll
            for (int u = 0; u < UT_FIX_CHUNK; ++u)
                if (j + u < nc)
                    v[r] += t[r][u];
    }
#pragma unroll
    for (int r = 0; r < UT_FIX_ROWS; ++r)
        if (m0 + r < p.M)
            p.out[(size_t)(m0 + r) * p.N + n] = __float2bfloat16_rn(v[r]);
    if (threadIdx.x == 0)
        W4Q_STAMP(48);
}

cudaError_t launch_fixup(const UParams &p, int sm_count, cudaStream_t stream)
{
    const FixShape fs = fix_shape(p.G2, p.M, p.KB, p.U, p.P, p.split, sm_count);
    auto fn = fs.rows == 4 ? (fs.chunk == 4 ? umma_fixup_kernel<4, 4> : umma_fixup_kernel<4, 8>)
                           : (fs.chunk == 4 ? umma_fixup_kernel<8, 4> : umma_fixup_kernel<8, 8>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G2, (unsigned)((p.M + fs.rows - 1) / fs.rows));
    cfg.blockDim = dim3(UT_PAIR_ROWS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <int NP>
cudaError_t launch_umma_np(const UParams &p, cudaStream_t stream)
{
    auto fn = w4_umma_kernel<NP>;
    static std::atomic<unsigned long long> opted_in{0};
    cudaError_t e = smem_opt_in_once(opted_in, fn, ut_smem<NP>());
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(UT_THREADS);
    cfg.dynamicSmemBytes = ut_smem<NP>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

size_t ut_align(size_t v) { return (v + 255) / 256 * 256; }

// Workspace: [x operand (K/256) * NP * 512][partials P * 2 * M * 256 fp32].
struct UtLayout {
    size_t xs, partial, total;
};

UtLayout ut_layout(const W4Plan &pl)
{
    UtLayout L;
    size_t o = 0;
    L.xs = o;
    o += ut_align((size_t)pl.KB * pl.NP * 512);
    L.partial = o;
    o += pl.partial_bytes;
    L.total = o;
    return L;
}

}  // namespace

size_t w4_umma_workspace(const W4Plan &plan) { return ut_layout(plan).total; }

size_t w4_umma_partial_bytes(int P, int M) { return (size_t)P * 2 * M * UT_PAIR_ROWS * sizeof(float); }

cudaError_t launch_w4_umma(const W4Plan &plan, const void *x, const void *packed, void *out,
                           void *workspace, unsigned *err, cudaStream_t stream)
{
    const UtLayout L = ut_layout(plan);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    UParams p = {};
    p.packed = static_cast<const uint8_t *>(packed);
    p.xs = ws + L.xs;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.partial = reinterpret_cast<float *>(ws + L.partial);
    p.err = err;
    p.M = plan.M;
    p.N = plan.N;
    p.K = plan.K;
    p.KB = plan.KB;
    p.G = plan.G;
    p.G2 = plan.G2;
    p.P = plan.P;
    p.split = plan.split;
    p.U = (long long)plan.G2 * plan.KB;
    const long long pieces = (long long)(plan.K / 64) * plan.NP * 4;
    const int blocks = (int)((pieces + 255) / 256);
    // programmatic dependent launch: the preparation launches while the
    // previous kernel finishes and waits for it in griddepcontrol.wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, act_prep_umma_kernel,
                                       static_cast<const __nv_bfloat16 *>(x), plan.M, plan.K,
                                       plan.NP, ws + L.xs);
    if (e != cudaSuccess)
        return e;
    switch (plan.NP) {
    case 16: e = launch_umma_np<16>(p, stream); break;
    case 32: e = launch_umma_np<32>(p, stream); break;
    case 48: e = launch_umma_np<48>(p, stream); break;
    default: e = launch_umma_np<64>(p, stream); break;
    }
    if (e != cudaSuccess || !plan.fixup)
        return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return launch_fixup(p, sms, stream);
}

}  // namespace w4q

W4Q_STAMP_READER(w4q_timeline_read_umma)
