// gemv_w4.cu -- decode-sized W4A16 (M <= 8) / W4A8 linear layer on sm_103a.
// (W4A16 at M >= 9 is a contraction for the tcgen05 tensor core:
// gemv_w4_umma.cu.)
//
//   out[M,N] = x[M,K] . dequant(Wq)[N,K]^T,   dequant(q) = (q - z) * s
//
// ("test_int4_quantized_gemm.py": the dequant + F.linear reference, the W4A8
// bucket kernels and the W4A16 tile kernels; this is a new design for GB300,
// not their code.)
//
// Two launches per call, both with programmatic dependent launch: each
// starts while the kernel before it on the stream finishes and waits for it
// in griddepcontrol.wait before it reads anything that kernel wrote.
//  1. A prologue that zeroes the split-K counters.  Except for W4A16 at
//     M <= 2 (see below), it (act_prep, a few CTAs per activation row) also
//     prepares the activation operand in the workspace, super-block-major
//     ([K/256][M][256 + 8 pad] bf16 and [K/256][M][8] fp32, so one bulk copy
//     moves a stage's rows):
//       W4A16:  per row and 256-column super-block, x' = x * 2^sigma (the
//               W4A16 rule below), X', and the row factor c;
//       W4A8:   sx = fp32(max|x| / 127) per (row, group of 32) or per row,
//               xq = clamp(rint(fp32(x / sx))), x' = xq * 2^121 (2^117 on
//               upper halves), X'[g] = 2^-12 * sum xq (exact), group scale
//               sx * 2^12.
//  2. w4_kernel (it starts streaming weights while the prologue runs): one
//     CTA = 8 consumer warps + 1 producer warp.
//       * The weight is read once: each stage is one 19456-byte bulk copy
//         (TMA engine) of the 8 packed tiles (16 rows x 256 K: codes,
//         scales, zeros) of a 128-row group, plus one copy each of the
//         matching prepared activation rows, into a multi-stage
//         shared-memory ring guarded by mbarriers (the TMA issue rate, about
//         one copy per 70 SM cycles, is a real limit).  Weights carry an L2
//         evict-first hint, activations evict-last.
//       * W4A16 activation rule: per row m and 256-column super-block b,
//         sigma from max |x| over the super-block (so x' stays finite),
//         x' = x * 2^sigma exactly, with an extra 2^-4 on the upper eight
//         columns of every 16-column step, X'[g] = 2^(sigma-133) *
//         sum_{k in g} x_k, and c = 2^(133 - sigma), the factor that takes
//         the super-block's sums back to output units (applied once per
//         stage).  At M <= 2 the producer warp prepares each stage this way
//         itself, from x as given (L2-resident, read with plain loads), one
//         stage behind its weight copies: that keeps two global round trips
//         and a kernel boundary off the critical path of the call.  At
//         M >= 3 the preparation would cost the producer warp's scheduler
//         more than the consumers sharing it can give, so the prologue does
//         it; so it would for W4A8 at any M (its quantizer's divisions).
//       * Consumer warp w owns row tile w of the CTA's 128-row tile group.
//         A lane's 16 bytes of a sub-block hold its A fragments of four
//         m16n8k16 MMAs; masking a word with 0x000F000F / 0x00F000F0 turns
//         its codes into the bf16 numbers q * 2^-133 / q * 2^-129 (exact
//         subnormals / first normals), so dequant is one shift and four ANDs
//         per eight codes.  The 2^4 between the two masks is what the 2^-4
//         on the upper columns of x' undoes.  The tensor core then sums
//         q * x' over each group of 32; the zero point enters as
//         D - z * X'[g] and the scale as acc += s * (D - z * X'[g]) (fp32).
//         For W4A8 every product and partial sum is an exact multiple of
//         2^-12 below 2^12, so the group dot is the exact integer dot.
//       * Work partition: units (tile group, 256-K super-block) are split
//         into P contiguous ranges, one per CTA (balanced "stream-K" ranges
//         over all SM slots by default, or a fixed split of each group's K).
//         A group that one CTA covers entirely is written directly.  For the
//         other groups every contributing warp writes its fp32 partial and
//         bumps a per-row-tile counter; the warp that bumps it last sums the
//         partials in CTA order (deterministic, no floating-point atomics,
//         no waiting on other CTAs) and writes the outputs.
//       * Every wait is bounded (one second of %globaltimer); on expiry the
//         kernel sets a bit in the error word, drains its copies and returns.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "timeline.cuh"
#include "w4_stage.cuh"

// Ring waits of this file: sleeping in mbarrier.try_wait (the default) or
// spinning on it.
#ifdef W4Q_SPIN_WAITS
#define W4Q_RING_WAIT mbar_wait_bounded
#else
#define W4Q_RING_WAIT mbar_wait_sleep
#endif

// Weight stages each CTA issues before its wait for the previous kernel
// (39936 x 6656, W4A8: 3 stages 32.3 us at M = 1 against 32.9 us with 2 or 4).
#ifndef W4Q_SK_PREFETCH
#define W4Q_SK_PREFETCH 3
#endif
static_assert(W4Q_SK_PREFETCH >= 1, "stage 0 is issued before the wait");

namespace w4q {

namespace {


__host__ __device__ __forceinline__ long long range_begin(const Params &p, int c)
{
    if (p.split == 0)
        return (long long)c * p.U / p.P;
    const int g = c / p.split, j = c % p.split;
    return (long long)g * p.KB + (long long)j * p.KB / p.split;
}

// The CTA whose range holds unit u (the largest c with range_begin(c) <= u).
__device__ __forceinline__ int range_owner(const Params &p, long long u)
{
    if (p.split == 0)
        return (int)(((u + 1) * p.P - 1) / p.U);
    const int g = (int)(u / p.KB), b = (int)(u % p.KB);
    return g * p.split + (int)(((long long)(b + 1) * p.split - 1) / p.KB);
}

// W4A16 prepares its activation operand inside the main kernel up to this
// many rows per accumulator slot (MP), in the prologue above.
#ifndef W4Q_INPREP_MAX_MP
#define W4Q_INPREP_MAX_MP 2
#endif
__host__ __device__ constexpr bool in_kernel_prep(W4Mode mode, int mp)
{
    return mode == W4Mode::A16 && mp <= W4Q_INPREP_MAX_MP;
}

template <int NB, W4Mode MODE>
__host__ __device__ constexpr int stage_bytes()
{
    // codes, x' rows, X' rows, and per row the W4A8 group scales (W4A16: the
    // stage's row factor c in the row's first word)
    return WARPS * TILE_BYTES + NB * 8 * XROW + NB * 8 * SROW * 2;
}

template <int NB, W4Mode MODE>
__host__ __device__ constexpr int stages_for()
{
    int s = NB == 1 ? 4 : (NB == 4 ? 3 : 4);
    while (s > 2 && s * stage_bytes<NB, MODE>() + 16 * s > 227 * 1024)
        --s;
    return s;
}

template <int NB, W4Mode MODE>
__host__ __device__ constexpr int smem_for()
{
    // + barriers (full, empty) + a 16-byte zero row (the B rows of the
    // column-packed stage that are zero)
    return stages_for<NB, MODE>() * stage_bytes<NB, MODE>() + (2 * stages_for<NB, MODE>() * 8 + 15) / 16 * 16 + 16;
}

template <int NB, W4Mode MODE, int MP>
__global__ void __launch_bounds__(THREADS, (NB <= 4 ? 2 : 1)) w4_kernel(const Params p)
{
    constexpr bool DOTS = MODE == W4Mode::A8_DOTS;
    constexpr int STAGES = stages_for<NB, MODE>();
    constexpr int SB = stage_bytes<NB, MODE>();
    constexpr int XOFF = WARPS * TILE_BYTES;     // activation rows within a stage
    constexpr int SOFF = XOFF + NB * 8 * XROW;   // group sums within a stage
    constexpr int GOFF = SOFF + NB * 8 * SROW;   // group scales / row factors within a stage
    constexpr bool A16 = MODE == W4Mode::A16;
    constexpr bool INPREP = in_kernel_prep(MODE, MP);  // x' prepared by the producer warp

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * SB);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + STAGES);
    constexpr int ZOFF = (2 * STAGES * 8 + 15) / 16 * 16;
    const uint32_t zrow = smem_addr(smem + STAGES * SB + ZOFF);  // 16 zero bytes

    // Hardware warp 0 is the producer (role index WARPS): the schedulers favour
    // low warp ids, and the W4A16 producer's preparation must not wait behind
    // eight ready consumer warps.  Hardware warps 1 .. 8 are consumers 0 .. 7.
    const int hw_warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warp = hw_warp == 0 ? WARPS : hw_warp - 1;
    const int c = blockIdx.x;
    const long long u0 = range_begin(p, c), u1 = range_begin(p, c + 1);
    const int n_iter = (int)(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // W4A16: the weight copy's arrival + the producer warp's (x' written)
            mbar_init(full0 + 8 * s, INPREP ? 2 : 1);
            mbar_init(empty0 + 8 * s, WARPS);
        }
        *reinterpret_cast<uint4 *>(smem + STAGES * SB + ZOFF) = make_uint4(0u, 0u, 0u, 0u);
        fence_barrier_init();
    }
    {   // activation rows m >= M of every stage stay zero (never copied into)
        const int pad_rows = NB * 8 - p.M;
        const int xper = pad_rows * (XROW / 16);
        const int sper = pad_rows * (SROW / 16) * 2;
        for (int i = threadIdx.x; i < STAGES * (xper + sper); i += THREADS) {
            const int s = i / (xper + sper), rem = i % (xper + sper);
            uint8_t *dst = rem < xper
                               ? smem + s * SB + XOFF + (p.M + rem / (XROW / 16)) * XROW +
                                     (rem % (XROW / 16)) * 16
                               : (rem - xper < pad_rows * 2
                                      ? smem + s * SB + SOFF + (p.M + (rem - xper) / 2) * SROW
                                      : smem + s * SB + GOFF +
                                            (p.M + (rem - xper - pad_rows * 2) / 2) * SROW) +
                                     ((rem - xper) % 2) * 16;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        W4Q_STAMP(10);
    pdl_launch_dependents();  // the next call's preparation may launch and wait

    // stage i processes unit u0 + i = (g, b); both sides step (g, b) along
    const int g_first = (int)(u0 / p.KB), b_first = (int)(u0 % p.KB);
    int issued = 0;
    if (warp == WARPS) {
        if constexpr (INPREP) {
            // ------------------------------------- producer, W4A16 (whole warp)
            // Lane 0 issues the weight copies; the warp prepares x' one stage
            // behind them, from x loaded PD stages ahead of its preparation
            // (so the load latency stays hidden when the preparation is the
            // longer path).  Before waiting for slot i the warp has prepared
            // every stage up to i - 1, so the consumers can always free it.
            constexpr int PD = MP <= 4 ? 2 : 1;
            const uint64_t pol_w = policy_evict_first();
            int g = g_first, b = b_first;   // unit of the next weight copy
            int tdone = 0;                  // stages prepared
            int nload = 0, lb = b_first;    // stages loaded; super-block of the next
            uint4 raw[PD][MP];              // x of stages tdone .. tdone + PD - 1
            auto issue_w = [&](int i) {
                if (lane == 0) {
                    const int slot = i % STAGES;
                    const uint32_t bar = full0 + 8 * slot;
                    mbar_arrive_expect_tx(bar, (uint32_t)(WARPS * TILE_BYTES));
                    bulk_g2s(smem_addr(smem + slot * SB),
                             p.packed + ((size_t)g * p.KB + b) * (WARPS * TILE_BYTES),
                             WARPS * TILE_BYTES, bar, pol_w);
                }
                if (++b == p.KB) {
                    b = 0;
                    ++g;
                }
            };
            auto load_into = [&](uint4 (&dst)[MP]) {
                if (nload < n_iter)
                    load_stage_a16<MP>(p.xin, p.M, p.K, lb, lane, dst);
                ++nload;
                if (++lb == p.KB)
                    lb = 0;
            };
            auto prepare = [&]() {
                const int slot = tdone % STAGES;
                uint8_t *st = smem + slot * SB;
                prep_stage_a16<MP>(raw[0], p.M, lane, st + XOFF, st + SOFF, st + GOFF);
                __syncwarp();  // orders every lane's writes before lane 0's release
                if (lane == 0)
                    mbar_arrive(full0 + 8 * slot);
                ++tdone;
#pragma unroll
                for (int d = 0; d + 1 < PD; ++d)
#pragma unroll
                    for (int m = 0; m < MP; ++m)
                        raw[d][m] = raw[d + 1][m];
                load_into(raw[PD - 1]);
            };
            const int pro = n_iter < STAGES ? n_iter : STAGES;
            const int first = pro < W4Q_SK_PREFETCH ? pro : W4Q_SK_PREFETCH;
            for (int i = 0; i < first; ++i)
                issue_w(i);
            pdl_wait();  // x may come from the previous kernel
            if (lane == 0)
                W4Q_STAMP(11);
#pragma unroll
            for (int d = 0; d < PD; ++d)
                load_into(raw[d]);
            if (n_iter > 0)
                prepare();
            for (int i = first; i < pro; ++i)
                issue_w(i);
            issued = pro;
            while (tdone < pro - 1)
                prepare();
            for (int i = pro; i < n_iter; ++i) {
                const int slot = i % STAGES;
                const uint32_t use = (uint32_t)(i / STAGES);
                const bool got = W4Q_RING_WAIT(empty0 + 8 * slot, (use - 1) & 1);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0)
                        report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                issue_w(i);
                issued = i + 1;
                prepare();  // stage i - 1
            }
            // the last stage (after an error, every issued one, so that the
            // drain below sees each phase complete)
            while (tdone < issued)
                prepare();
        } else if (lane == 0) {
            // --------------------- producer, activation operand from the prologue
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            const uint32_t xbytes = (uint32_t)p.M * XROW, sbytes = (uint32_t)p.M * SROW;
            constexpr bool COPY_G = MODE != W4Mode::A8_DOTS;  // group scales / row factors
            const uint32_t act_bytes = xbytes + sbytes * (COPY_G ? 2u : 1u);
            auto issue_w = [&](int i, int g, int b) {
                const int slot = i % STAGES;
                const uint32_t bar = full0 + 8 * slot;
                mbar_arrive_expect_tx(bar, (uint32_t)(WARPS * TILE_BYTES) + act_bytes);
                bulk_g2s(smem_addr(smem + slot * SB),
                         p.packed + ((size_t)g * p.KB + b) * (WARPS * TILE_BYTES),
                         WARPS * TILE_BYTES, bar, pol_w);
            };
            auto issue_x = [&](int i, int b) {
                const int slot = i % STAGES;
                const uint32_t bar = full0 + 8 * slot;
                bulk_g2s(smem_addr(smem + slot * SB + XOFF),
                         p.x + (size_t)b * p.M * (XROW / 2), xbytes, bar, pol_x);
                bulk_g2s(smem_addr(smem + slot * SB + SOFF),
                         p.xsum + (size_t)b * p.M * (SROW / 4), sbytes, bar, pol_x);
                if (COPY_G)
                    bulk_g2s(smem_addr(smem + slot * SB + GOFF),
                             p.gscale + (size_t)b * p.M * (SROW / 4), sbytes, bar, pol_x);
            };
            // Prologue: two stages of weights go out at once; the activation
            // copies follow as soon as act_prep has finished.  The other
            // stages wait until stage 0 has landed, so that at kernel start
            // every CTA's first stage is not queued behind the whole ring of
            // every other CTA.
            const int pro = n_iter < STAGES ? n_iter : STAGES;
            const int first = pro < W4Q_SK_PREFETCH ? pro : W4Q_SK_PREFETCH;
            int g = g_first, b = b_first;
            for (int i = 0; i < first; ++i) {
                issue_w(i, g, b);
                if (++b == p.KB) {
                    b = 0;
                    ++g;
                }
            }
            pdl_wait();  // the activations come from act_prep, launched just before
            W4Q_STAMP(11);
            int xb = b_first;
            for (int i = 0; i < first; ++i) {
                issue_x(i, xb);
                if (++xb == p.KB)
                    xb = 0;
            }
            issued = first;
            if (pro > first && !W4Q_RING_WAIT(full0, 0u))
                report_error(p.err, ERR_FULL_WAIT);
            for (int i = first; i < pro; ++i) {
                issue_w(i, g, b);
                issue_x(i, xb);
                if (++b == p.KB) {
                    b = 0;
                    ++g;
                }
                if (++xb == p.KB)
                    xb = 0;
            }
            issued = pro;
            for (int i = pro; i < n_iter; ++i) {
                const int slot = i % STAGES;
                const uint32_t use = (uint32_t)(i / STAGES);
                if (!W4Q_RING_WAIT(empty0 + 8 * slot, (use - 1) & 1)) {
                    report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                issue_w(i, g, b);
                issue_x(i, b);
                issued = i + 1;
                if (++b == p.KB) {
                    b = 0;
                    ++g;
                }
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        pdl_wait();  // the prologue's outputs (counters, W4A8 operand) are read below
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
            acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
        int cur_g = g_first;
        bool ok = true;
        const int r = lane >> 2, c2 = 2 * (lane & 3);

        auto flush = [&](int g) {
            if (DOTS)
                return;
            if constexpr (NB == 1 && MP < 8) {
                // add the slots: lanes of one row hold other groups of the same outputs
                if (MP == 1) {
                    acc[0][0] += acc[0][1];
                    acc[0][2] += acc[0][3];
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (MP <= 2)
                        acc[0][e] += __shfl_xor_sync(0xffffffffu, acc[0][e], 1);
                    acc[0][e] += __shfl_xor_sync(0xffffffffu, acc[0][e], 2);
                }
            }
            const int tile = g * WARPS + warp;
            if (tile >= p.T)
                return;
            const long long gb = (long long)g * p.KB, ge = gb + p.KB;
            if (gb >= u0 && ge <= u1) {  // the whole group is ours: write the outputs
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = nb * 8 + c2 + (e & 1);
                        const int n = tile * 16 + r + 8 * (e >> 1);
                        if (m < p.M && n < p.N)
                            p.out[(size_t)m * p.N + n] = __float2bfloat16_rn(acc[nb][e]);
                    }
                return;
            }
            // shared group: publish this warp's partial, count it, and let the
            // last of the group's contributors sum all partials in CTA order
            const size_t seg = (size_t)p.M * GROUP_ROWS;
            const int slot = (g == g_first) ? 0 : 1;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = nb * 8 + c2 + (e & 1);
                    const int row = r + 8 * (e >> 1);
                    if (m < p.M)
                        p.partial[(size_t)(c * 2 + slot) * seg + (size_t)m * GROUP_ROWS +
                                  warp * 16 + row] = acc[nb][e];
                }
            const int cf = range_owner(p, gb), cl = range_owner(p, ge - 1);
            unsigned last = 0;
            __syncwarp();  // the warp's partial writes are ordered before lane 0's release
            if (lane == 0)
                last = (atomic_add_acq_rel(&p.counters[(size_t)g * WARPS + warp], 1u) ==
                        (unsigned)(cl - cf));
            last = __shfl_sync(0xffffffffu, last, 0);
            __syncwarp();  // lane 0's acquire is ordered before every lane's reads
            if (!last)
                return;
            const int slot0 = (range_begin(p, cf) == gb) ? 0 : 1;
            const int nc = cl - cf + 1;
            // this lane's outputs i = lane + 32 k (M * 16 of them per row tile);
            // the loads of all of them go out together, eight contributors at
            // a time, and each output is summed in CTA order
            constexpr int MMAX = NB == 1 ? MP : NB * 8;  // M <= MMAX
            constexpr int NV = MMAX * 16 / 32 > 0 ? MMAX * 16 / 32 : 1;
            const float *first[NV], *rest[NV];
            bool live[NV];
            float v[NV];
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int i = lane + 32 * k, m = i / 16, row = i % 16;
                live[k] = i < p.M * 16;
                const size_t off = (size_t)(live[k] ? m : 0) * GROUP_ROWS + warp * 16 + row;
                first[k] = p.partial + (size_t)(cf * 2 + slot0) * seg + off;
                rest[k] = p.partial + (size_t)(cf * 2 + 2) * seg + off;  // slot 0 of cf+1..
                v[k] = live[k] ? __ldcg(first[k]) : 0.f;
            }
            for (int j = 0; j + 1 < nc; j += 8) {
                float t[NV][8];
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        t[k][q] = (live[k] && j + q + 1 < nc)
                                      ? __ldcg(rest[k] + (size_t)(j + q) * 2 * seg) : 0.f;
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (j + q + 1 < nc)
                            v[k] += t[k][q];
            }
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int i = lane + 32 * k, m = i / 16, n = tile * 16 + i % 16;
                if (live[k] && n < p.N)
                    p.out[(size_t)m * p.N + n] = __float2bfloat16_rn(v[k]);
            }
        };

        int g = g_first, b = b_first;
        for (int i = 0; i < n_iter; ++i) {
            if (g != cur_g) {
                flush(cur_g);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
                    acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
                cur_g = g;
            }
            const int slot = i % STAGES;
            if (!W4Q_RING_WAIT(full0 + 8 * slot, (uint32_t)(i / STAGES) & 1)) {
                report_error(p.err, ERR_FULL_WAIT);
                ok = false;
                break;
            }
            if (i == 0 && lane == 0 && warp == 0)
                W4Q_STAMP(13);
            const int tile = g * WARPS + warp;
            if (tile < p.T)
            {
                if constexpr (NB == 1 && MP < 8)
                    compute_stage_packed<MP, DOTS, MODE == W4Mode::A8, A16>(
                        smem_addr(smem + slot * SB + warp * TILE_BYTES),
                        smem_addr(smem + slot * SB + XOFF), smem_addr(smem + slot * SB + SOFF),
                        smem_addr(smem + slot * SB + GOFF), zrow, lane, acc, p, tile, b);
                else
                    compute_stage<NB, DOTS, MODE == W4Mode::A8, A16>(
                        smem_addr(smem + slot * SB + warp * TILE_BYTES),
                        smem_addr(smem + slot * SB + XOFF), smem_addr(smem + slot * SB + SOFF),
                        smem_addr(smem + slot * SB + GOFF), lane, acc, p, tile, b);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * slot);
            if (++b == p.KB) {
                b = 0;
                ++g;
            }
        }
        if (lane == 0 && warp == 0)
            W4Q_STAMP(14);
        if (ok && n_iter > 0)
            flush(cur_g);
        if (lane == 0 && warp == 0)
            W4Q_STAMP(15);
    }

    __syncthreads();
    if (threadIdx.x == 0)
        W4Q_STAMP(16);
    // Drain: every issued stage's copies must have landed before the CTA's
    // shared memory goes away (only the error path can leave some pending).
    if (warp == WARPS && lane == 0) {
        for (int s = 0; s < STAGES && s < issued; ++s) {
            const int last_use = (issued - 1 - s) / STAGES;
            if (!W4Q_RING_WAIT(full0 + 8 * s, (uint32_t)last_use & 1)) {
                report_error(p.err, ERR_DRAIN_WAIT);
                break;
            }
        }
    }
}

// The prologue (see the file comment).  Both kernels zero the split-K
// counters after the previous kernel on the stream has finished with them;
// act_prep also writes the activation operand, super-block-major:
// xp[(k/256)*M + m][264] (16 pad bytes per row), xsum and gscale
// [(g/8)*M + m][8] (W4A16: the row factor c in the row's first word).
constexpr int PREP_THREADS = 256;
constexpr int PREP_CHUNK = PREP_THREADS * 8;  // columns one act_prep CTA transforms

__global__ void __launch_bounds__(PREP_THREADS) splitk_reset_kernel(unsigned *__restrict__ counters,
                                                                    int ncounters)
{
    if (threadIdx.x == 0)
        W4Q_STAMP(1);
    pdl_launch_dependents();  // the main kernel may start streaming weights
    pdl_wait();               // the previous kernel may still use these counters
    if (threadIdx.x == 0)
        W4Q_STAMP(2);
    for (int i = blockIdx.x * PREP_THREADS + threadIdx.x; i < ncounters; i += gridDim.x * PREP_THREADS)
        counters[i] = 0u;
}

// Largest |x| over the whole row m of x (bf16 [.][K]), for every thread of
// the block: magnitudes of bf16 numbers order as their bit patterns, so the
// reduction runs on integers.  The row is read from L2 by every block that
// needs it.
__device__ __forceinline__ float row_absmax(const __nv_bfloat16 *__restrict__ x, int m, int K)
{
    __shared__ uint32_t wmax[32];
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
    uint32_t h = 0u;
#pragma unroll 4
    for (int j = threadIdx.x; j < K / 8; j += blockDim.x) {
        const uint4 v = row[j];
        h = __vmaxu2(h, __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                 __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
    }
    h = max(h & 0xFFFFu, h >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = h;
    __syncthreads();
    h = 0u;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
        h = max(h, wmax[w]);
    return __uint_as_float(h << 16);
}

// grid = (M, ceil(K / PREP_CHUNK)); 8 consecutive values per thread, 4
// consecutive threads per group of 32, one warp per 256-column super-block.
// W4A8 (A16 false): ROW = one activation scale for the whole row (every
// block of the row finds the row's max itself), else one per group of 32.
template <bool A16, bool ROW>
__global__ void __launch_bounds__(PREP_THREADS) act_prep_kernel(
    const __nv_bfloat16 *__restrict__ x, int M, int K, __nv_bfloat16 *__restrict__ xp,
    float *__restrict__ xsum, float *__restrict__ gscale, unsigned *__restrict__ counters,
    int ncounters)
{
    if (threadIdx.x == 0)
        W4Q_STAMP(4);
    pdl_launch_dependents();  // the main kernel may start streaming weights
    pdl_wait();               // x (and this workspace) may belong to the previous kernel
    if (threadIdx.x == 0)
        W4Q_STAMP(5);
    const int nblk = gridDim.x * gridDim.y;
    const int bid = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = bid * PREP_THREADS + threadIdx.x; i < ncounters; i += nblk * PREP_THREADS)
        counters[i] = 0u;
    const int m = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
    const int n8 = K / 8;
    const int i = blockIdx.y * PREP_THREADS + threadIdx.x;
    const bool live = i < n8;
    const uint4 raw = live ? row[i] : make_uint4(0u, 0u, 0u, 0u);  // before the row pass: one round trip
    const float arow = ROW ? row_absmax(x, m, K) : 0.f;
    float v[8];
    if (live) {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = bf16lo_to_f32(w[j]);
            v[2 * j + 1] = bf16hi_to_f32(w[j]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = 0.f;
    }
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        a = fmaxf(a, fabsf(v[j]));
    int sigma = 121;  // x' = value * 2^sigma on lower half-steps (2^(sigma-4) upper)
    if (A16) {
        // the power-of-two prescale from max |x| over the warp's super-block
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        int e = 0;
        if (a > 0.f)
            (void)frexpf(a, &e);  // a < 2^e
        sigma = min(max(128 - e, 6), 259);
        if (live && (i & 31) == 0)
            gscale[((size_t)(i / 32) * M + m) * 8] = ldexpf(1.0f, 133 - sigma);
    } else {
        // one scale per group of 32 (or per row, ROW): sx = fp32(max |x| / 127),
        // xq = clamp(rint(x / sx))
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        if (ROW)
            a = arow;
        const float sxg = __fdiv_rn(a, 127.0f);
        if (a == 0.f) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = 0.f;
        } else {
            act_code8(v, sxg);
        }
        const int g = i / 4;  // x 2^12: the group dots come out of the MMA scaled by 2^-12
        if (live && (i & 3) == 0)
            gscale[((size_t)(g / 8) * M + m) * 8 + (g % 8)] = sxg * 4096.0f;
    }
    float part = 0.f;
    if (live) {
        const int k0 = 8 * i;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            part += v[j];
        // columns 8i .. 8i+7: upper half of a 16-column step when i is odd
        const int sh = (i & 1) ? sigma - 4 : sigma;
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            ow[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(ldexpf(v[2 * j], sh))) |
                    ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(ldexpf(v[2 * j + 1], sh)))
                     << 16);
        const uint4 o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        const size_t dst = ((size_t)(k0 / 256) * M + m) * 264 + (k0 % 256);
        *reinterpret_cast<uint4 *>(xp + dst) = o;
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    if (live && (i & 3) == 0) {
        const int g = i / 4;
        xsum[((size_t)(g / 8) * M + m) * 8 + (g % 8)] = ldexpf(part, A16 ? sigma - 133 : -12);
    }
}

// W4A8 activation quantizer alone (int8 output, one fp32 scale per (row,
// group of 32), or per row (ROW); the test view of the same rule act_prep
// applies).  One CTA per row; 4 consecutive threads per group.
template <bool ROW>
__global__ void __launch_bounds__(512) act_quant_i8_kernel(const __nv_bfloat16 *__restrict__ x,
                                                           int K, int8_t *__restrict__ xq,
                                                           float *__restrict__ sx)
{
    const int m = blockIdx.x;
    const float arow = ROW ? row_absmax(x, m, K) : 0.f;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
    const int n8 = K / 8;
    for (int i0 = 0; i0 < n8; i0 += blockDim.x) {  // blockDim is a multiple of 32
        const int i = i0 + threadIdx.x;
        float f[8];
        if (i < n8) {
            const uint4 v = row[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
                f[j] = (j & 1) ? bf16hi_to_f32(w[j / 2]) : bf16lo_to_f32(w[j / 2]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                f[j] = 0.f;
        }
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            a = fmaxf(a, fabsf(f[j]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        if (ROW)
            a = arow;
        const float s = __fdiv_rn(a, 127.0f);
        if (i < n8) {
            if (ROW ? i == 0 : (i & 3) == 0)
                sx[ROW ? (size_t)m : (size_t)m * (K / 32) + i / 4] = s;
            uint32_t q[2] = {0u, 0u};
            if (a == 0.f) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    f[j] = 0.f;
            } else {
                act_code8(f, s);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                q[j / 4] |= (uint32_t)(uint8_t)(int8_t)f[j] << (8 * (j % 4));
            reinterpret_cast<uint2 *>(xq + (size_t)m * K)[i] = make_uint2(q[0], q[1]);
        }
    }
}

// ------------------------------------------------------------------ host

template <int NB, W4Mode MODE>
int ctas_per_sm(int dev)
{
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64)
        return 1;
    if (cache[dev] == 0) {
        auto fn = w4_kernel<NB, MODE, 8>;  // occupancy is set by shared memory, not MP
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_for<NB, MODE>());
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, THREADS, smem_for<NB, MODE>()) !=
                cudaSuccess ||
            n < 1)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

int nb_for(int M) { return M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8)); }

// Rows of x per accumulator slot at NB = 1 (M rounded up to a power of two).
#ifndef W4Q_MP_MIN
#define W4Q_MP_MIN 1
#endif
int mp_for(int M)
{
    const int mp = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
    return mp < W4Q_MP_MIN ? W4Q_MP_MIN : mp;
}


template <int NB, W4Mode MODE, int MP>
cudaError_t launch_main(const Params &p, cudaStream_t stream)
{
    auto fn = w4_kernel<NB, MODE, MP>;
    // the dynamic shared-memory opt-in, once per device (a bit per device)
    static std::atomic<unsigned long long> opted_in{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit == 0 || !(opted_in.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_for<NB, MODE>());
        if (e != cudaSuccess)
            return e;
        opted_in.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem_for<NB, MODE>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <W4Mode MODE>
cudaError_t dispatch_main(const W4Plan &plan, const Params &p, cudaStream_t stream)
{
    if (plan.NB == 1) {
        switch (mp_for(plan.M)) {
        case 1: return launch_main<1, MODE, 1>(p, stream);
        case 2: return launch_main<1, MODE, 2>(p, stream);
        case 4: return launch_main<1, MODE, 4>(p, stream);
        default: return launch_main<1, MODE, 8>(p, stream);
        }
    }
    // W4A16 above 8 rows runs on the tcgen05 kernel; W4A8 is planned up to 8 rows
    return cudaErrorInvalidValue;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace layout: [x' bf16 (K/256)*M*264][X' f32 (K/256)*M*8]
//                   [group scales / row factors f32 (K/256)*M*8] (not for
//                   W4A16 at MP <= 2), then
//                   [counters u32 G*8][partials f32 P*2*M*128], 256-byte aligned.
struct WsLayout {
    size_t xp, xsum, gscale, counters, partial, total;
};

WsLayout ws_layout(const W4Plan &pl, W4Mode mode)
{
    WsLayout L;
    // the operand the prologue prepares (W4A16 at MP <= 2: none, the main kernel does it)
    const bool a8 = !in_kernel_prep(mode, mp_for(pl.M));
    size_t o = 0;
    L.xp = o;
    o += a8 ? align_up((size_t)pl.KB * pl.M * XROW, 256) : 0;
    L.xsum = o;
    o += a8 ? align_up((size_t)pl.KB * pl.M * SROW, 256) : 0;
    L.gscale = o;
    o += a8 ? align_up((size_t)pl.KB * pl.M * SROW, 256) : 0;
    L.counters = o;
    o += pl.fixup ? align_up((size_t)pl.G * WARPS * 4, 256) : 0;
    L.partial = o;
    o += pl.partial_bytes;
    L.total = o;
    return L;
}

// The K split C (CTAs per cluster) of the cluster kernel for M <= 8, or 0
// when no split fits its shared memory.  Model: two CTAs per SM; a call
// takes about (waves of CTAs) x (super-blocks per CTA + 2) stage times, the
// + 2 standing for each CTA's fixed part (activation preparation, ramp,
// cluster reduction); ties go to the smaller split.
// The measured split table (tune_splits.py): the fastest K split of listed
// M <= 8 calls on a GPU with this many SMs.
struct SplitEntry {
    int sms, kind, M, N, K, split, ns;
};
const SplitEntry kSplitTable[] = {
#include "split_table.inc"
    {0, 0, 0, 0, 0, 0, 0}};

// kind: 0 W4A16, 1 W4A8 with a scale per group, 2 W4A8 with a scale per row
int table_split(int sms, int kind, int M, int N, int K)
{
    for (const SplitEntry &e : kSplitTable)
        if (e.sms == sms && e.kind == kind && e.M == M && e.N == N && e.K == K)
            return e.split;
    return -1;
}

int cluster_choice(int M, int G, int KB, int sm_count)
{
    const long long slots = 2LL * (sm_count > 0 ? sm_count : 1);
    int best = 0;
    long long best_cost = 0;
    for (int C = 1; C <= 8 && C <= KB; ++C) {
        if (w4_cluster_ring(M, KB, C) == 0)
            continue;
        const long long waves = ((long long)G * C + slots - 1) / slots;
        const long long cost = waves * ((KB + C - 1) / C + 2);
        if (best == 0 || cost < best_cost) {
            best = C;
            best_cost = cost;
        }
    }
    return best;
}

}  // namespace

bool w4_plan(int M, int N, int K, int split, int sm_count, W4Mode mode, W4Plan *plan,
             bool act_row, bool compact)
{
    if (M < 1 || M > 64 || N < 1 || K < 256 || K % 256 != 0)
        return false;
    if (mode != W4Mode::A16 && M > 8)
        return false;  // W4A8 serves decode rows (the pages' buckets are 1..4)
    W4Plan pl = {};
    pl.M = M;
    pl.N = N;
    pl.K = K;
    pl.KB = K / 256;
    pl.T = (N + 15) / 16;
    pl.G = (pl.T + WARPS - 1) / WARPS;
    pl.NB = nb_for(M);
#ifndef W4Q_UMMA_MIN_M
#define W4Q_UMMA_MIN_M 9
#endif
    pl.umma = (mode == W4Mode::A16) && M >= W4Q_UMMA_MIN_M;  // W4A16 on the tcgen05 tensor core
    pl.fold = pl.umma;  // the dequantized weight is rounded to bf16 there
    pl.NP = (M + 15) / 16 * 16;
    pl.G2 = (pl.G + 1) / 2;
    const int groups = pl.umma ? pl.G2 : pl.G;  // work-unit rows: tile groups or pairs
    const long long U = (long long)groups * pl.KB;
    // M <= 8: the cluster kernel (one launch, no workspace) takes the
    // library's own choice and explicit splits of 1..8 whenever the slice
    // of activations it keeps in shared memory fits; stream-K (split 0),
    // larger explicit splits and the longest K stay on the stream-K kernel.
    if (compact && (pl.umma || mode != W4Mode::A16))
        return false;  // the compact metadata is read by the cluster kernel (W4A16, M <= 8)
    if (!pl.umma && split < 0) {
        // a measured choice for this call, if the table has one
        const int t = table_split(sm_count, mode == W4Mode::A16 ? 0 : (act_row ? 2 : 1), M, N, K);
        if (t >= 0 && t <= pl.KB)
            split = t;
    }
    if (!pl.umma) {
        int C = split < 0 ? cluster_choice(M, pl.G, pl.KB, sm_count)
                          : (split >= 1 && split <= 8 && w4_cluster_ring(M, pl.KB, split) > 0
                                 ? split : 0);
        if (compact && C == 0 && split <= 0)
            C = cluster_choice(M, pl.G, pl.KB, sm_count);  // never the stream-K kernel
        if (C > 0) {
            pl.cluster = C;
            pl.compact = compact;
            pl.split = C;
            pl.P = pl.G * C;
            pl.fixup = false;
            pl.partial_bytes = 0;
            *plan = pl;
            return true;
        }
    }
    if (compact)
        return false;  // no cluster split fits
    if (mode == W4Mode::A8_DOTS)
        split = 1;  // every unit is processed once; no accumulation across CTAs
    // Tensor-core path with few super-blocks and no more row-group pairs than
    // SMs: each CTA takes a pair's whole K.  The partial-sum launch a split
    // would need costs more than the CTA's extra stages (1536 x 512, M = 16:
    // 7.1 -> 4.8 us).
    if (split < 0 && pl.umma && pl.KB <= 4 && pl.G2 <= (sm_count > 0 ? sm_count : 1))
        split = 1;
    if (split < 0)
        split = 0;
    if (split >= 1) {
        if (split > pl.KB)
            return false;
        pl.split = split;
        pl.P = groups * split;
        pl.fixup = split > 1;
    } else {
        int dev = 0;
        cudaGetDevice(&dev);
        const int per_sm = pl.umma ? 1
                           : (mode == W4Mode::A16) ? ctas_per_sm<1, W4Mode::A16>(dev)
                                                   : ctas_per_sm<1, W4Mode::A8>(dev);
        const long long slots = (long long)(sm_count > 0 ? sm_count : 1) * per_sm;
        pl.split = 0;
        pl.P = (int)(U < slots ? U : slots);
        pl.fixup = !(U % pl.P == 0 && (U / pl.P) % pl.KB == 0);
    }
    if (mode == W4Mode::A8_DOTS)
        pl.fixup = false;
    pl.partial_bytes = !pl.fixup ? 0
                       : pl.umma ? w4_umma_partial_bytes(pl.P, M)
                                 : (size_t)pl.P * 2 * M * GROUP_ROWS * sizeof(float);
    *plan = pl;
    return true;
}

size_t w4_workspace_for(const W4Plan &plan, W4Mode mode)
{
    if (plan.cluster > 0)
        return 0;
    return plan.umma ? w4_umma_workspace(plan) : ws_layout(plan, mode).total;
}

cudaError_t launch_w4(const W4Plan &plan, W4Mode mode, const void *x, const void *packed,
                      void *out, int32_t *dots, void *workspace, unsigned *err,
                      cudaStream_t stream, bool act_row)
{
    if (plan.umma)
        return launch_w4_umma(plan, x, packed, out, workspace, err, stream);
    if (plan.cluster > 0)
        return launch_w4_cluster(plan, mode, act_row, x, packed, out, dots, err, stream);
    const WsLayout L = ws_layout(plan, mode);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    Params p = {};
    p.packed = static_cast<const uint8_t *>(packed);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.dots = dots;
    p.err = err;
    p.M = plan.M;
    p.N = plan.N;
    p.K = plan.K;
    p.KB = plan.KB;
    p.T = plan.T;
    p.G = plan.G;
    p.P = plan.P;
    p.split = plan.split;
    p.U = (long long)plan.G * plan.KB;
    p.x = reinterpret_cast<const __nv_bfloat16 *>(ws + L.xp);
    p.xsum = reinterpret_cast<const float *>(ws + L.xsum);
    p.gscale = reinterpret_cast<const float *>(ws + L.gscale);
    p.xin = static_cast<const __nv_bfloat16 *>(x);
    p.counters = reinterpret_cast<unsigned *>(ws + L.counters);
    p.partial = reinterpret_cast<float *>(ws + L.partial);
    const int ncounters = plan.fixup ? plan.G * WARPS : 0;
    unsigned *cnt = reinterpret_cast<unsigned *>(ws + L.counters);
    // programmatic dependent launch: the prologue launches while the
    // previous kernel finishes and waits for it in griddepcontrol.wait
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(PREP_THREADS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (in_kernel_prep(mode, mp_for(plan.M))) {
        const int nblk = (ncounters + PREP_THREADS - 1) / PREP_THREADS;
        cfg.gridDim = dim3((unsigned)(nblk < 1 ? 1 : (nblk > 16 ? 16 : nblk)));
        e = cudaLaunchKernelEx(&cfg, splitk_reset_kernel, cnt, ncounters);
    } else {
        cfg.gridDim = dim3((unsigned)plan.M, (unsigned)((plan.K + PREP_CHUNK - 1) / PREP_CHUNK));
        e = cudaLaunchKernelEx(&cfg, mode == W4Mode::A16 ? act_prep_kernel<true, false>
                                     : (act_row ? act_prep_kernel<false, true>
                                                : act_prep_kernel<false, false>),
                               static_cast<const __nv_bfloat16 *>(x),
                               plan.M, plan.K, reinterpret_cast<__nv_bfloat16 *>(ws + L.xp),
                               reinterpret_cast<float *>(ws + L.xsum),
                               reinterpret_cast<float *>(ws + L.gscale), cnt, ncounters);
    }
    if (e != cudaSuccess)
        return e;
    if (mode == W4Mode::A16)
        return dispatch_main<W4Mode::A16>(plan, p, stream);
    if (mode == W4Mode::A8)
        return dispatch_main<W4Mode::A8>(plan, p, stream);
    return dispatch_main<W4Mode::A8_DOTS>(plan, p, stream);
}

cudaError_t launch_act_quant_i8(const void *x, int M, int K, int8_t *xq, float *sx, bool row,
                                cudaStream_t stream)
{
    if (row)
        act_quant_i8_kernel<true><<<M, 512, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), K,
                                                         xq, sx);
    else
        act_quant_i8_kernel<false><<<M, 512, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), K,
                                                          xq, sx);
    return cudaGetLastError();
}

}  // namespace w4q

W4Q_STAMP_READER(w4q_timeline_read_w4)
