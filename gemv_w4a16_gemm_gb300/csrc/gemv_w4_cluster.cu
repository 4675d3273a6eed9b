// gemv_w4_cluster.cu -- decode-sized W4A16 / W4A8 linear layer for 1 <= M <= 8
// on sm_103a, one thread-block cluster per 128-row group:
//
//   out[M,N] = x[M,K] . dequant(Wq)[N,K]^T,   dequant(q) = (q - z) * s
//
// ("test_int4_quantized_gemm.py": the dequant + F.linear reference and the
// W4A8 bucket kernels; a GB300 design of this library, not their code.)
//
// One launch per call, no workspace:
//  * The grid is (C, G): cluster g (C CTAs along x) owns the 128-row group g
//    of the packed weight, and its CTA of rank r streams the contiguous
//    super-blocks [r*KB/C, (r+1)*KB/C) of K (KB = K/256).  C is the call's
//    K split (1..8).
//  * The weight stream of each CTA starts before griddepcontrol.wait: the
//    first stages are in flight while the kernel before it on the stream
//    finishes (the weights are not written by that kernel).
//  * After the wait, all nine warps prepare the CTA's slice of the
//    activations in shared memory, once for all its stages:
//      W4A16: per row and super-block a power-of-two prescale sigma,
//             x' = x * 2^sigma (2^(sigma-4) on the upper eight columns of
//             every 16-column step), X'[g] = 2^(sigma-133) * sum_{k in g} x,
//             c = 2^(133 - sigma);
//      W4A8:  symmetric int8 xq = clamp(rint(x / sx), -127, 127) in IEEE
//             fp32, with sx = fp32(max|x| / 127) over a group of 32 or over
//             the whole row; x' = xq * 2^121 (2^117 upper), X' = 2^-12 *
//             sum xq, and sx * 2^12 per group.  The row scale needs the max
//             over all of K: each CTA reduces its slice and sends its maxima
//             to every other CTA of the cluster (asynchronous stores into
//             their shared memory that count on their barriers); each CTA
//             takes the max of the C slices' values.
//  * Eight consumer warps each own one 16-row tile and run the same stage
//    arithmetic as the stream-K kernel (w4_stage.cuh): bf16 m16n8k16 MMAs on
//    the masked nibbles, exact per-group dots, the fp32 scale / zero update.
//  * Split-K reduction: every CTA of rank r > 0 sends its 128 x MP fp32 sums
//    into slot r - 1 of rank 0's shared memory with asynchronous stores
//    whose bytes count on a barrier of rank 0, and leaves; rank 0 waits for
//    all the bytes, adds the C ranks' sums in rank order (fixed order: the
//    result does not depend on timing) and writes them as bf16.  The only
//    wait on other CTAs is rank 0's, on data already sent.  The barriers
//    that receive remote bytes are initialised before a cluster-wide
//    arrive (relaxed) that every thread passes at the start, and each CTA
//    waits on that cluster barrier before its first remote store.
//  * Every ring wait is bounded (one second of %globaltimer): on expiry the
//    kernel sets a bit in the error word, still passes the cluster barriers
//    (every thread reaches them on every path), drains its copies and
//    returns.
#include <atomic>

#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "timeline.cuh"
#include "w4_stage.cuh"

#ifdef W4Q_SPIN_WAITS
#define W4Q_RING_WAIT mbar_wait_bounded
#else
#define W4Q_RING_WAIT mbar_wait_sleep
#endif

// Largest rows-per-slot count at which consumers take ring stages two at a
// time (measured: a gain at one row per slot, a loss at two on 6656 x 4096 and
// 8448 x 6656).
#ifndef W4Q_CL_PAIR_MP
#define W4Q_CL_PAIR_MP 1
#endif

namespace w4q {

namespace {

constexpr int MAX_CLUSTER = 8;   // portable cluster size
constexpr int CTA_SMEM_MAX = 113 * 1024;  // two CTAs per SM

struct CParams {
    const uint8_t *packed;
    const __nv_bfloat16 *x;  // bf16 [M][K], as given
    __nv_bfloat16 *out;      // bf16 [M][N]
    int32_t *dots;           // W4A8 group-dot export: int32 [M][N][K/32]
    unsigned *err;
    int M, N, K, KB, T, G, C, smax, R;  // R: weight ring stages (2..4)
};

// ------------------------------------------------------------ cluster PTX

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The split form: arrive (relaxed: nothing before it needs publishing
// beyond the barrier initialisation, which its fence releases) at the
// start, wait before the first remote operation.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// 16 bytes from registers into another CTA's shared memory (shared::cluster
// addresses of the data and of that CTA's barrier), counted on the barrier
// as transaction bytes.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint4 v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
                 : "memory");
}

// The shared::cluster address of this CTA's shared-memory address `addr` in
// the CTA of rank `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}

// ----------------------------------------------------------- smem layout

struct CLayout {
    int ring, xr, xs, xg, red, recv, rowmax, zero, bars, total;
};

// [ring: R x 19456][x': smax x MP x 528][X': smax x MP x 32][factors:
// smax x MP x 32][partial sums: 128 x MP f32][received sums (rank 0):
// (C-1) x 128 x MP f32][row maxima: own + received, C x 8 u32][16 zero
// bytes][barriers: 2R ring + received sums + received maxima, x 8]
__host__ __device__ inline CLayout c_layout(int mp, int smax, int R, int C, int tile_bytes)
{
    CLayout L;
    int o = 0;
    L.ring = o;
    o += R * WARPS * tile_bytes;
    L.xr = o;
    o += smax * mp * XROW;
    L.xs = o;
    o += smax * mp * SROW;
    L.xg = o;
    o += smax * mp * SROW;
    L.red = o;
    o += GROUP_ROWS * mp * 4;
    L.recv = o;
    o += (C - 1) * GROUP_ROWS * mp * 4;
    L.rowmax = o;
    o += C * 32;
    L.zero = o;
    o += 16;
    L.bars = o;
    o += (2 * R + 2) * 8;
    L.total = (o + 127) / 128 * 128;
    return L;
}

// W4A8: one super-block's int8 activations from the raw bf16 of MP rows
// (lane l holds columns 8l .. 8l + 7), with the scale of the lane's group of
// 32 (its 4 lanes) or, ROW, of the whole row (arow = the row's max |x|):
// x' = xq * 2^121 (2^117 on the odd lanes, the upper half of a 16-column
// step), X'[g] = 2^-12 * sum xq, and the group scale sx * 2^12.
template <int MP, bool ROW>
__device__ __forceinline__ void prep_stage_a8(const uint4 (&raw)[MP], int M, int lane,
                                              const float (&arow)[MP], uint8_t *xdst,
                                              uint8_t *sdst, uint8_t *gdst)
{
#pragma unroll
    for (int m = 0; m < MP; ++m) {
        const uint32_t w[4] = {raw[m].x, raw[m].y, raw[m].z, raw[m].w};
        float v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = bf16lo_to_f32(w[j]);
            v[2 * j + 1] = bf16hi_to_f32(w[j]);
        }
        float a = 0.f;
        if (ROW) {
            a = arow[m];
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                a = fmaxf(a, fabsf(v[j]));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        }
        const float sx = __fdiv_rn(a, 127.0f);
        if (a == 0.f) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = 0.f;
        } else {
            act_code8(v, sx);
        }
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            part += v[j];
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        // |xq| <= 127 has at most 7 significant bits: xq * 2^sh is exact in bf16
        const float f = __uint_as_float((uint32_t)(((lane & 1) ? 117 : 121) + 127) << 23);
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * j] * f, v[2 * j + 1] * f);
            ow[j] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        if (m < M) {
            *reinterpret_cast<uint4 *>(xdst + m * XROW + 16 * lane) =
                make_uint4(ow[0], ow[1], ow[2], ow[3]);
            if ((lane & 3) == 0) {
                *reinterpret_cast<float *>(sdst + m * SROW + 4 * (lane >> 2)) = part * 0x1p-12f;
                *reinterpret_cast<float *>(gdst + m * SROW + 4 * (lane >> 2)) = sx * 4096.0f;
            }
        }
    }
}

// Tile bytes: the standard metadata (bf16 scale, u8 zero) or the compact one
// (u8 scale and zero codes; the fp16 row steps after the tiles).
constexpr int CMP_TILE_BYTES = 2304;

template <W4Mode MODE, bool ROW, int MP, bool CMP>
__global__ void __launch_bounds__(THREADS, 2) w4_cluster_kernel(const CParams p)
{
    constexpr bool DOTS = MODE == W4Mode::A8_DOTS;
    constexpr bool A16 = MODE == W4Mode::A16;
    constexpr int TB = CMP ? CMP_TILE_BYTES : TILE_BYTES;
    constexpr int SB = WARPS * TB;  // one stage: the 8 tiles of a super-block
    const int R = p.R;

    extern __shared__ __align__(128) uint8_t smem[];
    const CLayout L = c_layout(MP, p.smax, R, p.C, TB);
    uint8_t *xr = smem + L.xr, *xs = smem + L.xs, *xg = smem + L.xg;
    float *red = reinterpret_cast<float *>(smem + L.red);
    uint32_t *rowmax = reinterpret_cast<uint32_t *>(smem + L.rowmax);
    const uint32_t full0 = smem_addr(smem + L.bars), empty0 = full0 + 8 * R;
    const uint32_t recv_bar = empty0 + 8 * R;  // rank 0: the other ranks' sums have landed
    const uint32_t max_bar = recv_bar + 8;     // ROW: the other ranks' row maxima have landed
    const uint32_t zrow = smem_addr(smem + L.zero);

    // hardware warp 0 produces (the schedulers favour low warp ids); 1..8
    // are the consumers of row tiles 0..7
    const int hw_warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warp = hw_warp == 0 ? WARPS : hw_warp - 1;
    const uint32_t rank = cluster_rank();
    const int g = blockIdx.y;
    const int b0 = (int)((long long)rank * p.KB / p.C);
    const int S = (int)((long long)(rank + 1) * p.KB / p.C) - b0;  // stages of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, WARPS);
        }
        mbar_init(recv_bar, 1);
        mbar_init(max_bar, 1);
        // the bytes the other ranks will send (the phase completes when they
        // have all landed; a rank's bytes may arrive before this)
        if (!DOTS && rank == 0)
            mbar_arrive_expect_tx(recv_bar, (uint32_t)((p.C - 1) * GROUP_ROWS * MP * 4));
        if (ROW)
            mbar_arrive_expect_tx(max_bar, (uint32_t)((p.C - 1) * 32));
        fence_barrier_init();
    }
    // zero: the 16-byte zero row, this rank's row maxima, and the activation
    // rows m >= M of every stage (read by the MMAs, never stored)
    if (threadIdx.x < 8)
        rowmax[8 * rank + threadIdx.x] = 0u;  // this rank's slot
    if (threadIdx.x == 8)
        *reinterpret_cast<uint4 *>(smem + L.zero) = make_uint4(0u, 0u, 0u, 0u);
    {
        const int pad = MP - p.M;
        const int xper = pad * (XROW / 16), sper = pad * (SROW / 16);
        const int per = xper + 2 * sper;
        for (int i = threadIdx.x; i < S * per; i += THREADS) {
            const int s = i / per, rem = i % per;
            uint8_t *dst;
            if (rem < xper)
                dst = xr + (s * MP + p.M + rem / (XROW / 16)) * XROW + (rem % (XROW / 16)) * 16;
            else if (rem < xper + sper)
                dst = xs + (s * MP + p.M + (rem - xper) / 2) * SROW + ((rem - xper) % 2) * 16;
            else
                dst = xg + (s * MP + p.M + (rem - xper - sper) / 2) * SROW +
                      ((rem - xper - sper) % 2) * 16;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __syncthreads();
    cluster_arrive_relaxed();  // every CTA's barriers are initialised (waited on below)
    if (threadIdx.x == 0)
        W4Q_STAMP(20);
    pdl_launch_dependents();  // the next kernel on the stream may launch and prefetch

    // -------------------------------------------- weight prefetch (no wait)
    const uint8_t *wsrc = p.packed + ((size_t)g * p.KB + b0) * SB;
    int issued = 0;
    const int pro = S < R ? S : R;
    if (warp == WARPS && lane == 0) {
        const uint64_t pol = policy_evict_first();
        for (int i = 0; i < pro; ++i) {
            mbar_arrive_expect_tx(full0 + 8 * i, (uint32_t)SB);
            bulk_g2s(smem_addr(smem + L.ring + i * SB), wsrc + (size_t)i * SB, SB, full0 + 8 * i,
                     pol);
        }
        issued = pro;
    }

    // ------------------------------------- the slice's activation operand
    pdl_wait();  // x may come from the kernel launched before this one
    if (threadIdx.x == 0)
        W4Q_STAMP(21);
    if constexpr (A16) {
        for (int s = hw_warp; s < S; s += WARPS + 1) {
            uint4 raw[MP];
            load_stage_a16<MP>(p.x, p.M, p.K, b0 + s, lane, raw);
            prep_stage_a16<MP>(raw, p.M, lane, xr + s * MP * XROW, xs + s * MP * SROW,
                               xg + s * MP * SROW);
        }
    } else {
        float arow[MP];
#pragma unroll
        for (int m = 0; m < MP; ++m)
            arow[m] = 0.f;
        if constexpr (ROW) {
            // pass 1: the raw slice into the x' rows, and this CTA's max |x| per row
            for (int s = hw_warp; s < S; s += WARPS + 1) {
                uint4 raw[MP];
                load_stage_a16<MP>(p.x, p.M, p.K, b0 + s, lane, raw);
#pragma unroll
                for (int m = 0; m < MP; ++m) {
                    uint32_t h = __vmaxu2(__vmaxu2(raw[m].x & 0x7FFF7FFFu, raw[m].y & 0x7FFF7FFFu),
                                          __vmaxu2(raw[m].z & 0x7FFF7FFFu, raw[m].w & 0x7FFF7FFFu));
                    h = max(h & 0xFFFFu, h >> 16);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
                    if (m < p.M) {
                        *reinterpret_cast<uint4 *>(xr + (s * MP + m) * XROW + 16 * lane) = raw[m];
                        if (lane == 0)
                            atomicMax(&rowmax[8 * rank + m], h);
                    }
                }
            }
            __syncthreads();  // this CTA's slice maxima are complete
            cluster_wait();   // every CTA's barriers are initialised
            // send them into slot `rank` of every other CTA's row maxima
            if (threadIdx.x < p.C && threadIdx.x != rank) {
                const uint32_t *own = rowmax + 8 * rank;
                const uint32_t dst = peer_addr(smem_addr(own), threadIdx.x);
                const uint32_t bar = peer_addr(max_bar, threadIdx.x);
                st_async_v4(dst, make_uint4(own[0], own[1], own[2], own[3]), bar);
                st_async_v4(dst + 16, make_uint4(own[4], own[5], own[6], own[7]), bar);
            }
            if (p.C > 1 && !mbar_wait_sleep(max_bar, 0u))
                report_error(p.err, ERR_FULL_WAIT);
            // the row's max over the C slices (magnitudes order as bf16 bits)
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                uint32_t h = 0u;
                for (int c = 0; c < p.C; ++c)
                    h = max(h, rowmax[8 * c + m]);
                arow[m] = __uint_as_float(h << 16);
            }
        }
        for (int s = hw_warp; s < S; s += WARPS + 1) {
            uint4 raw[MP];
            if constexpr (ROW) {
#pragma unroll
                for (int m = 0; m < MP; ++m)
                    raw[m] = m < p.M ? *reinterpret_cast<const uint4 *>(xr + (s * MP + m) * XROW +
                                                                        16 * lane)
                                     : make_uint4(0u, 0u, 0u, 0u);
                __syncwarp();  // every lane has read its raw chunk before any is overwritten
            } else {
                load_stage_a16<MP>(p.x, p.M, p.K, b0 + s, lane, raw);
            }
            prep_stage_a8<MP, ROW>(raw, p.M, lane, arow, xr + s * MP * XROW, xs + s * MP * SROW,
                                   xg + s * MP * SROW);
        }
    }
    __syncthreads();  // the slice's activation operand is complete
    if (threadIdx.x == 0)
        W4Q_STAMP(22);

    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    const int tile = g * WARPS + warp;
    if (warp == WARPS) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = pro; i < S; ++i) {
                const int slot = i % R;
                if (!W4Q_RING_WAIT(empty0 + 8 * slot, (uint32_t)(i / R - 1) & 1)) {
                    report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * slot, (uint32_t)SB);
                bulk_g2s(smem_addr(smem + L.ring + slot * SB), wsrc + (size_t)i * SB, SB,
                         full0 + 8 * slot, pol);
                issued = i + 1;
            }
        }
    } else {
        // ----------------------------------------------------- consumers
        // compact metadata: this lane's row steps (ds of rows r, r + 8, then
        // dz), stored after the tiles of the packed buffer
        float rs[4] = {1.f, 1.f, 1.f, 1.f};
        if constexpr (CMP) {
            const int n = (g * WARPS + warp) * 16 + (lane >> 2);
            const __half *st = reinterpret_cast<const __half *>(
                p.packed + (size_t)p.G * WARPS * p.KB * CMP_TILE_BYTES);
            rs[0] = __half2float(st[2 * n]);
            rs[1] = __half2float(st[2 * (n + 8)]);
            rs[2] = __half2float(st[2 * n + 1]);
            rs[3] = __half2float(st[2 * (n + 8) + 1]);
        }
        auto stage = [&](int i) {
            const int slot = i % R;
            if (tile < p.T) {
                const uint32_t wbase = smem_addr(smem + L.ring + slot * SB + warp * TB);
                const uint32_t xb = smem_addr(xr + i * MP * XROW);
                const uint32_t sb = smem_addr(xs + i * MP * SROW);
                const uint32_t gb = smem_addr(xg + i * MP * SROW);
                if constexpr (MP < 8)
                    compute_stage_packed<MP, DOTS, !A16, A16, CMP, 1>(wbase, xb, sb, gb, zrow, lane,
                                                                   acc, p, tile, b0 + i, rs);
                else
                    compute_stage<1, DOTS, !A16, A16, CMP>(wbase, xb, sb, gb, lane, acc, p, tile,
                                                           b0 + i, rs);
            }
        };
        auto ready = [&](int i) -> bool {
            const bool got = W4Q_RING_WAIT(full0 + 8 * (i % R), (uint32_t)(i / R) & 1);
            if (!__all_sync(0xffffffffu, got)) {  // the whole warp leaves together
                if (lane == 0)
                    report_error(p.err, ERR_FULL_WAIT);
                return false;
            }
            return true;
        };
        auto release = [&](int i) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * (i % R));
        };
        if constexpr (MP <= W4Q_CL_PAIR_MP) {
            // Two stages at a time when both are in the ring, so that their
            // MMA chains interleave (measured at M = 1: 18.1 -> 17.6 us on
            // 6656 x 19968; at MP = 4 the doubled register state made it
            // slower).
            int i = 0;
            for (; i + 1 < S; i += 2) {
                if (!ready(i) || !ready(i + 1)) {
                    i = S + 1;
                    break;
                }
                stage(i);
                stage(i + 1);
                release(i);
                release(i + 1);
            }
            if (i == S - 1 && ready(i)) {
                stage(i);
                release(i);
            }
        } else {
            for (int i = 0; i < S; ++i) {
                if (!ready(i))
                    break;
                stage(i);
                release(i);
            }
        }
        if (!DOTS) {
            // add the accumulator slots (lanes of one row hold other groups of
            // the same outputs), then park this warp's 16 x MP sums
            const int r = lane >> 2, c2 = 2 * (lane & 3);
            if constexpr (MP < 8) {
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
            if (c2 < MP) {  // slot 0 of the columns: (row, m) = (r or r + 8, c2 + (e & 1))
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = c2 + (e & 1);
                    if (MP == 1 && (e & 1))
                        continue;
                    if (m < MP)
                        red[(warp * 16 + r + 8 * (e >> 1)) * MP + m] = acc[0][e];
                }
            }
        }
    }

    if (threadIdx.x == 32)
        W4Q_STAMP(23);
    // ---------------------------------------------- split-K over the cluster
    if constexpr (!ROW)
        cluster_wait();  // every CTA's barriers are initialised (ROW waited above)
    if (!DOTS) {
        __syncthreads();  // this CTA's 128 x MP sums are complete
        const int n4 = GROUP_ROWS * MP / 4;  // 16-byte pieces of them
        if (rank != 0) {
            // send them into slot rank - 1 of rank 0's received sums, and go
            const uint32_t dst = peer_addr(smem_addr(smem + L.recv) + (rank - 1) * (n4 * 16), 0u);
            const uint32_t bar = peer_addr(recv_bar, 0u);
            for (int i = threadIdx.x; i < n4; i += THREADS)
                st_async_v4(dst + 16 * i, reinterpret_cast<const uint4 *>(red)[i], bar);
        } else {
            if (p.C > 1 && !mbar_wait_sleep(recv_bar, 0u))
                report_error(p.err, ERR_FULL_WAIT);
            const float *recv = reinterpret_cast<const float *>(smem + L.recv);
            for (int t = threadIdx.x; t < GROUP_ROWS * p.M; t += THREADS) {
                const int row = t % GROUP_ROWS, m = t / GROUP_ROWS;
                float v = red[row * MP + m];
                for (int c = 1; c < p.C; ++c)
                    v += recv[(c - 1) * GROUP_ROWS * MP + row * MP + m];
                const int n = g * GROUP_ROWS + row;
                if (n < p.N)
                    p.out[(size_t)m * p.N + n] = __float2bfloat16_rn(v);
            }
        }
    }

    if (threadIdx.x == 0)
        W4Q_STAMP(25);
    // Drain: every issued stage's copy must have landed before the shared
    // memory goes away (only the error path can leave one pending).
    if (warp == WARPS && lane == 0) {
        for (int s = 0; s < R && s < issued; ++s) {
            const int last_use = (issued - 1 - s) / R;
            if (!W4Q_RING_WAIT(full0 + 8 * s, (uint32_t)last_use & 1)) {
                report_error(p.err, ERR_DRAIN_WAIT);
                break;
            }
        }
    }
}

template <W4Mode MODE, bool ROW, int MP, bool CMP>
cudaError_t launch_t(const CParams &p, int smem, cudaStream_t stream)
{
    auto fn = w4_cluster_kernel<MODE, ROW, MP, CMP>;
    // the dynamic shared-memory opt-in, once per device (a bit per device)
    static std::atomic<unsigned long long> opted_in{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit == 0 || !(opted_in.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, CTA_SMEM_MAX);
        if (e != cudaSuccess)
            return e;
        opted_in.fetch_or(bit, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.C, (unsigned)p.G);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <W4Mode MODE, bool ROW, bool CMP = false>
cudaError_t dispatch_mp(const CParams &p, int mp, int smem, cudaStream_t stream)
{
    switch (mp) {
    case 1: return launch_t<MODE, ROW, 1, CMP>(p, smem, stream);
    case 2: return launch_t<MODE, ROW, 2, CMP>(p, smem, stream);
    case 4: return launch_t<MODE, ROW, 4, CMP>(p, smem, stream);
    default: return launch_t<MODE, ROW, 8, CMP>(p, smem, stream);
    }
}

int mp_of(int M) { return M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8)); }

}  // namespace

// The weight-ring depth for these sizes (4 stages, fewer where the slice's
// activation operand needs the room), or 0 when even 2 do not fit in the
// shared memory of one of two CTAs per SM.
int w4_cluster_ring(int M, int KB, int C)
{
    if (C < 1 || C > MAX_CLUSTER || C > KB || M < 1 || M > 8)
        return 0;
    const int smax = (KB + C - 1) / C;
    for (int R = 4; R >= 2; --R)
        if (c_layout(mp_of(M), smax, R, C, TILE_BYTES).total <= CTA_SMEM_MAX)
            return R;
    return 0;
}

cudaError_t launch_w4_cluster(const W4Plan &plan, W4Mode mode, bool act_row, const void *x,
                              const void *packed, void *out, int32_t *dots, unsigned *err,
                              cudaStream_t stream)
{
    const bool cmp = plan.compact;
    CParams p;
    p.packed = static_cast<const uint8_t *>(packed);
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.dots = dots;
    p.err = err;
    p.M = plan.M;
    p.N = plan.N;
    p.K = plan.K;
    p.KB = plan.KB;
    p.T = plan.T;
    p.G = plan.G;
    p.C = plan.cluster;
    p.smax = (plan.KB + plan.cluster - 1) / plan.cluster;
    p.R = w4_cluster_ring(plan.M, plan.KB, plan.cluster);
    if (p.R == 0)
        return cudaErrorInvalidValue;
    const int mp = mp_of(plan.M);
    const int smem = c_layout(mp, p.smax, p.R, p.C, cmp ? CMP_TILE_BYTES : TILE_BYTES).total;
    if (cmp)  // compact metadata: W4A16 only
        return mode == W4Mode::A16 ? dispatch_mp<W4Mode::A16, false, true>(p, mp, smem, stream)
                                   : cudaErrorInvalidValue;
    if (mode == W4Mode::A16)
        return dispatch_mp<W4Mode::A16, false>(p, mp, smem, stream);
    if (mode == W4Mode::A8)
        return act_row ? dispatch_mp<W4Mode::A8, true>(p, mp, smem, stream)
                       : dispatch_mp<W4Mode::A8, false>(p, mp, smem, stream);
    return act_row ? dispatch_mp<W4Mode::A8_DOTS, true>(p, mp, smem, stream)
                   : dispatch_mp<W4Mode::A8_DOTS, false>(p, mp, smem, stream);
}

}  // namespace w4q

W4Q_STAMP_READER(w4q_timeline_read_cluster)
