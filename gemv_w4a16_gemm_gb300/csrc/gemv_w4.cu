// gemv_w4.cu -- decode-sized W4A16 / W4A8 linear layer on sm_103a.
//
//   out[M,N] = x[M,K] . dequant(Wq)[N,K]^T,   dequant(q) = (q - z) * s
//
// ("test_int4_quantized_gemm.py": the dequant + F.linear reference, the W4A8
// bucket kernels and the W4A16 tile kernels; this is a new design for GB300,
// not their code.)
//
// Design (one CTA = 8 consumer warps + 1 producer warp):
//  * The weight is read once, as whole 2432-byte packed tiles (16 rows x 256
//    K, codes + scales + zeros), by 1-D bulk copies (TMA engine) into a
//    multi-stage shared-memory ring guarded by mbarriers; the activation
//    chunk of the same 256 K rides along in the same stage.  Weights carry
//    an L2 evict-first hint, activations evict-last.
//  * Consumer warp w owns row tile w of the CTA's 128-row tile group.  A
//    lane's 16 bytes of a sub-block are exactly its four bf16 A fragments of
//    four m16n8k16 MMAs (the layout is built for this), so dequant is two
//    ALU ops per pair of codes: LOP3 puts a nibble into the mantissa of
//    bf16 128.0, and one packed bf16 subtract of (128 + z) leaves the exact
//    integer q - z.  The tensor core then sums (q - z) * x over each group
//    of 32 exactly; the fp32 group sum is scaled by s and accumulated
//    (M <= 16).  For M > 16 the scaled weight (q - z) * s is rounded to bf16
//    once and the MMA accumulates over all of K (per-group fp32 scaling
//    would cost more ALU than the tensor core saves).
//  * W4A8: activations are int8 values held as exact bf16 integers, so the
//    per-group MMA sum (|D| <= 60960 < 2^24) is the exact integer dot; the
//    same kernel then scales by s in fp32 and by the row scale at the end.
//  * Work partition: units (tile group, 256-K super-block) are split into
//    P contiguous ranges, one per CTA (balanced "stream-K" ranges over all
//    SM slots by default, or a fixed split of each group's K).  A group that
//    one CTA covers entirely is written directly; the other groups write
//    fp32 partials that a fixup kernel sums in CTA order (deterministic, no
//    atomics).  The fixup is launched with programmatic dependent launch.
//  * Every wait is bounded (one second of %globaltimer); on expiry the
//    kernel sets a bit in the error word, drains its copies and returns.
#include "common.cuh"
#include "kernels.h"

namespace w4q {

namespace {

constexpr int TILE_BYTES = 2432;
constexpr int WARPS = 8;                   // consumer warps = row tiles per tile group
constexpr int THREADS = (WARPS + 1) * 32;  // + one producer warp
constexpr int XROW = 512 + 16;             // one activation row's 256-K chunk, padded

struct Params {
    const uint8_t *packed;
    const __nv_bfloat16 *x;  // bf16 [M][K]; W4A8: the int8 activations as bf16
    const float *sx;         // W4A8 per-row activation scales
    __nv_bfloat16 *out;      // bf16 [M][N]
    int32_t *dots;           // group-dot export: int32 [M][N][K/32]
    float *partial;          // fp32 [P][2][M][128]
    unsigned *err;
    int M, N, K, KB, T, G, P, split;
    long long U;
};

__host__ __device__ __forceinline__ long long range_begin(const Params &p, int c)
{
    if (p.split == 0)
        return (long long)c * p.U / p.P;
    const int g = c / p.split, j = c % p.split;
    return (long long)g * p.KB + (long long)j * p.KB / p.split;
}

template <int NB>
__host__ __device__ constexpr int stages_for()
{
    return NB <= 2 ? 4 : (NB == 4 ? 3 : 4);
}

template <int NB>
__host__ __device__ constexpr int smem_for()
{
    return stages_for<NB>() * (WARPS * TILE_BYTES + NB * 8 * XROW) + 2 * stages_for<NB>() * 8;
}

// One stage = one 16 x 256 tile for this warp: 4 sub-blocks of 64 K (two
// groups each), 4 k16 steps per sub-block.
template <int NB, bool FOLD, bool DOTS>
__device__ __forceinline__ void compute_stage(uint32_t wbase, uint32_t xbase, int lane,
                                              float (&acc)[NB][4], const Params &p, int tile,
                                              int b)
{
    const int r = lane >> 2;
    const uint4 sc0 = lds128(wbase + 2048 + 16 * r);
    const uint4 sc1 = lds128(wbase + 2048 + 128 + 16 * r);
    const uint4 zz = lds128(wbase + 2304 + 16 * r);
    const uint32_t scw[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
    const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
    // ldmatrix.x4 row addresses: matrix lane>>3 = (step +lane>>4, k half (lane>>3)&1)
    const uint32_t xlane = xbase + (lane & 7) * XROW + 32 * (lane >> 4) + 16 * ((lane >> 3) & 1);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

#pragma unroll
    for (int sbk = 0; sbk < 4; ++sbk) {
        const uint4 wq = lds128(wbase + 512 * sbk + 16 * lane);
        const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
        uint32_t bf[NB][4][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const uint32_t a = xlane + nb * 8 * XROW + 32 * (4 * sbk);
            ldmatrix_x4(a, bf[nb][0][0], bf[nb][0][1], bf[nb][1][0], bf[nb][1][1]);
            ldmatrix_x4(a + 64, bf[nb][2][0], bf[nb][2][1], bf[nb][3][0], bf[nb][3][1]);
        }
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            const int g = 2 * sbk + gi;
            // (128 + z) in both bf16 halves, rows r and r + 8
            const uint32_t zsrc = zw[g >> 1];
            const uint32_t zb = (uint32_t)((2 * g) & 3);
            const uint32_t zr = prmt(zsrc, 0x43u, 0x4040u + 0x0101u * zb);
            const uint32_t zr8 = prmt(zsrc, 0x43u, 0x4040u + 0x0101u * (zb + 1));
            const uint32_t sp = scw[g];
            uint32_t s2r = 0, s2r8 = 0;
            if (FOLD) {
                s2r = prmt(sp, sp, 0x1010u);
                s2r8 = prmt(sp, sp, 0x3232u);
            }
            float d[NB][4];
#pragma unroll
            for (int st = 0; st < 2; ++st) {
                const uint32_t w = wv[2 * gi + st];
                uint32_t a[4];
                a[0] = bf16x2_sub(and_or(w, 0x000F000Fu, 0x43004300u), zr);
                a[1] = bf16x2_sub(and_or(w >> 4, 0x000F000Fu, 0x43004300u), zr8);
                a[2] = bf16x2_sub(and_or(w >> 8, 0x000F000Fu, 0x43004300u), zr);
                a[3] = bf16x2_sub(and_or(w >> 12, 0x000F000Fu, 0x43004300u), zr8);
                if (FOLD) {
                    a[0] = bf16x2_mul(a[0], s2r);
                    a[1] = bf16x2_mul(a[1], s2r8);
                    a[2] = bf16x2_mul(a[2], s2r);
                    a[3] = bf16x2_mul(a[3], s2r8);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
                        mma_bf16(acc[nb], a, bf[nb][2 * gi + st][0], bf[nb][2 * gi + st][1],
                                 acc[nb]);
                } else {
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        if (st == 0)
                            mma_bf16(d[nb], a, bf[nb][0 + 2 * gi][0], bf[nb][0 + 2 * gi][1], zero4);
                        else
                            mma_bf16(d[nb], a, bf[nb][1 + 2 * gi][0], bf[nb][1 + 2 * gi][1], d[nb]);
                    }
                }
            }
            if (!FOLD) {
                if (DOTS) {
                    const int c2 = 2 * (lane & 3);
                    const int G = p.K / 32, gg = b * 8 + g;
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int m = nb * 8 + c2 + (e & 1);
                            const int n = tile * 16 + r + 8 * (e >> 1);
                            if (m < p.M && n < p.N)
                                p.dots[((size_t)m * p.N + n) * G + gg] = (int32_t)d[nb][e];
                        }
                } else {
                    const float sr = bf16lo_to_f32(sp), sr8 = bf16hi_to_f32(sp);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        acc[nb][0] = fmaf(sr, d[nb][0], acc[nb][0]);
                        acc[nb][1] = fmaf(sr, d[nb][1], acc[nb][1]);
                        acc[nb][2] = fmaf(sr8, d[nb][2], acc[nb][2]);
                        acc[nb][3] = fmaf(sr8, d[nb][3], acc[nb][3]);
                    }
                }
            }
        }
    }
}

// The dequantized weight is folded into bf16 for W4A16 at M > 16 (NB >= 4).
template <int NB, W4Mode MODE>
__host__ __device__ constexpr bool fold_for()
{
    return MODE == W4Mode::A16 && NB >= 4;
}

template <int NB, W4Mode MODE>
__global__ void __launch_bounds__(THREADS, (NB <= 4 ? 2 : 1)) w4_kernel(const Params p)
{
    constexpr bool FOLD = fold_for<NB, MODE>();
    constexpr bool A8 = MODE != W4Mode::A16;
    constexpr bool DOTS = MODE == W4Mode::A8_DOTS;
    constexpr int STAGES = stages_for<NB>();
    constexpr int WST = WARPS * TILE_BYTES;
    constexpr int XST = NB * 8 * XROW;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sw = smem;
    uint8_t *sxb = smem + STAGES * WST;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sxb + STAGES * XST);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const long long u0 = range_begin(p, c), u1 = range_begin(p, c + 1);
    const int n_iter = (int)(u1 - u0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, WARPS);
        }
        fence_barrier_init();
    }
    {   // activation rows m >= M of every stage stay zero (never copied into)
        const int pad_rows = NB * 8 - p.M;
        const int per_stage = pad_rows * (XROW / 16);
        for (int i = threadIdx.x; i < STAGES * per_stage; i += THREADS) {
            const int s = i / per_stage, rem = i % per_stage;
            const int row = p.M + rem / (XROW / 16), col = rem % (XROW / 16);
            *reinterpret_cast<uint4 *>(sxb + s * XST + row * XROW + col * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __syncthreads();

    int issued = 0;
    if (warp == WARPS) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
            auto tiles_of = [&](int i) {
                const int g = (int)((u0 + i) / p.KB);
                const int nt = p.T - g * WARPS;
                return nt < WARPS ? nt : WARPS;
            };
            auto issue_w = [&](int i) {
                const long long u = u0 + i;
                const int g = (int)(u / p.KB), b = (int)(u % p.KB);
                const int slot = i % STAGES, nt = tiles_of(i);
                const uint32_t bar = full0 + 8 * slot;
                mbar_arrive_expect_tx(bar, (uint32_t)(nt * TILE_BYTES + p.M * 512));
                for (int w = 0; w < nt; ++w)
                    bulk_g2s(smem_addr(sw + slot * WST + w * TILE_BYTES),
                             p.packed + ((size_t)(g * WARPS + w) * p.KB + b) * TILE_BYTES,
                             TILE_BYTES, bar, pol_w);
            };
            auto issue_x = [&](int i) {
                const int b = (int)((u0 + i) % p.KB);
                const int slot = i % STAGES;
                const uint32_t bar = full0 + 8 * slot;
                for (int m = 0; m < p.M; ++m)
                    bulk_g2s(smem_addr(sxb + slot * XST + m * XROW),
                             p.x + (size_t)m * p.K + (size_t)b * 256, 512, bar, pol_x);
            };
            const int pro = n_iter < STAGES ? n_iter : STAGES;
            for (int i = 0; i < pro; ++i)
                issue_w(i);
            pdl_wait();  // activations may come from the kernel launched just before
            for (int i = 0; i < pro; ++i)
                issue_x(i);
            issued = pro;
            for (int i = pro; i < n_iter; ++i) {
                const int slot = i % STAGES;
                const uint32_t use = (uint32_t)(i / STAGES);
                if (!mbar_wait_bounded(empty0 + 8 * slot, (use - 1) & 1)) {
                    report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                issue_w(i);
                issue_x(i);
                issued = i + 1;
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        pdl_wait();
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
            acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
        const int g_first = (int)(u0 / p.KB);
        int cur_g = g_first;
        bool ok = true;

        auto flush = [&](int g) {
            if (DOTS)
                return;
            const int tile = g * WARPS + warp;
            if (tile >= p.T)
                return;
            const long long gb = (long long)g * p.KB, ge = gb + p.KB;
            const bool complete = gb >= u0 && ge <= u1;
            const int slot = (g == g_first) ? 0 : 1;
            const int r = lane >> 2, c2 = 2 * (lane & 3);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = r + 8 * (e >> 1);
                    const int m = nb * 8 + c2 + (e & 1);
                    const int n = tile * 16 + row;
                    if (m < p.M && n < p.N) {
                        if (complete) {
                            const float v = A8 ? acc[nb][e] * p.sx[m] : acc[nb][e];
                            p.out[(size_t)m * p.N + n] = __float2bfloat16_rn(v);
                        } else {
                            p.partial[((size_t)(c * 2 + slot) * p.M + m) * 128 + warp * 16 + row] =
                                acc[nb][e];
                        }
                    }
                }
        };

        for (int i = 0; i < n_iter; ++i) {
            const long long u = u0 + i;
            const int g = (int)(u / p.KB), b = (int)(u % p.KB);
            if (g != cur_g) {
                flush(cur_g);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb)
                    acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
                cur_g = g;
            }
            const int slot = i % STAGES;
            if (!mbar_wait_bounded(full0 + 8 * slot, (uint32_t)(i / STAGES) & 1)) {
                report_error(p.err, ERR_FULL_WAIT);
                ok = false;
                break;
            }
            const int tile = g * WARPS + warp;
            if (tile < p.T)
                compute_stage<NB, FOLD, DOTS>(smem_addr(sw + slot * WST + warp * TILE_BYTES),
                                              smem_addr(sxb + slot * XST), lane, acc, p, tile, b);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * slot);
        }
        if (ok && n_iter > 0)
            flush(cur_g);
    }

    pdl_launch_dependents();
    __syncthreads();
    // Drain: every issued stage's copies must have landed before the CTA's
    // shared memory goes away (only the error path can leave some pending).
    if (warp == WARPS && lane == 0) {
        for (int s = 0; s < STAGES && s < issued; ++s) {
            const int last_use = (issued - 1 - s) / STAGES;
            if (!mbar_wait_bounded(full0 + 8 * s, (uint32_t)last_use & 1)) {
                report_error(p.err, ERR_DRAIN_WAIT);
                break;
            }
        }
    }
}

// Sums the partials of every tile group that several CTAs share, in CTA
// order, and writes its bf16 outputs.
template <bool A8>
__global__ void __launch_bounds__(256) w4_fixup_kernel(const Params p)
{
    pdl_wait();
    const int g = blockIdx.x;
    const long long gb = (long long)g * p.KB, ge = gb + p.KB;
    int lo = 0, hi = p.P - 1;  // the CTA holding unit gb: largest c with begin(c) <= gb
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (range_begin(p, mid) <= gb)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int c_first = lo;
    if (range_begin(p, c_first + 1) >= ge)
        return;  // the whole group lies in one CTA's range: written directly
    for (int i = threadIdx.x; i < p.M * 128; i += blockDim.x) {
        const int m = i / 128, row = i % 128;
        const int n = g * 128 + row;
        if (n >= p.N)
            continue;
        float v = 0.f;
        for (int c = c_first; c < p.P && range_begin(p, c) < ge; ++c) {
            const int slot = (range_begin(p, c) / p.KB == g) ? 0 : 1;
            v += p.partial[((size_t)(c * 2 + slot) * p.M + m) * 128 + row];
        }
        if (A8)
            v *= p.sx[m];
        p.out[(size_t)m * p.N + n] = __float2bfloat16_rn(v);
    }
}

// W4A8 activation quantizer: per row, sx = fp32(max|x| / 127),
// xq = clamp(rint(fp32(x / sx)), -127, 127), 0 for an all-zero row.
// OUT_BF16 writes xq as exact bf16 integers (the MMA operand); otherwise int8.
template <bool OUT_BF16>
__global__ void __launch_bounds__(512) act_quant_kernel(const __nv_bfloat16 *__restrict__ x,
                                                        int K, void *__restrict__ xq,
                                                        float *__restrict__ sx)
{
    pdl_launch_dependents();
    __shared__ float red[16];
    const int m = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
    const int n8 = K / 8;
    float a = 0.f;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            a = fmaxf(a, fmaxf(fabsf(bf16lo_to_f32(w[j])), fabsf(bf16hi_to_f32(w[j]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = a;
    __syncthreads();
    a = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        a = fmaxf(a, red[i]);
    const float s = __fdiv_rn(a, 127.0f);
    if (threadIdx.x == 0)
        sx[m] = s;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        const uint4 v = row[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float q[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            q[2 * j] = bf16lo_to_f32(w[j]);
            q[2 * j + 1] = bf16hi_to_f32(w[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            q[j] = (a == 0.f) ? 0.f : fminf(fmaxf(rintf(__fdiv_rn(q[j], s)), -127.f), 127.f);
        if (OUT_BF16) {
            uint4 o;
            o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[0])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[1])) << 16);
            o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[2])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[3])) << 16);
            o.z = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[4])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[5])) << 16);
            o.w = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[6])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(q[7])) << 16);
            reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(xq) + (size_t)m * K)[i] = o;
        } else {
            uint2 o;
            o.x = (uint32_t)(uint8_t)(int8_t)q[0] | ((uint32_t)(uint8_t)(int8_t)q[1] << 8) |
                  ((uint32_t)(uint8_t)(int8_t)q[2] << 16) | ((uint32_t)(uint8_t)(int8_t)q[3] << 24);
            o.y = (uint32_t)(uint8_t)(int8_t)q[4] | ((uint32_t)(uint8_t)(int8_t)q[5] << 8) |
                  ((uint32_t)(uint8_t)(int8_t)q[6] << 16) | ((uint32_t)(uint8_t)(int8_t)q[7] << 24);
            reinterpret_cast<uint2 *>(static_cast<int8_t *>(xq) + (size_t)m * K)[i] = o;
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
        auto fn = w4_kernel<NB, MODE>;
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_for<NB>());
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, THREADS, smem_for<NB>()) !=
                cudaSuccess ||
            n < 1)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

int nb_for(int M) { return M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8)); }

template <W4Mode MODE>
int ctas_per_sm_for(int NB, int dev)
{
    switch (NB) {
    case 1: return ctas_per_sm<1, MODE>(dev);
    case 2: return ctas_per_sm<2, MODE>(dev);
    case 4: return ctas_per_sm<4, MODE>(dev);
    default: return ctas_per_sm<8, MODE>(dev);
    }
}

template <int NB, W4Mode MODE>
cudaError_t launch_main(const Params &p, cudaStream_t stream, bool pdl)
{
    auto fn = w4_kernel<NB, MODE>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_for<NB>());
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem_for<NB>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <W4Mode MODE>
cudaError_t dispatch_main(const W4Plan &plan, const Params &p, cudaStream_t stream, bool pdl)
{
    switch (plan.NB) {
    case 1: return launch_main<1, MODE>(p, stream, pdl);
    case 2: return launch_main<2, MODE>(p, stream, pdl);
    case 4: return launch_main<4, MODE>(p, stream, pdl);
    default: return launch_main<8, MODE>(p, stream, pdl);
    }
}

template <bool A8>
cudaError_t launch_fixup(const Params &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w4_fixup_kernel<A8>, p);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

bool w4_plan(int M, int N, int K, int split, int sm_count, W4Mode mode, W4Plan *plan)
{
    if (M < 1 || M > 64 || N < 1 || K < 256 || K % 256 != 0)
        return false;
    W4Plan pl = {};
    pl.M = M;
    pl.N = N;
    pl.K = K;
    pl.KB = K / 256;
    pl.T = (N + 15) / 16;
    pl.G = (pl.T + WARPS - 1) / WARPS;
    pl.NB = nb_for(M);
    pl.fold = (mode == W4Mode::A16) && M > 16;
    const long long U = (long long)pl.G * pl.KB;
    if (mode == W4Mode::A8_DOTS)
        split = 1;  // every unit is processed once; no accumulation across CTAs
    if (split < 0)
        split = 0;
    if (split >= 1) {
        if (split > pl.KB)
            return false;
        pl.split = split;
        pl.P = pl.G * split;
        pl.fixup = split > 1;
    } else {
        int dev = 0;
        cudaGetDevice(&dev);
        const int per_sm = (mode == W4Mode::A16) ? ctas_per_sm_for<W4Mode::A16>(pl.NB, dev)
                                                 : ctas_per_sm_for<W4Mode::A8>(pl.NB, dev);
        const long long slots = (long long)(sm_count > 0 ? sm_count : 1) * per_sm;
        pl.split = 0;
        pl.P = (int)(U < slots ? U : slots);
        pl.fixup = !(U % pl.P == 0 && (U / pl.P) % pl.KB == 0);
    }
    if (mode == W4Mode::A8_DOTS)
        pl.fixup = false;
    pl.partial_bytes = pl.fixup ? (size_t)pl.P * 2 * M * 128 * sizeof(float) : 0;
    *plan = pl;
    return true;
}

size_t w4_workspace_for(const W4Plan &plan, W4Mode mode)
{
    size_t bytes = plan.partial_bytes;
    if (mode != W4Mode::A16)
        bytes += align_up((size_t)plan.M * plan.K * 2, 256) + align_up((size_t)plan.M * 4, 256);
    return bytes;
}

cudaError_t launch_w4(const W4Plan &plan, W4Mode mode, const void *x, const void *packed,
                      void *out, int32_t *dots, void *workspace, unsigned *err,
                      cudaStream_t stream)
{
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
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e;
    if (mode == W4Mode::A16) {
        p.x = static_cast<const __nv_bfloat16 *>(x);
        p.partial = reinterpret_cast<float *>(ws);
        e = dispatch_main<W4Mode::A16>(plan, p, stream, false);
        if (e == cudaSuccess && plan.fixup)
            e = launch_fixup<false>(p, stream);
        return e;
    }
    __nv_bfloat16 *xq = reinterpret_cast<__nv_bfloat16 *>(ws);
    float *sx = reinterpret_cast<float *>(ws + align_up((size_t)plan.M * plan.K * 2, 256));
    p.x = xq;
    p.sx = sx;
    p.partial = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(sx) +
                                          align_up((size_t)plan.M * 4, 256));
    act_quant_kernel<true><<<plan.M, 512, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x),
                                                       plan.K, xq, sx);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (mode == W4Mode::A8_DOTS)
        return dispatch_main<W4Mode::A8_DOTS>(plan, p, stream, true);
    e = dispatch_main<W4Mode::A8>(plan, p, stream, true);
    if (e == cudaSuccess && plan.fixup)
        e = launch_fixup<true>(p, stream);
    return e;
}

cudaError_t launch_act_quant_i8(const void *x, int M, int K, int8_t *xq, float *sx,
                                cudaStream_t stream)
{
    act_quant_kernel<false><<<M, 512, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), K, xq,
                                                   sx);
    return cudaGetLastError();
}

}  // namespace w4q
