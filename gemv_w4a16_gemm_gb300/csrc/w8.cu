// w8.cu -- int8 weight-only GEMV on sm_103a:
//
//   out[m,n] = bf16_RN( fp32( sum_k x[m,k] * W[n,k] ) * scales[n] )
//
// ("gpt-fast issue #114": WeightOnlyInt8Linear.forward computes
// F.linear(x, W.to(bf16)) * scales; its fused Inductor reduction streams W
// once, keeps x resident, accumulates in fp32 and applies the scale at the
// end.  This kernel is a new GB300 design with the same arithmetic.)
//
// Design (one CTA per SM and call: 16 consumer warps + 1 producer warp):
//  * CTA c owns a contiguous range of whole rows; those rows are one
//    contiguous stretch of W, streamed through a shared-memory ring by 1-D
//    bulk copies (TMA engine, L2 evict-first), RW rows per stage (RW fixed
//    at compile time: 4 rows for K <= 8192 and M <= 2, else 2 rows).
//  * Lane (w, l) owns the 16-byte columns k = 16*(256*ch + 32*w + l) + 0..15
//    of every row; the matching activations sit in its registers as fp32
//    pairs for the whole kernel, so each weight byte costs one PRMT (it
//    lands in the mantissa of 2^23 + 128 + b) and, per two bytes, one packed
//    f32x2 subtraction and M packed f32x2 FMAs (8192 x 8192 at M = 1: 13.2
//    -> 12.5 us against the scalar FADD / FFMA form).
//  * The RW rows of a stage are unrolled, so their FMA chains (two per row
//    and m) are independent and overlap.  The warp reduces its RW x M sums
//    with a reduce-scatter (VP - 1 shuffles of data instead of 5 per value;
//    14.2 -> 13.2 us); each warp parks its per-row sums in shared memory,
//    and the CTA sums the 16 warp partials in a fixed order, multiplies by
//    the row scale and rounds once to bf16.
#include "common.cuh"
#include "kernels.h"
#include "timeline.cuh"

// Ring waits of this file: sleeping in mbarrier.try_wait (the default) or
// spinning on it.
#ifdef W4Q_SPIN_WAITS
#define W4Q_RING_WAIT mbar_wait_bounded
#else
#define W4Q_RING_WAIT mbar_wait_sleep
#endif

#ifndef W4Q_W8_RS
#define W4Q_W8_RS 1
#endif
#ifndef W4Q_W8_F2
#define W4Q_W8_F2 1
#endif

namespace w4q {

namespace {

// Packed fp32 pairs (f32x2: two independent correctly rounded operations
// per instruction); .x / lo is the low half.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

constexpr int CWARPS = 16;                  // consumer warps
constexpr int THREADS = (CWARPS + 1) * 32;  // + producer warp
constexpr int STAGE_BYTES = 32768;
constexpr int MAX_ROWS = 64;                // rows per CTA
constexpr int LANE_SPAN = CWARPS * 32 * 16; // bytes of a row covered per lane chunk

struct W8Params {
    const int8_t *W;
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *scales;
    __nv_bfloat16 *out;
    unsigned *err;
    int N, K, P;
};

// ST ring stages.  With 3 (M = 1) a CTA fits twice on an SM, so the next
// call's CTA on the same SM starts, and streams its first stages, while
// this one is still running; with 5 it holds a deeper ring alone.
template <int M, int CH, int RW, int ST>
__global__ void __launch_bounds__(THREADS, (ST <= 3 ? 2 : 1)) w8_kernel(const W8Params p)
{
    constexpr int STAGES = ST;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float *red = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);  // [CWARPS][MAX_ROWS][M]
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + CWARPS * MAX_ROWS * M);
    const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int r0 = (int)((long long)c * p.N / p.P), r1 = (int)((long long)(c + 1) * p.N / p.P);
    const int rows = r1 - r0;
    const int n_iter = (rows + RW - 1) / RW;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, CWARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        W4Q_STAMP(30);
    pdl_launch_dependents();  // the next call's preparation may launch and wait

    int issued = 0;
    if (warp == CWARPS) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < n_iter; ++i) {
                const int slot = i % STAGES;
                if (i >= STAGES &&
                    !W4Q_RING_WAIT(empty0 + 8 * slot, (uint32_t)(i / STAGES - 1) & 1)) {
                    report_error(p.err, ERR_EMPTY_WAIT);
                    break;
                }
                const int ra = r0 + i * RW;
                const int nr = (r1 - ra) < RW ? (r1 - ra) : RW;
                const uint32_t bytes = (uint32_t)nr * (uint32_t)p.K;
                mbar_arrive_expect_tx(full0 + 8 * slot, bytes);
                bulk_g2s(smem_addr(ring + slot * STAGE_BYTES), p.W + (size_t)ra * p.K, bytes,
                         full0 + 8 * slot, pol);
                issued = i + 1;
            }
        }
    } else {
        pdl_wait();  // x may come from the kernel launched before this one
        if (warp == 0 && lane == 0)
            W4Q_STAMP(31);
        // activations of this lane's columns, fp32, for the whole kernel
        float xr[CH][16][M];
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
            const int k0 = ch * LANE_SPAN + (warp * 32 + lane) * 16;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if (k0 < p.K) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)m * p.K + k0);
                    const uint4 v0 = src[0], v1 = src[1];
                    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        xr[ch][2 * e][m] = bf16lo_to_f32(w[e]);
                        xr[ch][2 * e + 1][m] = bf16hi_to_f32(w[e]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        xr[ch][e][m] = 0.f;
                }
            }
        }
#if W4Q_W8_F2
        uint64_t xp[CH][8][M];  // (x[2e], x[2e + 1]) pairs
#pragma unroll
        for (int ch = 0; ch < CH; ++ch)
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int m = 0; m < M; ++m)
                    xp[ch][e][m] = f32x2_pack(xr[ch][2 * e][m], xr[ch][2 * e + 1][m]);
#endif
        for (int i = 0; i < n_iter; ++i) {
            const int slot = i % STAGES;
            if (!W4Q_RING_WAIT(full0 + 8 * slot, (uint32_t)(i / STAGES) & 1)) {
                report_error(p.err, ERR_FULL_WAIT);
                break;
            }
            const int ra = r0 + i * RW;
            const int nr = (r1 - ra) < RW ? (r1 - ra) : RW;
            const uint32_t base = smem_addr(ring + slot * STAGE_BYTES);
            float acc[RW][M][2];
#if W4Q_W8_F2
            // Even and odd bytes of a word go to the two halves of one packed
            // fp32 pair: one f32x2 subtraction and one f32x2 FMA per two
            // weights, each half the same correctly rounded operation as the
            // scalar form (the accumulators see the same sums in the same order).
            uint64_t acc2[RW][M];
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m)
                    acc2[j][m] = 0ull;  // (+0, +0)
            const uint64_t bias2 = f32x2_pack(-8388736.0f, -8388736.0f);
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                if (j < nr) {
#pragma unroll
                    for (int ch = 0; ch < CH; ++ch) {
                        const int k0 = ch * LANE_SPAN + (warp * 32 + lane) * 16;
                        if (k0 < p.K) {
                            const uint4 v = lds128(base + (uint32_t)(j * p.K + k0));
                            const uint32_t wd[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u,
                                                    v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
                            for (int q = 0; q < 4; ++q)
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    // bytes [u, 0, 0, 0x4B]: 2^23 + u, u = b + 128
                                    const uint64_t f2 = f32x2_add(
                                        f32x2_pack(
                                            __uint_as_float(prmt(wd[q], 0x4B000000u, 0x7440u + 2 * h)),
                                            __uint_as_float(prmt(wd[q], 0x4B000000u, 0x7441u + 2 * h))),
                                        bias2);
#pragma unroll
                                    for (int m = 0; m < M; ++m)
                                        acc2[j][m] = f32x2_fma(f2, xp[ch][2 * q + h][m], acc2[j][m]);
                                }
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m)
                    f32x2_unpack(acc2[j][m], acc[j][m][0], acc[j][m][1]);
#else
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m)
                    acc[j][m][0] = acc[j][m][1] = 0.f;
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                if (j < nr) {
#pragma unroll
                    for (int ch = 0; ch < CH; ++ch) {
                        const int k0 = ch * LANE_SPAN + (warp * 32 + lane) * 16;
                        if (k0 < p.K) {
                            const uint4 v = lds128(base + (uint32_t)(j * p.K + k0));
                            const uint32_t wd[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u,
                                                    v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
                            for (int q = 0; q < 4; ++q)
#pragma unroll
                                for (int bt = 0; bt < 4; ++bt) {
                                    // bytes [u, 0, 0, 0x4B]: 2^23 + u, u = b + 128
                                    const float f =
                                        __uint_as_float(prmt(wd[q], 0x4B000000u, 0x7440u + bt)) -
                                        8388736.0f;
#pragma unroll
                                    for (int m = 0; m < M; ++m)
                                        acc[j][m][bt & 1] =
                                            fmaf(f, xr[ch][4 * q + bt][m], acc[j][m][bt & 1]);
                                }
                        }
                    }
                }
            }
#endif
            __syncwarp();
            if (lane == 0)
                mbar_arrive(empty0 + 8 * slot);
#if W4Q_W8_RS
            // The warp's sums of its RW x M values, reduced and scattered: at
            // offset o = 16, 8, .. each lane keeps the half of its values that
            // its offset bit selects and adds its partner's copy of that half,
            // so log2(VP) steps move VP - 1 values instead of 5 VP; then the
            // lanes holding one value sum it.  Lane (32 / VP) idx ends with
            // value idx.
            constexpr int V = RW * M, VP = V <= 2 ? 2 : (V <= 4 ? 4 : 8);
            float v[VP];
#pragma unroll
            for (int idx = 0; idx < VP; ++idx)
                v[idx] = idx < V ? acc[idx / M][idx % M][0] + acc[idx / M][idx % M][1] : 0.f;
#pragma unroll
            for (int n = VP, o = 16; n > 1; n >>= 1, o >>= 1) {
                const bool hi = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < n / 2; ++i) {
                    const float send = hi ? v[i] : v[i + n / 2];
                    const float keep = hi ? v[i + n / 2] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
#pragma unroll
            for (int o = 16 / VP; o > 0; o >>= 1)
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
            {
                const int idx = lane / (32 / VP), j = idx / M, m = idx % M;
                if (lane % (32 / VP) == 0 && idx < V && j < nr)
                    red[(warp * MAX_ROWS + (ra - r0 + j)) * M + m] = v[0];
            }
#else
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float v = acc[j][m][0] + acc[j][m][1];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0 && j < nr)
                        red[(warp * MAX_ROWS + (ra - r0 + j)) * M + m] = v;
                }
#endif
        }
    }
    __syncthreads();
    if (threadIdx.x == 0)
        W4Q_STAMP(32);
    for (int i = threadIdx.x; i < rows * M; i += THREADS) {
        const int row = i / M, m = i % M;
        float s = 0.f;
        for (int w = 0; w < CWARPS; ++w)
            s += red[(w * MAX_ROWS + row) * M + m];
        const float sc = __bfloat162float(p.scales[r0 + row]);
        p.out[(size_t)m * p.N + r0 + row] = __float2bfloat16_rn(s * sc);
    }
    if (warp == CWARPS && lane == 0) {
        for (int s = 0; s < STAGES && s < issued; ++s) {
            const int last_use = (issued - 1 - s) / STAGES;
            if (!W4Q_RING_WAIT(full0 + 8 * s, (uint32_t)last_use & 1)) {
                report_error(p.err, ERR_DRAIN_WAIT);
                break;
            }
        }
    }
}

template <int M, int CH, int RW, int ST>
cudaError_t launch_t(const W8Params &p, cudaStream_t stream)
{
    const int smem = ST * STAGE_BYTES + CWARPS * MAX_ROWS * M * 4 + 2 * ST * 8;
    static std::atomic<unsigned long long> opted_in{0};
    cudaError_t e = smem_opt_in_once(opted_in, w8_kernel<M, CH, RW, ST>, smem);
    if (e != cudaSuccess)
        return e;
    // programmatic dependent launch: the weight stream starts while the
    // previous kernel finishes; x is read after griddepcontrol.wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w8_kernel<M, CH, RW, ST>, p);
}

}  // namespace

// Supported: 1 <= M <= 4, K % 16 == 0, K <= 16384, M * ceil(K / 8192) <= 4.
bool w8_supported(int M, int K)
{
    if (M < 1 || M > 4 || K < 16 || K % 16 != 0 || K > STAGE_BYTES / 2)
        return false;
    const int ch = (K + LANE_SPAN - 1) / LANE_SPAN;
    return M * ch <= 4;
}

cudaError_t launch_w8(const void *x, const int8_t *W, const void *scales, void *out, int M, int N,
                      int K, int sm_count, unsigned *err, cudaStream_t stream)
{
    W8Params p;
    p.W = W;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.scales = static_cast<const __nv_bfloat16 *>(scales);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.err = err;
    p.N = N;
    p.K = K;
    int per_cta = (N + sm_count - 1) / sm_count;
    if (per_cta > MAX_ROWS)
        per_cta = MAX_ROWS;
    p.P = (N + per_cta - 1) / per_cta;
    const int ch = (K + LANE_SPAN - 1) / LANE_SPAN;  // 1: K <= 8192 (4 rows/stage), 2: <= 16384
    switch (M * 4 + ch) {
    case 1 * 4 + 1: return launch_t<1, 1, 4, 3>(p, stream);
    case 1 * 4 + 2: return launch_t<1, 2, 2, 5>(p, stream);
    case 2 * 4 + 1: return launch_t<2, 1, 4, 5>(p, stream);
    case 2 * 4 + 2: return launch_t<2, 2, 2, 5>(p, stream);
    case 3 * 4 + 1: return launch_t<3, 1, 2, 5>(p, stream);
    case 4 * 4 + 1: return launch_t<4, 1, 2, 5>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4q

W4Q_STAMP_READER(w4q_timeline_read_w8)
