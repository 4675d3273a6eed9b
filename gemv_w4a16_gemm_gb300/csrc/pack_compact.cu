// pack_compact.cu -- the compact W4 metadata: per (row, group of 32) a uint8
// scale code sc and a uint8 zero code zc, per row two fp16 steps ds and dz;
// scale = sc * ds, zero = zc * dz, dequant(q) = (q - zero) * scale.
// ("test_int4_quantized_gemm.py": CudaCoalescedInt4Tensor's scale /
// zero_point uint8 [N, K/32] and scale_step / zero_point_step float16
// [N, 1]; the page prints no dequant formula, and code x step for both is
// the reading this library takes.)
//
// Quantizer, per row, in fp64 and in this order (the decisions are IEEE
// operations, so any correct fp64 implementation takes the same ones):
//   s*_g = (max - min) / 15 (a constant group c: |c| / 15, or 1 for c = 0);
//   ds = the smallest fp16 >= max_g s*_g / 255;
//   sc_g = min(255, max(1, ceil(s*_g / ds)));   s_g = sc_g * ds (exact);
//   z*_g = clamp(-min / s_g, 0, 15);
//   dz = the smallest fp16 >= max_g z*_g / 255 (1 when all z*_g are 0);
//   zc_g = min(255, rint(z*_g / dz));           z_g = zc_g * dz (exact);
//   q = clamp(rint(w / s_g + z_g), 0, 15).
//
// Layout (include/w4q.h): 2304-byte tiles (16 rows x 256 K) in the order of
// the standard layout, [2048 B codes as there][128 B scale codes][128 B
// zero codes], the pair (row r, row r + 8) of group g at 2048 + 16 r + 2 g
// and 2176 + 16 r + 2 g; then the steps (ds, dz) of every row, N padded to
// a multiple of 128 (padding all zero).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace w4q {

namespace {

constexpr int CTILE = 2304;

__host__ __device__ __forceinline__ size_t ctile_offset(int t, int b, int KB)
{
    return (((size_t)(t / 8) * KB + b) * 8 + t % 8) * CTILE;
}

__host__ __device__ __forceinline__ size_t csteps_offset(int N, int K)
{
    return (size_t)((N + 127) / 128) * 8 * (K / 256) * CTILE;
}

// The smallest fp16 >= v (v finite, >= 0), as bits; +inf past 65504.  In
// [2^e, 2^(e+1)) fp16 numbers are the multiples of 2^(e-10), below 2^-14
// the multiples of 2^-24.
__device__ uint16_t fp16_bits_round_up(double v)
{
    if (!(v > 0.0))
        return 0;
    if (v > 65504.0)
        return 0x7C00;
    int lsb = ilogb(v) - 10;
    if (lsb < -24)
        lsb = -24;
    const double m = ceil(scalbn(v, -lsb));
    const double r = scalbn(m, lsb);
    if (r > 65504.0)
        return 0x7C00;
    if (r < 0x1p-14)
        return (uint16_t)m;
    const int re = ilogb(r);
    return (uint16_t)(((re + 15) << 10) | (int)(scalbn(r, 10 - re) - 1024.0));
}

__device__ __forceinline__ double fp16_bits_value(uint16_t h)
{
    return (double)__half2float(__ushort_as_half(h));  // exact
}

// max / min of the 32 values of group g of row n (exact in fp32)
__device__ __forceinline__ void group_range(const __nv_bfloat16 *__restrict__ row, int g,
                                            float &mn, float &mx)
{
    const uint4 *src = reinterpret_cast<const uint4 *>(row + (size_t)g * 32);
    mx = -INFINITY;
    mn = INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = src[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = bf16lo_to_f32(w[j]), hi = bf16hi_to_f32(w[j]);
            mx = fmaxf(mx, fmaxf(lo, hi));
            mn = fminf(mn, fminf(lo, hi));
        }
    }
}

__device__ __forceinline__ double group_sstar(float mn, float mx)
{
    if (mx == mn)
        return mx == 0.0f ? 1.0 : fabs((double)mx) / 15.0;
    return ((double)mx - (double)mn) / 15.0;
}

__device__ __forceinline__ double warp_max(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One warp per row (padding rows get zero steps): the row's two steps.
__global__ void __launch_bounds__(256) pack_c_steps_kernel(const __nv_bfloat16 *__restrict__ W,
                                                           uint8_t *__restrict__ packed, int N,
                                                           int K, int Npad)
{
    const int n = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (n >= Npad)
        return;
    uint16_t *steps = reinterpret_cast<uint16_t *>(packed + csteps_offset(N, K));
    if (n >= N) {
        if (lane == 0)
            steps[2 * n] = steps[2 * n + 1] = 0;
        return;
    }
    const int G = K / 32;
    const __nv_bfloat16 *row = W + (size_t)n * K;
    double smax = 0.0;
    for (int g = lane; g < G; g += 32) {
        float mn, mx;
        group_range(row, g, mn, mx);
        smax = fmax(smax, group_sstar(mn, mx));
    }
    smax = warp_max(smax);
    const uint16_t dsb = fp16_bits_round_up(smax / 255.0);
    const double ds = fp16_bits_value(dsb);
    double zmax = 0.0;
    for (int g = lane; g < G; g += 32) {
        float mn, mx;
        group_range(row, g, mn, mx);
        const double sc = fmin(255.0, fmax(1.0, ceil(group_sstar(mn, mx) / ds)));
        const double zs = fmin(fmax(-(double)mn / (sc * ds), 0.0), 15.0);
        zmax = fmax(zmax, zs);
    }
    zmax = warp_max(zmax);
    const uint16_t dzb = zmax > 0.0 ? fp16_bits_round_up(zmax / 255.0) : (uint16_t)0x3C00;
    if (lane == 0) {
        steps[2 * n] = dsb;
        steps[2 * n + 1] = dzb;
    }
}

// One CTA per 16-row x 256-K tile: thread (rr, gg) quantizes row rr's group
// gg with its row's steps, then the CTA writes the tile's 2304 bytes.
__global__ void __launch_bounds__(128) pack_c_kernel(const __nv_bfloat16 *__restrict__ W,
                                                     uint8_t *__restrict__ packed, int N, int K)
{
    __shared__ uint8_t codes[16][256];
    __shared__ uint8_t scodes[16][8];
    __shared__ uint8_t zcodes[16][8];

    const int KB = K / 256;
    const int t = blockIdx.x / KB, b = blockIdx.x % KB;
    const int rr = threadIdx.x / 8, gg = threadIdx.x % 8;
    const int n = t * 16 + rr;
    const uint16_t *steps = reinterpret_cast<const uint16_t *>(packed + csteps_offset(N, K));

    if (n < N) {
        const __nv_bfloat16 *row = W + (size_t)n * K;
        const int g = b * 8 + gg;
        float mn, mx;
        group_range(row, g, mn, mx);
        const double ds = fp16_bits_value(steps[2 * n]), dz = fp16_bits_value(steps[2 * n + 1]);
        const double scf = fmin(255.0, fmax(1.0, ceil(group_sstar(mn, mx) / ds)));
        const double s = scf * ds;
        const double zs = fmin(fmax(-(double)mn / s, 0.0), 15.0);
        const double zcf = fmin(255.0, rint(zs / dz));
        const double z = zcf * dz;
        const uint4 *src = reinterpret_cast<const uint4 *>(row + (size_t)g * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = src[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const double lo = (double)bf16lo_to_f32(w[j]), hi = (double)bf16hi_to_f32(w[j]);
                codes[rr][gg * 32 + 8 * i + 2 * j] =
                    (uint8_t)fmin(fmax(rint(lo / s + z), 0.0), 15.0);
                codes[rr][gg * 32 + 8 * i + 2 * j + 1] =
                    (uint8_t)fmin(fmax(rint(hi / s + z), 0.0), 15.0);
            }
        }
        scodes[rr][gg] = (uint8_t)scf;
        zcodes[rr][gg] = (uint8_t)zcf;
    } else {
        for (int i = 0; i < 32; ++i)
            codes[rr][gg * 32 + i] = 0;
        scodes[rr][gg] = 0;
        zcodes[rr][gg] = 0;
    }
    __syncthreads();

    uint32_t *tile = reinterpret_cast<uint32_t *>(packed + ctile_offset(t, b, KB));
    // nibble words: word 128*sb + 4*l + j, as in the standard layout
    for (int wi = threadIdx.x; wi < 512; wi += 128) {
        const int sb = wi / 128, l = (wi / 4) % 32, j = wi % 4;
        const int r = l / 4, c = 2 * (l % 4);
        uint32_t word = 0;
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = r + 8 * a;
                    const int col = 64 * sb + 16 * j + c + 8 * e + h;
                    word |= (uint32_t)codes[row][col] << (8 * a + 4 * e + 16 * h);
                }
        tile[wi] = word;
    }
    // code words: word 4*r + g/2 holds (r, g), (r+8, g), (r, g+1), (r+8, g+1)
    if (threadIdx.x < 64) {
        const int wi = threadIdx.x & 31, r = wi / 4, g = 2 * (wi % 4);
        const uint8_t(*src)[8] = threadIdx.x < 32 ? scodes : zcodes;
        tile[512 + (threadIdx.x < 32 ? 0 : 32) + wi] =
            (uint32_t)src[r][g] | ((uint32_t)src[r + 8][g] << 8) | ((uint32_t)src[r][g + 1] << 16) |
            ((uint32_t)src[r + 8][g + 1] << 24);
    }
}

// The inverse view: codes, scale codes, zero codes and steps of rows < N.
__global__ void unpack_c_kernel(const uint8_t *__restrict__ packed, uint8_t *__restrict__ q,
                                uint8_t *__restrict__ sc, uint8_t *__restrict__ zc,
                                uint16_t *__restrict__ steps, int N, int K)
{
    const int KB = K / 256, G = K / 32;
    const size_t total = (size_t)N * K;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int n = (int)(i / K), k = (int)(i % K);
        const int t = n / 16, rr = n % 16, b = k / 256, kk = k % 256;
        const int sb = kk / 64, j = (kk % 64) / 16, col = kk % 16;
        const int r = rr % 8, prow = rr / 8, chi = col / 8, cc = col % 8;
        const int h = cc % 2, c = cc - h;
        const int l = 4 * r + c / 2;
        const int bit = 8 * prow + 4 * chi + 16 * h;
        const size_t tile = ctile_offset(t, b, KB);
        q[i] = (packed[tile + 512 * sb + 16 * l + 4 * j + bit / 8] >> (bit % 8)) & 0xF;
        if (kk % 32 == 0) {
            const int gg = kk / 32;
            sc[(size_t)n * G + k / 32] = packed[tile + 2048 + 16 * r + 2 * gg + prow];
            zc[(size_t)n * G + k / 32] = packed[tile + 2176 + 16 * r + 2 * gg + prow];
        }
        if (k == 0) {
            const uint16_t *st = reinterpret_cast<const uint16_t *>(packed + csteps_offset(N, K));
            steps[2 * n] = st[2 * n];
            steps[2 * n + 1] = st[2 * n + 1];
        }
    }
}

}  // namespace

size_t packed_bytes_compact(int N, int K)
{
    return csteps_offset(N, K) + (size_t)((N + 127) / 128) * 128 * 4;
}

cudaError_t launch_pack_compact(const void *W, void *packed, int N, int K, cudaStream_t stream)
{
    const int Npad = (N + 127) / 128 * 128;
    pack_c_steps_kernel<<<Npad / 8, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(W),
                                                     static_cast<uint8_t *>(packed), N, K, Npad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int tiles = (Npad / 128) * 8 * (K / 256);
    pack_c_kernel<<<tiles, 128, 0, stream>>>(static_cast<const __nv_bfloat16 *>(W),
                                             static_cast<uint8_t *>(packed), N, K);
    return cudaGetLastError();
}

cudaError_t launch_unpack_compact(const void *packed, uint8_t *q, uint8_t *sc, uint8_t *zc,
                                  void *steps, int N, int K, cudaStream_t stream)
{
    const size_t total = (size_t)N * K;
    const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    unpack_c_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint8_t *>(packed), q, sc, zc,
                                                static_cast<uint16_t *>(steps), N, K);
    return cudaGetLastError();
}

}  // namespace w4q
