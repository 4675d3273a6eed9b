// pack.cu -- INT4 group-wise asymmetric min-max quantizer and packer
// ("test_int4_quantized_gemm.py", _packed_with_dense: QuantConfig(bits=4,
// group_size=32, symmetric=False, method="min_max")), writing the tile layout
// documented in w4q.h, plus the inverse view used by the tests.
#include "common.cuh"
#include "kernels.h"

namespace w4q {

namespace {

constexpr int TILE_BYTES = 2432;

// Tiles are ordered (128-row group, super-block, row tile of the group).
__host__ __device__ __forceinline__ size_t tile_offset(int t, int b, int KB)
{
    return (((size_t)(t / 8) * KB + b) * 8 + t % 8) * TILE_BYTES;
}

// One CTA quantizes one 16-row x 256-K tile (every tile of the padded
// layout, all-zero rows included): thread (rr, gg) owns row rr and group gg
// (8 groups of 32), then the CTA writes the tile's 2432 bytes with coalesced
// 32-bit stores.
__global__ void __launch_bounds__(128) pack_kernel(const __nv_bfloat16 *__restrict__ W,
                                                   uint8_t *__restrict__ packed, int N, int K)
{
    __shared__ uint8_t codes[16][256];
    __shared__ uint16_t scales[16][8];
    __shared__ uint8_t zeros[16][8];

    const int KB = K / 256;
    const int t = blockIdx.x / KB, b = blockIdx.x % KB;
    const int rr = threadIdx.x / 8, gg = threadIdx.x % 8;
    const int n = t * 16 + rr;

    if (n < N) {
        const uint4 *src =
            reinterpret_cast<const uint4 *>(W + (size_t)n * K + (size_t)b * 256 + gg * 32);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 v = src[i];
            w[4 * i + 0] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        float mx = -INFINITY, mn = INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float lo = bf16lo_to_f32(w[i]), hi = bf16hi_to_f32(w[i]);
            mx = fmaxf(mx, fmaxf(lo, hi));
            mn = fminf(mn, fminf(lo, hi));
        }
        // scale: the smallest bf16 >= fl64(fl64(max - min) / 15); rounding
        // up twice (fp64 -> fp32 -> bf16) equals rounding up once.
        double t64;
        if (mx == mn) {
            const double c = fabs((double)mx);
            t64 = (c == 0.0) ? 1.0 : __ddiv_rn(c, 15.0);
        } else {
            t64 = __ddiv_rn(__dsub_rn((double)mx, (double)mn), 15.0);
        }
        const __nv_bfloat16 sb = __float2bfloat16_ru(__double2float_ru(t64));
        const float s = __bfloat162float(sb);
        // Codes from the stored scale.  w and s are bf16, so a w / s that is
        // not a half-integer is at least 2^-10 away from one while the fp32
        // quotient is within 2^-20: rint of the fp32 quotient is the exact
        // decision.
        const float z = fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.0f), 15.0f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float lo = bf16lo_to_f32(w[i]), hi = bf16hi_to_f32(w[i]);
            codes[rr][gg * 32 + 2 * i] =
                (uint8_t)fminf(fmaxf(rintf(__fdiv_rn(lo, s)) + z, 0.0f), 15.0f);
            codes[rr][gg * 32 + 2 * i + 1] =
                (uint8_t)fminf(fmaxf(rintf(__fdiv_rn(hi, s)) + z, 0.0f), 15.0f);
        }
        scales[rr][gg] = __bfloat16_as_ushort(sb);
        zeros[rr][gg] = (uint8_t)z;
    } else {
        for (int i = 0; i < 32; ++i)
            codes[rr][gg * 32 + i] = 0;
        scales[rr][gg] = 0;
        zeros[rr][gg] = 0;
    }
    __syncthreads();

    uint32_t *tile = reinterpret_cast<uint32_t *>(packed + tile_offset(t, b, KB));
    // nibble words: word index 128*sb + 4*l + j
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
    // scale words: word 32*(g/4) + 4*r + g%4 holds (s[r][g], s[r+8][g])
    if (threadIdx.x < 64) {
        const int wi = threadIdx.x;
        const int g = 4 * (wi / 32) + wi % 4, r = (wi / 4) % 8;
        tile[512 + wi] = (uint32_t)scales[r][g] | ((uint32_t)scales[r + 8][g] << 16);
    }
    // zero words: word 4*r + g/2 holds z[r][g], z[r+8][g], z[r][g+1], z[r+8][g+1]
    if (threadIdx.x >= 64 && threadIdx.x < 96) {
        const int wi = threadIdx.x - 64;
        const int r = wi / 4, g = 2 * (wi % 4);
        tile[576 + wi] = (uint32_t)zeros[r][g] | ((uint32_t)zeros[r + 8][g] << 8) |
                         ((uint32_t)zeros[r][g + 1] << 16) | ((uint32_t)zeros[r + 8][g + 1] << 24);
    }
}

// The inverse view: one thread per code, one per (row, group) for s and z.
__global__ void unpack_kernel(const uint8_t *__restrict__ packed, uint8_t *__restrict__ q,
                              uint16_t *__restrict__ scale, uint8_t *__restrict__ zero, int N,
                              int K)
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
        const size_t byte = tile_offset(t, b, KB) + 512 * sb + 16 * l + 4 * j + bit / 8;
        q[i] = (packed[byte] >> (bit % 8)) & 0xF;
        if (kk % 32 == 0) {
            const int gg = kk / 32;
            const size_t tile = tile_offset(t, b, KB);
            const size_t sbyte = tile + 2048 + 128 * (gg / 4) + 16 * r + 4 * (gg % 4) + 2 * prow;
            scale[(size_t)n * G + k / 32] =
                (uint16_t)(packed[sbyte] | ((uint16_t)packed[sbyte + 1] << 8));
            zero[(size_t)n * G + k / 32] = packed[tile + 2304 + 16 * r + 2 * gg + prow];
        }
    }
}

}  // namespace

cudaError_t launch_pack(const void *W, void *packed, int N, int K, cudaStream_t stream)
{
    const int tiles = ((N + 127) / 128) * 8 * (K / 256);
    pack_kernel<<<tiles, 128, 0, stream>>>(static_cast<const __nv_bfloat16 *>(W),
                                           static_cast<uint8_t *>(packed), N, K);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const void *packed, uint8_t *q, void *scale, uint8_t *zero, int N, int K,
                          cudaStream_t stream)
{
    const size_t total = (size_t)N * K;
    const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    unpack_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint8_t *>(packed), q,
                                              static_cast<uint16_t *>(scale), zero, N, K);
    return cudaGetLastError();
}

}  // namespace w4q
