// w4_stage.cuh -- the device-side building blocks shared by the two W4
// kernels for M <= 8 (gemv_w4.cu: stream-K over all SMs with a prologue;
// gemv_w4_cluster.cu: one thread-block cluster per 128-row group): the
// stage layout constants, the kernel parameters, the per-stage tensor-core
// group dots with their scale / zero update, and the W4A16 activation
// preparation of one 256-column super-block.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace w4q {

namespace {

constexpr int TILE_BYTES = 2432;
constexpr int WARPS = 8;                   // consumer warps = row tiles per tile group
constexpr int GROUP_ROWS = WARPS * 16;     // rows of one tile group
constexpr int THREADS = (WARPS + 1) * 32;  // + one producer warp
constexpr int XROW = 512 + 16;             // one activation row's 256-K chunk, padded
constexpr int SROW = 32;                   // one activation row's 8 group sums (fp32)

struct Params {
    const uint8_t *packed;
    const __nv_bfloat16 *x;  // W4A8: bf16 [K/256][M][264]: x' (prepared)
    const float *xsum;       // W4A8: fp32 [K/256][M][8]: X'
    const float *gscale;     // W4A8: fp32 [K/256][M][8]: activation scale x 2^12 per group
    const __nv_bfloat16 *xin;  // W4A16: bf16 [M][K], the activations as given
    __nv_bfloat16 *out;      // bf16 [M][N]
    int32_t *dots;           // group-dot export: int32 [M][N][K/32]
    float *partial;          // fp32 [P][2][M][GROUP_ROWS]
    unsigned *counters;      // [G][WARPS] arrivals per row tile (zeroed by the prologue)
    unsigned *err;
    int M, N, K, KB, T, G, P, split;
    long long U;
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// The stage functions read only p.M, p.N, p.K and p.dots (the W4A8
// group-dot export) from the kernel parameters, whichever kernel's they are.
//
// CMP: the tile holds the compact metadata (2304-byte tiles: uint8 scale
// codes at 2048 and zero codes at 2176, the pair of rows r, r + 8 of group
// g in word g / 2, bytes 2 (g % 2) and 2 (g % 2) + 1); rs holds this lane's
// row steps (ds of rows r, r + 8, then dz of rows r, r + 8) as fp32.  The
// scale sc * ds and the zero zc * dz are exact in fp32 (8 x 11 bits).

// bytes [c, 0, 0, 0x4B] = 2^23 + c: the byte c of word w at byte index i
__device__ __forceinline__ float byte_as_float(uint32_t w, uint32_t i)
{
    return __uint_as_float(prmt(w, 0x4B000000u, 0x7440u + i)) - 8388608.0f;
}

// Group g's scales sr, sr8 and negated zero points nzr, nzr8 of rows r and
// r + 8, from the standard metadata words (sw: the bf16 pair of the group,
// zw: the zero bytes' word) or the compact ones (sw: the scale codes' word,
// zw: the zero codes' word).
template <bool CMP>
__device__ __forceinline__ void group_meta(uint32_t sw, uint32_t zw, int g, const float (&rs)[4],
                                           float &sr, float &sr8, float &nzr, float &nzr8)
{
    const uint32_t zb = (uint32_t)((2 * g) & 3);  // byte of row r; row r + 8 follows
    if constexpr (CMP) {
        sr = byte_as_float(sw, zb) * rs[0];
        sr8 = byte_as_float(sw, zb + 1) * rs[1];
        nzr = -(byte_as_float(zw, zb) * rs[2]);
        nzr8 = -(byte_as_float(zw, zb + 1) * rs[3]);
    } else {
        sr = bf16lo_to_f32(sw);
        sr8 = bf16hi_to_f32(sw);
        nzr = -byte_as_float(zw, zb);
        nzr8 = -byte_as_float(zw, zb + 1);
    }
}

// The metadata words of group g for rows r, r + 8, read from the tile.
template <bool CMP>
__device__ __forceinline__ void group_meta_words(uint32_t wbase, int r, int g, uint32_t &sw,
                                                 uint32_t &zw)
{
    if constexpr (CMP) {
        sw = lds32(wbase + 2048 + 16 * r + 4 * (g >> 1));
        zw = lds32(wbase + 2176 + 16 * r + 4 * (g >> 1));
    } else {
        sw = lds32(wbase + 2048 + ((g & 4) ? 128 : 0) + 16 * r + 4 * (g & 3));
        zw = lds32(wbase + 2304 + 16 * r + 4 * (g >> 1));
    }
}

// One stage: this warp's 16 x 256 tile, 4 sub-blocks of 64 K (two groups
// each), 4 k16 steps per sub-block.  xbase: the stage's activation rows;
// sbase: the stage's group sums; gbase: per row, the W4A8 group scales (GS)
// or the stage's row factor c (SC: the stage's sum is scaled once by c).
template <int NB, bool DOTS, bool GS, bool SC, bool CMP = false, class PP>
__device__ __forceinline__ void compute_stage(uint32_t wbase, uint32_t xbase, uint32_t sbase,
                                              uint32_t gbase, int lane, float (&acc)[NB][4],
                                              const PP &p, int tile, int b,
                                              const float (&rs)[4] = {1.f, 1.f, 1.f, 1.f})
{
    const int r = lane >> 2, c2 = 2 * (lane & 3);
    // the metadata words: per group g the scale word scw[g] (compact: the
    // scale codes' word g / 2) and the zero word zw[g / 2]
    uint32_t scw[8], zw[4];
    if constexpr (CMP) {
        const uint4 sc0 = lds128(wbase + 2048 + 16 * r);
        const uint4 zz = lds128(wbase + 2176 + 16 * r);
        const uint32_t s4[4] = {sc0.x, sc0.y, sc0.z, sc0.w};
#pragma unroll
        for (int g = 0; g < 8; ++g)
            scw[g] = s4[g >> 1];
        zw[0] = zz.x; zw[1] = zz.y; zw[2] = zz.z; zw[3] = zz.w;
    } else {
        const uint4 sc0 = lds128(wbase + 2048 + 16 * r);
        const uint4 sc1 = lds128(wbase + 2048 + 128 + 16 * r);
        const uint4 zz = lds128(wbase + 2304 + 16 * r);
        scw[0] = sc0.x; scw[1] = sc0.y; scw[2] = sc0.z; scw[3] = sc0.w;
        scw[4] = sc1.x; scw[5] = sc1.y; scw[6] = sc1.z; scw[7] = sc1.w;
        zw[0] = zz.x; zw[1] = zz.y; zw[2] = zz.z; zw[3] = zz.w;
    }
    // ldmatrix.x4 row addresses: matrix lane>>3 = (step +lane>>4, k half (lane>>3)&1)
    const uint32_t xlane = xbase + (lane & 7) * XROW + 32 * (lane >> 4) + 16 * ((lane >> 3) & 1);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float sacc[NB][4];  // SC: this stage's sums, before the row factors
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
        sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
    float (&tgt)[NB][4] = SC ? sacc : acc;

    // group sums X' of this lane's two output columns, per n8 block
    float xs[NB][2][8];
    {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t a = sbase + (nb * 8 + c2 + e) * SROW;
                const uint4 v0 = lds128(a), v1 = lds128(a + 16);
                xs[nb][e][0] = __uint_as_float(v0.x);
                xs[nb][e][1] = __uint_as_float(v0.y);
                xs[nb][e][2] = __uint_as_float(v0.z);
                xs[nb][e][3] = __uint_as_float(v0.w);
                xs[nb][e][4] = __uint_as_float(v1.x);
                xs[nb][e][5] = __uint_as_float(v1.y);
                xs[nb][e][6] = __uint_as_float(v1.z);
                xs[nb][e][7] = __uint_as_float(v1.w);
            }
    }

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
            {
                float d[NB][4];
#pragma unroll
                for (int st = 0; st < 2; ++st) {
                    const uint32_t w = wv[2 * gi + st], t = w >> 8;
                    uint32_t a[4];  // q * 2^-133 (low nibbles), q * 2^-129 (high nibbles)
                    a[0] = w & 0x000F000Fu;
                    a[1] = t & 0x000F000Fu;
                    a[2] = w & 0x00F000F0u;
                    a[3] = t & 0x00F000F0u;
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        if (st == 0)
                            mma_bf16(d[nb], a, bf[nb][2 * gi][0], bf[nb][2 * gi][1], zero4);
                        else
                            mma_bf16(d[nb], a, bf[nb][2 * gi + 1][0], bf[nb][2 * gi + 1][1], d[nb]);
                    }
                }
                float sr, sr8, nzr, nzr8;
                group_meta<CMP>(scw[g], zw[g >> 1], g, rs, sr, sr8, nzr, nzr8);
                if (DOTS) {
                    const int G = p.K / 32, gg = b * 8 + g;
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int m = nb * 8 + c2 + (e & 1);
                            const int n = tile * 16 + r + 8 * (e >> 1);
                            const float dg = fmaf((e >> 1) ? nzr8 : nzr, xs[nb][e & 1][g], d[nb][e]);
                            if (m < p.M && n < p.N)
                                p.dots[((size_t)m * p.N + n) * G + gg] = (int32_t)rintf(dg * 4096.0f);
                        }
                } else {
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        // W4A8: times the activation scale of (column, group)
                        const float g0 = GS ? __uint_as_float(lds32(gbase + (nb * 8 + c2) * SROW + 4 * g)) : 1.f;
                        const float g1 = GS ? __uint_as_float(lds32(gbase + (nb * 8 + c2 + 1) * SROW + 4 * g)) : 1.f;
                        tgt[nb][0] = fmaf(GS ? sr * g0 : sr, fmaf(nzr, xs[nb][0][g], d[nb][0]), tgt[nb][0]);
                        tgt[nb][1] = fmaf(GS ? sr * g1 : sr, fmaf(nzr, xs[nb][1][g], d[nb][1]), tgt[nb][1]);
                        tgt[nb][2] = fmaf(GS ? sr8 * g0 : sr8, fmaf(nzr8, xs[nb][0][g], d[nb][2]), tgt[nb][2]);
                        tgt[nb][3] = fmaf(GS ? sr8 * g1 : sr8, fmaf(nzr8, xs[nb][1][g], d[nb][3]), tgt[nb][3]);
                    }
                }
            }
        }
    }
    if (SC) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const float ca = __uint_as_float(lds32(gbase + (nb * 8 + c2) * SROW));
            const float cb = __uint_as_float(lds32(gbase + (nb * 8 + c2 + 1) * SROW));
            acc[nb][0] = fmaf(ca, sacc[nb][0], acc[nb][0]);
            acc[nb][1] = fmaf(cb, sacc[nb][1], acc[nb][1]);
            acc[nb][2] = fmaf(ca, sacc[nb][2], acc[nb][2]);
            acc[nb][3] = fmaf(cb, sacc[nb][3], acc[nb][3]);
        }
    }
}


// One stage at NB = 1 with MP = 1, 2 or 4 rows of x per accumulator slot:
// the 8 columns of the m16n8k16 accumulator hold 8 / MP groups x MP rows
// (column n: group slot n / MP, row n % MP).  For the MMAs of a group, the
// B columns of the other slots are zero: ldmatrix takes each row's address
// per lane, so those lanes point at a 16-byte zero row (zaddr) and the others
// at the x' row of their column.  One accumulator thus sums the dots of
// 8 / MP groups side by side, and the fp32 scale / zero update runs once per
// 8 / MP groups instead of once per group.  The lanes of one accumulator row
// hold different slots of the same outputs; the flush adds them.  GS, SC: as
// for compute_stage.  CHAINS: accumulators a round's groups are spread over
// (0: 4 at MP = 1, 1 above; see below).
template <int MP, bool DOTS, bool GS, bool SC, bool CMP = false, int CHAINS = 0, class PP>
__device__ __forceinline__ void compute_stage_packed(uint32_t wbase, uint32_t xbase,
                                                     uint32_t sbase, uint32_t gbase, uint32_t zaddr,
                                                     int lane, float (&acc)[1][4], const PP &p,
                                                     int tile, int b,
                                                     const float (&rs)[4] = {1.f, 1.f, 1.f, 1.f})
{
    constexpr int GP = 8 / MP;  // groups per accumulator round
    const int r = lane >> 2, c2 = 2 * (lane & 3);
    // ldmatrix.x4 row of this lane: matrix q = (step +q>>1, k half q&1), B column n
    const int bn = lane & 7, q = lane >> 3, bslot = bn / MP;
    const uint32_t brow = xbase + (bn % MP) * XROW + 32 * (q >> 1) + 16 * (q & 1);
    const int s0 = c2 / MP, s1 = (c2 + 1) / MP, m0 = c2 % MP, m1 = (c2 + 1) % MP;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float sacc[1][4] = {{0.f, 0.f, 0.f, 0.f}};  // SC: this stage's sums, before the row factors
    float (&tgt)[1][4] = SC ? sacc : acc;
    uint32_t wv[16];  // word of step st: codes of rows r, r + 8 (step = 2 * group + half)
#pragma unroll
    for (int sbk = 0; sbk < 4; ++sbk) {
        const uint4 wq = lds128(wbase + 512 * sbk + 16 * lane);
        wv[4 * sbk] = wq.x;
        wv[4 * sbk + 1] = wq.y;
        wv[4 * sbk + 2] = wq.z;
        wv[4 * sbk + 3] = wq.w;
    }
    // A round's groups go to NACC accumulators.  Their columns are disjoint
    // (a group's MMAs add exact zeros to the other groups' columns), so one
    // accumulator can take them all, and adding several afterwards is exact.
    // Several give shorter MMA dependency chains, one saves the adds: at
    // MP >= 2 the rounds already give independent chains (W4A8 39936 x 6656:
    // M = 2 33.9 -> 32.5 us, M = 4 36.7 -> 35.8 us with one), while the
    // stream-K kernel at MP = 1 keeps four (32.4 against 32.7 us with one).
    constexpr int NMAX = CHAINS > 0 ? CHAINS : (MP == 1 ? 4 : 1);
    constexpr int NACC = GP >= NMAX ? NMAX : GP, GPA = GP / NACC;
#pragma unroll
    for (int R = 0; R < MP; ++R) {
        float dacc[NACC][4];
#pragma unroll
        for (int pp = 0; pp < GP; ++pp) {  // group R * GP + pp: steps 2g, 2g + 1
            const int g = R * GP + pp, ai = pp / GPA;
            uint32_t bf[2][2];
            ldmatrix_x4(bslot == pp ? brow + 64 * g : zaddr, bf[0][0], bf[0][1], bf[1][0], bf[1][1]);
#pragma unroll
            for (int st = 0; st < 2; ++st) {
                const uint32_t w = wv[2 * g + st], t = w >> 8;
                uint32_t a[4];  // q * 2^-133 (low nibbles), q * 2^-129 (high nibbles)
                a[0] = w & 0x000F000Fu;
                a[1] = t & 0x000F000Fu;
                a[2] = w & 0x00F000F0u;
                a[3] = t & 0x00F000F0u;
                if (pp % GPA == 0 && st == 0)
                    mma_bf16(dacc[ai], a, bf[st][0], bf[st][1], zero4);
                else
                    mma_bf16(dacc[ai], a, bf[st][0], bf[st][1], dacc[ai]);
            }
        }
        float d[4] = {dacc[0][0], dacc[0][1], dacc[0][2], dacc[0][3]};
#pragma unroll
        for (int ai = 1; ai < NACC; ++ai)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                d[e] += dacc[ai][e];
        // the groups of this lane's two columns in this round
        const int g0 = R * GP + s0, g1 = R * GP + s1;
        // scales and negated zero points of the groups of this lane's two
        // columns (the same group unless MP == 1), rows r and r + 8
        uint32_t sw0, zw0;
        group_meta_words<CMP>(wbase, r, g0, sw0, zw0);
        float s0r, s0r8, nz0, nz08;
        group_meta<CMP>(sw0, zw0, g0, rs, s0r, s0r8, nz0, nz08);
        float s1r = s0r, s1r8 = s0r8, nz1 = nz0, nz18 = nz08;
        if (MP == 1) {
            uint32_t sw1, zw1;
            group_meta_words<CMP>(wbase, r, g1, sw1, zw1);
            group_meta<CMP>(sw1, zw1, g1, rs, s1r, s1r8, nz1, nz18);
        }
        const float xs0 = __uint_as_float(lds32(sbase + m0 * SROW + 4 * g0));
        const float xs1 = __uint_as_float(lds32(sbase + m1 * SROW + 4 * g1));
        if (DOTS) {
            const int G = p.K / 32;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = (e & 1) ? m1 : m0, g = (e & 1) ? g1 : g0;
                const int n = tile * 16 + r + 8 * (e >> 1);
                const float nz = (e & 1) ? ((e >> 1) ? nz18 : nz1) : ((e >> 1) ? nz08 : nz0);
                const float dg = fmaf(nz, (e & 1) ? xs1 : xs0, d[e]);
                if (m < p.M && n < p.N)
                    p.dots[((size_t)m * p.N + n) * G + b * 8 + g] = (int32_t)rintf(dg * 4096.0f);
            }
        } else {
            // W4A8: times the activation scale of (row of x, group)
            const float ga = GS ? __uint_as_float(lds32(gbase + m0 * SROW + 4 * g0)) : 1.f;
            const float gb = GS ? __uint_as_float(lds32(gbase + m1 * SROW + 4 * g1)) : 1.f;
            tgt[0][0] = fmaf(s0r * ga, fmaf(nz0, xs0, d[0]), tgt[0][0]);
            tgt[0][1] = fmaf(s1r * gb, fmaf(nz1, xs1, d[1]), tgt[0][1]);
            tgt[0][2] = fmaf(s0r8 * ga, fmaf(nz08, xs0, d[2]), tgt[0][2]);
            tgt[0][3] = fmaf(s1r8 * gb, fmaf(nz18, xs1, d[3]), tgt[0][3]);
        }
    }
    if (SC) {
        const float ca = __uint_as_float(lds32(gbase + m0 * SROW));
        const float cb = __uint_as_float(lds32(gbase + m1 * SROW));
        acc[0][0] = fmaf(ca, sacc[0][0], acc[0][0]);
        acc[0][1] = fmaf(cb, sacc[0][1], acc[0][1]);
        acc[0][2] = fmaf(ca, sacc[0][2], acc[0][2]);
        acc[0][3] = fmaf(cb, sacc[0][3], acc[0][3]);
    }
}

// W4A16: one stage's activation operand, prepared by the producer warp from
// super-block b of x (rows m < M, 256 columns; lane l holds columns
// 8l .. 8l + 7, so an odd lane holds the upper half of a 16-column step).
// Per row: sigma from max |x| over the super-block, x' = x * 2^sigma (upper
// halves 2^(sigma - 4)) as bf16, X'[g] = 2^(sigma - 133) * sum_{k in g} x_k,
// c = 2^(133 - sigma).  sigma keeps |x'| < 2^128, so every power-of-two
// product below is exact and x' is x scaled without rounding.
template <int MP>
__device__ __forceinline__ void load_stage_a16(const __nv_bfloat16 *__restrict__ x, int M, int K,
                                               int b, int lane, uint4 (&raw)[MP])
{
#pragma unroll
    for (int m = 0; m < MP; ++m)
        raw[m] = m < M ? __ldcg(reinterpret_cast<const uint4 *>(x + (size_t)m * K +
                                                               (size_t)b * 256) + lane)
                       : make_uint4(0u, 0u, 0u, 0u);
}

// The MP rows are processed together (rows m >= M hold zeros and are not
// stored), so that their reduction chains overlap.
template <int MP>
__device__ __forceinline__ void prep_stage_a16(const uint4 (&raw)[MP], int M, int lane,
                                               uint8_t *xdst, uint8_t *sdst, uint8_t *cdst)
{
    constexpr int NW = (MP + 1) / 2;
    // max |x| per row: magnitudes of bf16 numbers order as their bit
    // patterns; two rows per word (16-bit lanes) for the warp reduction
    uint32_t mx[NW];
#pragma unroll
    for (int j = 0; j < NW; ++j)
        mx[j] = 0u;
#pragma unroll
    for (int m = 0; m < MP; ++m) {
        const uint32_t h = __vmaxu2(__vmaxu2(raw[m].x & 0x7FFF7FFFu, raw[m].y & 0x7FFF7FFFu),
                                    __vmaxu2(raw[m].z & 0x7FFF7FFFu, raw[m].w & 0x7FFF7FFFu));
        mx[m / 2] |= max(h & 0xFFFFu, h >> 16) << (16 * (m & 1));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < NW; ++j)
            mx[j] = __vmaxu2(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], o));
    float part[MP];
#pragma unroll
    for (int m = 0; m < MP; ++m) {
        const uint32_t a = (mx[m / 2] >> (16 * (m & 1))) & 0xFFFFu;
        // e with max |x| < 2^e (e = 0 for an all-zero row), from the bf16 bits:
        // a normal number with biased exponent E is below 2^(E - 126); a
        // subnormal q * 2^-133 with q < 2^nb is below 2^(nb - 133)
        const int e = a >= 0x80u ? (int)(a >> 7) - 126 : (a != 0u ? (32 - __clz((int)a)) - 133 : 0);
        const int sigma = min(max(128 - e, 6), 259);
        const int sh = (lane & 1) ? sigma - 4 : sigma;
        const uint32_t w[4] = {raw[m].x, raw[m].y, raw[m].z, raw[m].w};
        float v[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = bf16lo_to_f32(w[j]);
            v[2 * j + 1] = bf16hi_to_f32(w[j]);
        }
        part[m] = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
        // 2^sh in factors of at most 2^127 (sh <= 259)
        const float f1 = __uint_as_float((uint32_t)(min(sh, 127) + 127) << 23);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] *= f1;
        if (sigma > 127) {  // the same for the whole warp
            const int a2 = min(max(sh - 127, 0), 127);
            const float f2 = __uint_as_float((uint32_t)(a2 + 127) << 23);
            const float f3 = __uint_as_float((uint32_t)(max(sh - 254, 0) + 127) << 23);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = v[j] * f2 * f3;
        }
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);  // .x low
            ow[j] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        if (m < M) {
            *reinterpret_cast<uint4 *>(xdst + m * XROW + 16 * lane) =
                make_uint4(ow[0], ow[1], ow[2], ow[3]);
            if (lane == 0)
                *reinterpret_cast<float *>(cdst + m * SROW) =
                    __uint_as_float((uint32_t)(260 - sigma) << 23);
        }
        // 2^(sigma - 133) = 2^(sigma - 132) * 2^-1, both normal for sigma in [6, 259]
        part[m] *= __uint_as_float((uint32_t)(sigma - 5) << 23);
    }
#pragma unroll
    for (int m = 0; m < MP; ++m)
        part[m] += __shfl_xor_sync(0xffffffffu, part[m], 1);
#pragma unroll
    for (int m = 0; m < MP; ++m)
        part[m] += __shfl_xor_sync(0xffffffffu, part[m], 2);
#pragma unroll
    for (int m = 0; m < MP; ++m)
        if (m < M && (lane & 3) == 0)
            *reinterpret_cast<float *>(sdst + m * SROW + 4 * (lane >> 2)) = part[m] * 0.5f;
}

}  // namespace

}  // namespace w4q
