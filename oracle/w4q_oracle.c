/*
 * w4q_oracle.c -- plain, slow, obviously correct CPU reference ("the oracle")
 * for the decode-sized weight-only quantized linear layer
 *
 *     out[M,N] = x[M,K] . dequant(Wq)[N,K]^T
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: everything below is written from the definitions.
 *
 * Floating point is fp64 unless a step is defined in another precision (the
 * W4A8 activation quantizer is defined in IEEE fp32 so that both sides take
 * the same integer decision; see oracle_act_quant).  Compile without
 * -ffast-math and with -ffp-contract=off.
 *
 * Sources (web pages, cited by title and section):
 *  [T]  "test_int4_quantized_gemm.py" (ExecuTorch CUDA backend tests):
 *       _packed_with_dense (QuantConfig(bits=4, group_size=32,
 *       symmetric=False, method="min_max")), the _dequant_matmul reference
 *       used by _check_close, Int4QuantizedGemmLegalityTest (K % 256, group
 *       32), Int4QuantizedGemmPrecisionTest (W4A8 vs W4A16 class).
 *  [G]  "gpt-fast issue #114: Question about the generated code of
 *       WeightOnlyInt8Linear": WeightOnlyInt8Linear.forward
 *       (F.linear(x, W.to(bf16)) * scales) and the fused reduction kernel.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - scale s per (row, group of 32) is stored as bf16 and is the smallest
 *    bf16 >= fl64(fl64(max - min) / 15)  (round toward +inf), so that
 *    |w - dequant| <= s/2 holds for every group that straddles zero;
 *  - a constant group (max == min == c) uses s = RU_bf16(|c| / 15), or 1.0
 *    when c == 0;
 *  - zero z = clamp(rint(-min / s), 0, 15), code q = clamp(rint(w / s) + z,
 *    0, 15), both from the STORED bf16 s, rint = round half to even;
 *  - dequant(q) = (q - z) * s.
 *
 * W4A8 comes in two activation granularities: one int8 scale per whole row
 * (oracle_act_quant_row / oracle_w4a8_row, the 39936 x 6656 W4A8
 * workload's scheme) and one per (row, group of 32) (oracle_act_quant /
 * oracle_w4a8, the finer variant that passes the pages' outlier case).
 *
 * parity pins: see the oracle tests (exact-rational brute force, invariants,
 * one-hot and all-ones special cases, library matmul cross-check).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define GROUP 32          /* quantization group along K ([T] GROUP_SIZE) */
#define TILE_ROWS 16      /* packed layout: rows per tile                */
#define TILE_K 256        /* packed layout: K per tile (8 groups)        */
#define TILE_BYTES 2432   /* 2048 nibble bytes + 256 scale + 128 zero    */
#define GROUP_TILES 8     /* packed layout: row tiles per 128-row group  */

/* ------------------------------------------------------------------ */
/* bf16 helpers                                                        */
/* ------------------------------------------------------------------ */

/* A bf16 number is the top 16 bits of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Smallest bf16 >= v, for finite v >= 0.  bf16 has 8 significant bits, so
 * for v = f * 2^e (f in [0.5, 1)) the spacing of bf16 numbers at v is
 * 2^(e-8), never finer than the subnormal spacing 2^-133.  ceil() of the
 * exactly scaled value picks the next grid point at or above v. */
static uint16_t bf16_round_up(double v)
{
    if (v == 0.0)
        return 0;
    int e;
    (void)frexp(v, &e);
    int lsb = e - 8;
    if (lsb < -133)
        lsb = -133;
    double m = ceil(ldexp(v, -lsb));
    float r = (float)ldexp(m, lsb); /* at most 8 significant bits: exact */
    uint32_t u;
    memcpy(&u, &r, sizeof u);
    return (uint16_t)(u >> 16);
}

static double clamp_code(double v)
{
    if (v < 0.0)
        return 0.0;
    if (v > 15.0)
        return 15.0;
    return v;
}

/* ------------------------------------------------------------------ */
/* INT4 group-wise asymmetric min-max quantizer  ([T] _packed_with_dense) */
/* ------------------------------------------------------------------ */

/* Quantize one group of 32 consecutive K-elements of one row. */
static void quantize_group(const uint16_t *w, uint8_t *q, uint16_t *s_out,
                           uint8_t *z_out)
{
    double mx = -INFINITY, mn = INFINITY;
    for (int i = 0; i < GROUP; ++i) {
        double v = bf16_to_double(w[i]);
        if (v > mx)
            mx = v;
        if (v < mn)
            mn = v;
    }
    uint16_t sb;
    if (mx == mn) {
        double c = fabs(mx);
        sb = (c == 0.0) ? (uint16_t)0x3F80 /* 1.0 */ : bf16_round_up(c / 15.0);
    } else {
        double range = mx - mn;
        sb = bf16_round_up(range / 15.0);
    }
    double s = bf16_to_double(sb);
    double z = clamp_code(rint(-mn / s));
    for (int i = 0; i < GROUP; ++i) {
        double v = bf16_to_double(w[i]);
        q[i] = (uint8_t)clamp_code(rint(v / s) + z);
    }
    *s_out = sb;
    *z_out = (uint8_t)z;
}

/* W: bf16 [N,K] row-major.  q: u8 [N,K] (one code per byte).
 * s: bf16 [N,K/32].  z: u8 [N,K/32].  K must be a multiple of 32. */
void oracle_quantize_w4(const uint16_t *W, int64_t N, int64_t K, uint8_t *q,
                        uint16_t *s, uint8_t *z)
{
    int64_t G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g)
            quantize_group(W + n * K + g * GROUP, q + n * K + g * GROUP,
                           s + n * G + g, z + n * G + g);
}

/* dequant(q)[n,k] = (q - z) * s, exact in fp64.  What: f64 [N,K]. */
void oracle_dequant_w4(const uint8_t *q, const uint16_t *s, const uint8_t *z,
                       int64_t N, int64_t K, double *What)
{
    int64_t G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int64_t g = k / GROUP;
            What[n * K + k] = ((double)q[n * K + k] - (double)z[n * G + g]) *
                              bf16_to_double(s[n * G + g]);
        }
}

/* ------------------------------------------------------------------ */
/* Packed layout (this library's own, documented in include/w4q.h)     */
/* ------------------------------------------------------------------ */

int64_t oracle_packed_bytes(int64_t N, int64_t K)
{
    if (N < 1 || K < TILE_K || K % TILE_K != 0)
        return 0;
    int64_t groups = (N + TILE_ROWS * GROUP_TILES - 1) / (TILE_ROWS * GROUP_TILES);
    return groups * GROUP_TILES * (K / TILE_K) * TILE_BYTES;
}

/* Byte offset of tile (row tile t, super-block b): tiles are ordered by
 * 128-row group, then super-block, then the group's 8 row tiles, so the 8
 * tiles of one (group, super-block) are contiguous. */
static int64_t tile_offset(int64_t t, int64_t b, int64_t KB)
{
    int64_t g = t / GROUP_TILES, w = t % GROUP_TILES;
    return ((g * KB + b) * GROUP_TILES + w) * TILE_BYTES;
}

/* Byte offset of the nibble holding q[n][k] inside the packed buffer and
 * the bit shift (0 or 4) inside that byte.  Layout of one tile (16 rows
 * n = 16t + 0..15, 256 K k = 256b + 0..255,
 * at tile_offset(t, b)):
 *   nibble region: sub-block sb = kk/64 at 512*sb; lane l at 16*l;
 *   little-endian 32-bit word j = (kk%64)/16 at 4*j; inside the word the
 *   nibble of element (row r + 8*a, col c + 8*e + h) of the 16x16 block
 *   sits at bit 8a + 4e + 16h (a, e, h in {0,1}), with r = l/4 and
 *   c = 2*(l%4). */
static void nibble_position(int64_t n, int64_t k, int64_t KB, int64_t *byte,
                            int *shift)
{
    int64_t t = n / TILE_ROWS, b = k / TILE_K;
    int rr = (int)(n % TILE_ROWS), kk = (int)(k % TILE_K);
    int sb = kk / 64, j = (kk % 64) / 16, col = kk % 16;
    int rlo = rr % 8, a = rr / 8;        /* row = r + 8a                 */
    int e = col / 8, cc = col % 8;       /* col = c + 8e + h             */
    int h = cc % 2, c = cc - h;          /* c = 2*(l%4)                  */
    int l = rlo * 4 + c / 2;
    int bit = 8 * a + 4 * e + 16 * h;
    int64_t tile = tile_offset(t, b, KB);
    *byte = tile + 512 * sb + 16 * l + 4 * j + bit / 8;
    *shift = bit % 8;
}

/* Byte offsets of the bf16 scale and the u8 zero of (row n, group g). */
static void meta_position(int64_t n, int64_t g, int64_t KB, int64_t *sbyte,
                          int64_t *zbyte)
{
    int64_t t = n / TILE_ROWS, b = g / (TILE_K / GROUP);
    int rr = (int)(n % TILE_ROWS), gg = (int)(g % (TILE_K / GROUP));
    int r = rr % 8, half = rr / 8;
    int64_t tile = tile_offset(t, b, KB);
    *sbyte = tile + 2048 + 128 * (gg / 4) + 16 * r + 4 * (gg % 4) + 2 * half;
    *zbyte = tile + 2304 + 16 * r + 2 * gg + half;
}

/* Write q/s/z into the packed layout.  Padding rows (N up to a multiple of
 * 128) are zero. */
void oracle_pack_w4(const uint8_t *q, const uint16_t *s, const uint8_t *z,
                    int64_t N, int64_t K, uint8_t *packed)
{
    int64_t KB = K / TILE_K, G = K / GROUP;
    memset(packed, 0, (size_t)oracle_packed_bytes(N, K));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t byte;
            int shift;
            nibble_position(n, k, KB, &byte, &shift);
            packed[byte] |= (uint8_t)((q[n * K + k] & 0xF) << shift);
        }
        for (int64_t g = 0; g < G; ++g) {
            int64_t sbyte, zbyte;
            meta_position(n, g, KB, &sbyte, &zbyte);
            packed[sbyte] = (uint8_t)(s[n * G + g] & 0xFF);
            packed[sbyte + 1] = (uint8_t)(s[n * G + g] >> 8);
            packed[zbyte] = z[n * G + g];
        }
    }
}

/* Inverse of oracle_pack_w4 for rows 0..N-1. */
void oracle_unpack_w4(const uint8_t *packed, int64_t N, int64_t K, uint8_t *q,
                      uint16_t *s, uint8_t *z)
{
    int64_t KB = K / TILE_K, G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t byte;
            int shift;
            nibble_position(n, k, KB, &byte, &shift);
            q[n * K + k] = (uint8_t)((packed[byte] >> shift) & 0xF);
        }
        for (int64_t g = 0; g < G; ++g) {
            int64_t sbyte, zbyte;
            meta_position(n, g, KB, &sbyte, &zbyte);
            s[n * G + g] =
                (uint16_t)(packed[sbyte] | ((uint16_t)packed[sbyte + 1] << 8));
            z[n * G + g] = packed[zbyte];
        }
    }
}

/* ------------------------------------------------------------------ */
/* W4A16: dequant, then the plain matmul  ([T] _dequant_matmul)        */
/* ------------------------------------------------------------------ */

/* out[m, n - n0] = sum_k x[m,k] * (q[n,k] - z[n,g]) * s[n,g] in fp64, for
 * rows n0 <= n < n1 of the weight.  x: bf16 [M,K].  out: f64 [M, n1-n0]. */
void oracle_w4a16(const uint16_t *x, const uint8_t *q, const uint16_t *s,
                  const uint8_t *z, int64_t M, int64_t N, int64_t K,
                  int64_t n0, int64_t n1, double *out)
{
    (void)N;
    int64_t G = K / GROUP, W = n1 - n0;
#pragma omp parallel for schedule(static)
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t g = k / GROUP;
                double wq = ((double)q[n * K + k] - (double)z[n * G + g]) *
                            bf16_to_double(s[n * G + g]);
                acc += bf16_to_double(x[m * K + k]) * wq;
            }
            out[m * W + (n - n0)] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* Compact metadata: uint8 scale / zero codes on per-row fp16 steps     */
/* ([T] CudaCoalescedInt4Tensor: scale and zero_point uint8 [N, K/32],  */
/* scale_step and zero_point_step float16 [N, 1]; the page prints no    */
/* dequant formula, so this is the reading taken: code x step for both) */
/* ------------------------------------------------------------------ */

/* fp16 bits -> double (exact). */
static double fp16_to_double(uint16_t h)
{
    int e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);
    return (h & 0x8000) ? -v : v;
}

/* Smallest fp16 >= v, for finite v >= 0 (+inf bits past 65504).  An fp16
 * number in [2^e, 2^(e+1)) is a multiple of 2^(e-10); below 2^-14 the
 * subnormals are multiples of 2^-24. */
static uint16_t fp16_round_up(double v)
{
    if (v <= 0.0)
        return 0;
    int e;
    (void)frexp(v, &e); /* v in [2^(e-1), 2^e) */
    int lsb = (e - 1) - 10;
    if (lsb < -24)
        lsb = -24;
    double m = ceil(ldexp(v, -lsb)); /* whole multiples of 2^lsb */
    double r = ldexp(m, lsb);
    if (r > 65504.0)
        return 0x7C00;
    if (r < ldexp(1.0, -14))
        return (uint16_t)m; /* subnormal: the mantissa field is m */
    int re;
    double f = frexp(r, &re); /* r = f * 2^re, f in [0.5, 1) */
    uint16_t mant = (uint16_t)(ldexp(f, 11) - 1024.0);
    return (uint16_t)(((re - 1 + 15) << 10) | mant);
}

/* One row n of W (bf16 [K]) in the compact format:
 *   per group g: mn, mx; s*_g = (mx - mn) / 15 (a constant group c:
 *   |c| / 15, or 1 for c = 0);
 *   scale step ds = RU_fp16(max_g s*_g / 255); scale code
 *   sc_g = min(255, ceil(s*_g / ds)); scale s_g = sc_g * ds (>= s*_g);
 *   z*_g = clamp(-mn / s_g, 0, 15); zero step dz = RU_fp16(max_g z*_g / 255)
 *   (1 when every z*_g is 0); zero code zc_g = min(255, rint(z*_g / dz));
 *   zero z_g = zc_g * dz;
 *   q = clamp(rint(w / s_g + z_g), 0, 15)  (fp64, in this order);
 *   dequant(q) = (q - z_g) * s_g.
 * steps[2n] = ds, steps[2n + 1] = dz (fp16 bits). */
static void quantize_row_c(const uint16_t *w, int64_t K, uint8_t *q, uint8_t *sc,
                           uint8_t *zc, uint16_t *steps)
{
    int64_t G = K / GROUP;
    double smax = 0.0;
    for (int64_t g = 0; g < G; ++g) {
        double mx = -INFINITY, mn = INFINITY;
        for (int i = 0; i < GROUP; ++i) {
            double v = bf16_to_double(w[g * GROUP + i]);
            if (v > mx) mx = v;
            if (v < mn) mn = v;
        }
        double st = (mx == mn) ? (mx == 0.0 ? 1.0 : fabs(mx) / 15.0) : (mx - mn) / 15.0;
        if (st > smax)
            smax = st;
    }
    uint16_t dsb = fp16_round_up(smax / 255.0);
    double ds = fp16_to_double(dsb);
    double zmax = 0.0;
    for (int64_t g = 0; g < G; ++g) {
        double mx = -INFINITY, mn = INFINITY;
        for (int i = 0; i < GROUP; ++i) {
            double v = bf16_to_double(w[g * GROUP + i]);
            if (v > mx) mx = v;
            if (v < mn) mn = v;
        }
        double st = (mx == mn) ? (mx == 0.0 ? 1.0 : fabs(mx) / 15.0) : (mx - mn) / 15.0;
        double c = ceil(st / ds);
        if (c > 255.0) c = 255.0;
        if (c < 1.0) c = 1.0;
        sc[g] = (uint8_t)c;
        double zs = clamp_code(-mn / ((double)sc[g] * ds));
        if (zs > zmax)
            zmax = zs;
    }
    uint16_t dzb = zmax > 0.0 ? fp16_round_up(zmax / 255.0) : (uint16_t)0x3C00; /* 1.0 */
    double dz = fp16_to_double(dzb);
    for (int64_t g = 0; g < G; ++g) {
        double mn = INFINITY;
        for (int i = 0; i < GROUP; ++i) {
            double v = bf16_to_double(w[g * GROUP + i]);
            if (v < mn) mn = v;
        }
        double s = (double)sc[g] * ds;
        double zs = clamp_code(-mn / s);
        double c = rint(zs / dz);
        if (c > 255.0) c = 255.0;
        zc[g] = (uint8_t)c;
        double z = (double)zc[g] * dz;
        for (int i = 0; i < GROUP; ++i) {
            double t = bf16_to_double(w[g * GROUP + i]) / s;
            q[g * GROUP + i] = (uint8_t)clamp_code(rint(t + z));
        }
    }
    steps[0] = dsb;
    steps[1] = dzb;
}

/* W bf16 [N,K] -> q u8 [N,K], sc u8 [N,K/32], zc u8 [N,K/32], steps fp16 [N][2]. */
void oracle_quantize_w4c(const uint16_t *W, int64_t N, int64_t K, uint8_t *q, uint8_t *sc,
                         uint8_t *zc, uint16_t *steps)
{
    int64_t G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        quantize_row_c(W + n * K, K, q + n * K, sc + n * G, zc + n * G, steps + 2 * n);
}

/* dequant(q)[n,k] = (q - zc * dz_n) * (sc * ds_n), exact in fp64. */
void oracle_dequant_w4c(const uint8_t *q, const uint8_t *sc, const uint8_t *zc,
                        const uint16_t *steps, int64_t N, int64_t K, double *What)
{
    int64_t G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double ds = fp16_to_double(steps[2 * n]), dz = fp16_to_double(steps[2 * n + 1]);
        for (int64_t k = 0; k < K; ++k) {
            int64_t g = k / GROUP;
            double s = (double)sc[n * G + g] * ds, z = (double)zc[n * G + g] * dz;
            What[n * K + k] = ((double)q[n * K + k] - z) * s;
        }
    }
}

/* Compact packed layout (this library's own): tiles of 16 rows x 256 K as
 * in the standard layout but 2304 bytes, [2048 B codes][128 B scale codes]
 * [128 B zero codes], the code pair (row r, row r + 8) of group g at
 * 2048 + 16 r + 2 g (scales) and 2176 + 16 r + 2 g (zeros); after all
 * tiles, the fp16 steps (ds, dz) of every row (N padded to 128, padding
 * zero). */
#define CTILE_BYTES 2304

int64_t oracle_packed_bytes_c(int64_t N, int64_t K)
{
    if (N < 1 || K < TILE_K || K % TILE_K != 0)
        return 0;
    int64_t groups = (N + TILE_ROWS * GROUP_TILES - 1) / (TILE_ROWS * GROUP_TILES);
    return groups * GROUP_TILES * (K / TILE_K) * CTILE_BYTES + groups * 128 * 4;
}

static int64_t ctile_offset(int64_t t, int64_t b, int64_t KB)
{
    int64_t g = t / GROUP_TILES, w = t % GROUP_TILES;
    return ((g * KB + b) * GROUP_TILES + w) * CTILE_BYTES;
}

/* The same nibble placement inside a tile as the standard layout. */
static void cnibble_position(int64_t n, int64_t k, int64_t KB, int64_t *byte, int *shift)
{
    int64_t t = n / TILE_ROWS, b = k / TILE_K;
    int rr = (int)(n % TILE_ROWS), kk = (int)(k % TILE_K);
    int sb = kk / 64, j = (kk % 64) / 16, col = kk % 16;
    int rlo = rr % 8, a = rr / 8;
    int e = col / 8, cc = col % 8;
    int h = cc % 2, c = cc - h;
    int l = rlo * 4 + c / 2;
    int bit = 8 * a + 4 * e + 16 * h;
    *byte = ctile_offset(t, b, KB) + 512 * sb + 16 * l + 4 * j + bit / 8;
    *shift = bit % 8;
}

void oracle_pack_w4c(const uint8_t *q, const uint8_t *sc, const uint8_t *zc,
                     const uint16_t *steps, int64_t N, int64_t K, uint8_t *packed)
{
    int64_t KB = K / TILE_K, G = K / GROUP;
    int64_t total = oracle_packed_bytes_c(N, K);
    int64_t tiles = total - ((N + 127) / 128) * 128 * 4;
    memset(packed, 0, (size_t)total);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t byte;
            int shift;
            cnibble_position(n, k, KB, &byte, &shift);
            packed[byte] |= (uint8_t)((q[n * K + k] & 0xF) << shift);
        }
        int64_t t = n / TILE_ROWS;
        int rr = (int)(n % TILE_ROWS), r = rr % 8, half = rr / 8;
        for (int64_t g = 0; g < G; ++g) {
            int64_t base = ctile_offset(t, g / 8, KB);
            int gg = (int)(g % 8);
            packed[base + 2048 + 16 * r + 2 * gg + half] = sc[n * G + g];
            packed[base + 2176 + 16 * r + 2 * gg + half] = zc[n * G + g];
        }
        memcpy(packed + tiles + 4 * n, steps + 2 * n, 4);
    }
}

void oracle_unpack_w4c(const uint8_t *packed, int64_t N, int64_t K, uint8_t *q, uint8_t *sc,
                       uint8_t *zc, uint16_t *steps)
{
    int64_t KB = K / TILE_K, G = K / GROUP;
    int64_t tiles = oracle_packed_bytes_c(N, K) - ((N + 127) / 128) * 128 * 4;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t byte;
            int shift;
            cnibble_position(n, k, KB, &byte, &shift);
            q[n * K + k] = (uint8_t)((packed[byte] >> shift) & 0xF);
        }
        int64_t t = n / TILE_ROWS;
        int rr = (int)(n % TILE_ROWS), r = rr % 8, half = rr / 8;
        for (int64_t g = 0; g < G; ++g) {
            int64_t base = ctile_offset(t, g / 8, KB);
            int gg = (int)(g % 8);
            sc[n * G + g] = packed[base + 2048 + 16 * r + 2 * gg + half];
            zc[n * G + g] = packed[base + 2176 + 16 * r + 2 * gg + half];
        }
        memcpy(steps + 2 * n, packed + tiles + 4 * n, 4);
    }
}

/* out[m, n - n0] = sum_k x[m,k] * (q - zc dz) * (sc ds) in fp64. */
void oracle_w4a16c(const uint16_t *x, const uint8_t *q, const uint8_t *sc, const uint8_t *zc,
                   const uint16_t *steps, int64_t M, int64_t N, int64_t K, int64_t n0,
                   int64_t n1, double *out)
{
    (void)N;
    int64_t G = K / GROUP, W = n1 - n0;
#pragma omp parallel for schedule(static)
    for (int64_t n = n0; n < n1; ++n) {
        double ds = fp16_to_double(steps[2 * n]), dz = fp16_to_double(steps[2 * n + 1]);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t g = k / GROUP;
                double wq = ((double)q[n * K + k] - (double)zc[n * G + g] * dz) *
                            ((double)sc[n * G + g] * ds);
                acc += bf16_to_double(x[m * K + k]) * wq;
            }
            out[m * W + (n - n0)] = acc;
        }
    }
}

/* ------------------------------------------------------------------ */
/* W4A8: symmetric int8 activations, one scale per (row, group of 32)   */
/* ([T] W4A8 bucket kernels, Int4QuantizedGemmPrecisionTest)            */
/* ------------------------------------------------------------------ */

/* Per row m and group g of 32 columns, in IEEE fp32 (round to nearest even):
 *   a = max_{k in g} |x[m,k]|,  sx[m,g] = a / 127,
 *   xq[m,k] = clamp(rint(x[m,k] / sx[m,g]), -127, 127),  xq = 0 when a == 0.
 * One scale per group keeps an outlier channel from flattening the rest of
 * its row (the precision test's outlier case fails with one scale per row).
 * fp32 is the precision of the decision on both sides: x / sx with an fp32
 * sx can fall within an fp64 rounding of a half-integer. */
void oracle_act_quant(const uint16_t *x, int64_t M, int64_t K, int8_t *xq,
                      float *sx)
{
    int64_t G = K / GROUP;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t g = 0; g < G; ++g) {
            float a = 0.0f;
            for (int64_t i = 0; i < GROUP; ++i) {
                float v = fabsf(bf16_to_float(x[m * K + g * GROUP + i]));
                if (v > a)
                    a = v;
            }
            volatile float sxg = a / 127.0f;
            sx[m * G + g] = sxg;
            for (int64_t i = 0; i < GROUP; ++i) {
                int64_t k = g * GROUP + i;
                if (a == 0.0f) {
                    xq[m * K + k] = 0;
                    continue;
                }
                volatile float t = bf16_to_float(x[m * K + k]) / sxg;
                float r = rintf(t);
                if (r > 127.0f)
                    r = 127.0f;
                if (r < -127.0f)
                    r = -127.0f;
                xq[m * K + k] = (int8_t)r;
            }
        }
}

/* The per-row variant: one symmetric int8 scale for each whole activation
 * row, the scheme of the 39936 x 6656 W4A8 workload ("per-row symmetric
 * int8 (scale=absmax/127)").  Per row m, in IEEE fp32 (round to nearest
 * even):
 *   a = max_k |x[m,k]|,  sx[m] = a / 127,
 *   xq[m,k] = clamp(rint(x[m,k] / sx[m]), -127, 127),  xq = 0 when a == 0.
 * The same fp32 decision rule as oracle_act_quant, over the row instead of
 * the group.  sx: f32 [M]. */
void oracle_act_quant_row(const uint16_t *x, int64_t M, int64_t K, int8_t *xq,
                          float *sx)
{
    for (int64_t m = 0; m < M; ++m) {
        float a = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = fabsf(bf16_to_float(x[m * K + k]));
            if (v > a)
                a = v;
        }
        volatile float sxm = a / 127.0f;
        sx[m] = sxm;
        for (int64_t k = 0; k < K; ++k) {
            if (a == 0.0f) {
                xq[m * K + k] = 0;
                continue;
            }
            volatile float t = bf16_to_float(x[m * K + k]) / sxm;
            float r = rintf(t);
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            xq[m * K + k] = (int8_t)r;
        }
    }
}

/* D[m][n][g] = sum_{k in group g} (q[n,k] - z[n,g]) * xq[m,k], exact int. */
void oracle_w4a8_group_dots(const int8_t *xq, const uint8_t *q,
                            const uint8_t *z, int64_t M, int64_t N, int64_t K,
                            int32_t *D)
{
    int64_t G = K / GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t g = 0; g < G; ++g) {
                int32_t acc = 0;
                for (int64_t i = 0; i < GROUP; ++i) {
                    int64_t k = g * GROUP + i;
                    acc += ((int32_t)q[n * K + k] - (int32_t)z[n * G + g]) *
                           (int32_t)xq[m * K + k];
                }
                D[(m * N + n) * G + g] = acc;
            }
}

/* out[m, n - n0] = sum_g sx[m,g] * s[n,g] * D[m][n][g] in fp64. */
void oracle_w4a8(const int8_t *xq, const float *sx, const uint8_t *q,
                 const uint16_t *s, const uint8_t *z, int64_t M, int64_t N,
                 int64_t K, int64_t n0, int64_t n1, double *out)
{
    (void)N;
    int64_t G = K / GROUP, W = n1 - n0;
#pragma omp parallel for schedule(static)
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                int64_t d = 0;
                for (int64_t i = 0; i < GROUP; ++i) {
                    int64_t k = g * GROUP + i;
                    d += ((int64_t)q[n * K + k] - (int64_t)z[n * G + g]) *
                         (int64_t)xq[m * K + k];
                }
                acc += (double)sx[m * G + g] * bf16_to_double(s[n * G + g]) * (double)d;
            }
            out[m * W + (n - n0)] = acc;
        }
}

/* Per-row W4A8: out[m, n - n0] = sx[m] * sum_g s[n,g] * D[m][n][g] in
 * fp64, with D the exact integer group dots and sx: f32 [M] from
 * oracle_act_quant_row. */
void oracle_w4a8_row(const int8_t *xq, const float *sx, const uint8_t *q,
                     const uint16_t *s, const uint8_t *z, int64_t M, int64_t N,
                     int64_t K, int64_t n0, int64_t n1, double *out)
{
    (void)N;
    int64_t G = K / GROUP, W = n1 - n0;
#pragma omp parallel for schedule(static)
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                int64_t d = 0;
                for (int64_t i = 0; i < GROUP; ++i) {
                    int64_t k = g * GROUP + i;
                    d += ((int64_t)q[n * K + k] - (int64_t)z[n * G + g]) *
                         (int64_t)xq[m * K + k];
                }
                acc += bf16_to_double(s[n * G + g]) * (double)d;
            }
            out[m * W + (n - n0)] = (double)sx[m] * acc;
        }
}

/* ------------------------------------------------------------------ */
/* W8: int8 weight-only linear  ([G] WeightOnlyInt8Linear.forward)     */
/* ------------------------------------------------------------------ */

/* out[m, n - n0] = (sum_k x[m,k] * W[n,k]) * scales[n] in fp64.
 * x: bf16 [M,K]; W: int8 [N,K]; scales: bf16 [N]. */
void oracle_w8(const uint16_t *x, const int8_t *W, const uint16_t *scales,
               int64_t M, int64_t N, int64_t K, int64_t n0, int64_t n1,
               double *out)
{
    (void)N;
    int64_t Wd = n1 - n0;
#pragma omp parallel for schedule(static)
    for (int64_t n = n0; n < n1; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += bf16_to_double(x[m * K + k]) * (double)W[n * K + k];
            out[m * Wd + (n - n0)] = acc * bf16_to_double(scales[n]);
        }
}

/* ------------------------------------------------------------------ */
/* threads                                                             */
/* ------------------------------------------------------------------ */

int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
