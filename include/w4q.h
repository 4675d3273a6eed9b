/*
 * w4q.h -- C ABI of the GB300 (sm_103a) weight-only quantized linear layer
 *
 *     out[M,N] = x[M,K] . dequant(Wq)[N,K]^T        (decode sizes, M <= 64)
 *
 * Three forms, as on the source pages:
 *   W4A16  INT4 weights, group-wise asymmetric min-max (group 32 along K,
 *          one scale and one zero point per group), bf16 activations.
 *          ("test_int4_quantized_gemm.py": _packed_with_dense with
 *          QuantConfig(bits=4, group_size=32, symmetric=False,
 *          method="min_max"); the dequant + F.linear reference.)
 *   W4A8   the same weights, activations quantized to symmetric int8
 *          inside the call, with one scale per whole row (w4a8_gemm_rowscale,
 *          scale = max|x| / 127 over the row) or one per (row, group of 32)
 *          (w4a8_gemm); each group's dot product is an exact integer, scaled
 *          in fp32.  ("test_int4_quantized_gemm.py": the W4A8 bucket kernels
 *          and Int4QuantizedGemmPrecisionTest.)
 *   W8     int8 weights with one bf16 scale per output row.
 *          ("gpt-fast issue #114": WeightOnlyInt8Linear.forward,
 *          F.linear(x, W.to(bf16)) * scales, and its fused reduction.)
 *
 * Conventions (every entry point):
 *   - Pointers marked "device" are device pointers owned by the caller; the
 *     library never frees, retains or allocates memory, and keeps no state
 *     except a per-device SM-count cache and two module variables (the
 *     device-side error word and the no-allocation scratch array).  Their
 *     device addresses are cached together with the id of the CUDA context
 *     they were looked up in and looked up again when another context is
 *     current, so calls after cudaDeviceReset (or any teardown and re-creation
 *     of the context) use the new context's copies; an error word set in a
 *     context that was torn down is lost with it.
 *   - Device pointers must be 16-byte aligned, else W4Q_ERR_MISALIGNED.
 *     Outputs must not alias inputs.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream) and never synchronize, except
 *     w4q_device_error.  They may be captured in a CUDA graph.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns a status, launches nothing and leaves the
 *     outputs untouched.  A failed launch returns W4Q_ERR_CUDA.  No call
 *     aborts or exits the process.
 *   - Results are bitwise reproducible for a given (M, N, K, split, device
 *     SM count): reductions run in a fixed order, with no floating-point
 *     atomics.  ("test_int4_quantized_gemm.py": repeated calls and CUDA
 *     graph replay are bitwise equal to eager.)
 *   - W4 shapes: 1 <= M <= 64, N >= 1, K a positive multiple of 256
 *     ("test_int4_quantized_gemm.py", Int4QuantizedGemmLegalityTest: K must
 *     be a multiple of 256), group == 32 (the only supported group size).
 *   - Non-finite inputs give unspecified (but memory-safe) outputs.
 *
 * Packed W4 layout (this library's own; the pages' storage is prior art):
 *   Rows are grouped in tiles of 16 and tiles in groups of 8 (128 rows; N
 *   is padded up to a multiple of 128 with all-zero rows), K in super-blocks
 *   of 256 (8 groups).  Tile (t, b), t < 8*ceil(N/128), b < K/256, is 2432
 *   bytes at offset (((t/8)*(K/256) + b)*8 + t%8)*2432, so the 8 tiles of a
 *   (128-row group, super-block) pair are one contiguous 19456-byte block:
 *     [0, 2048)     4-bit codes q.  Sub-block sb = kk/64 (kk = k - 256b) at
 *                   512*sb; "lane" l in 0..31 at +16*l; little-endian 32-bit
 *                   word j = (kk%64)/16 at +4*j.  Inside word j, with
 *                   r = l/4 and c = 2*(l%4), the nibble at bit 8a + 4e + 16h
 *                   (a, e, h in 0..1) is the code of row 16t + r + 8a and
 *                   column 256b + 64sb + 16j + c + 8e + h.  (One 16-byte
 *                   lane chunk holds the four bf16 A fragments of four
 *                   m16n8k16 MMAs for that lane; masking a word with
 *                   0x000F000F / 0x00F000F0, before and after a shift by 8,
 *                   yields them as exact multiples of a power of two.)
 *     [2048, 2304)  bf16 scales s.  The pair (s[16t+r][8b+g],
 *                   s[16t+r+8][8b+g]) is at 2048 + 128*(g/4) + 16*r +
 *                   4*(g%4), row r first (r in 0..7, g in 0..7).
 *     [2304, 2432)  u8 zero points z, the pair (z[16t+r][8b+g],
 *                   z[16t+r+8][8b+g]) at 2304 + 16*r + 2*g.
 *   Every field starts on a 16-byte boundary, so a CTA streams a whole
 *   128 x 256 block with one 1-D bulk copy and each lane reads 16-byte
 *   chunks.
 *
 * Quantizer (w4_pack_weights), per row n and group g of 32 columns, with
 * max/min over the group:
 *   s = the smallest bf16 >= fl64(fl64(max - min) / 15)   (round up, so
 *       |w - dequant| <= s/2 whenever min <= 0 <= max);
 *       a constant group c uses s = RU_bf16(|c| / 15), or 1.0 if c == 0;
 *   z = clamp(rint(-min / s), 0, 15);  q = clamp(rint(w / s) + z, 0, 15)
 *       (rint = round half to even; z and q use the stored bf16 s);
 *   dequant(q) = (q - z) * s.
 */
#ifndef W4Q_H
#define W4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4Q_OK = 0,
    W4Q_ERR_INVALID_ARG = 1,  /* null pointer, negative or zero size      */
    W4Q_ERR_UNSUPPORTED = 2,  /* M, K, group or split outside the ranges  */
    W4Q_ERR_MISALIGNED = 3,   /* a device pointer not 16-byte aligned     */
    W4Q_ERR_WORKSPACE = 4,    /* workspace missing or too small           */
    W4Q_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed     */
    W4Q_ERR_DEVICE = 6        /* a kernel reported a bounded-wait timeout */
} w4q_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *w4q_status_string(int status);

/* ---------------------------------------------------------------- W4 --- */

/* Bytes of the packed W4 buffer for an [N,K] weight:
 * ceil(N/128)*8*(K/256)*2432.  Returns 0 when (N, K, group) is unsupported. */
size_t w4_packed_bytes(int64_t N, int64_t K, int group);

/* Quantize a bf16 weight and write it in the packed layout above.
 *   W_bf16  device, bf16 [N,K] row-major (read only)
 *   packed  device, w4_packed_bytes(N,K,group) bytes (written, fully)
 * Defined by "test_int4_quantized_gemm.py", _packed_with_dense (INT4,
 * group 32, asymmetric min-max); the rounding choices are in the header
 * comment.  One launch; no workspace. */
int w4_pack_weights(const void *W_bf16, int64_t N, int64_t K, int group,
                    void *packed, void *stream);

/* Inverse view of the packed buffer, for tests and tools.
 *   q      device, u8 [N,K], one code per byte (written)
 *   scale  device, bf16 [N,K/32] (written)
 *   zero   device, u8 [N,K/32] (written)
 * Padding rows are not written. */
int w4_unpack_weights(const void *packed, int64_t N, int64_t K, int group,
                      uint8_t *q, void *scale_bf16, uint8_t *zero,
                      void *stream);

/* Workspace bytes needed by w4a16_gemm, w4a8_gemm and w4a8_gemm_rowscale
 * for these sizes on the current device with the library's own split
 * choice (0 if none is needed; a call on the cluster kernel, the usual case
 * at M <= 8, needs none).  One buffer of this size serves all three. */
size_t w4_workspace_bytes(int64_t M, int64_t N, int64_t K, int group);

/* Same, for an explicit split_k (see w4a16_gemm_split); 0 if unsupported. */
size_t w4_workspace_bytes_split(int64_t M, int64_t N, int64_t K, int group,
                                int split_k);

/* The split the library picks for a W4A16 call of these sizes on the
 * current device: 0 = balanced stream-K partition over all SMs, s >= 1 =
 * fixed K split (at M <= 8: s CTAs of one thread-block cluster per 128-row
 * group, where the call fits the cluster kernel).  At M <= 8 the choice is
 * the measured one of the library's split table when it lists the call for
 * this GPU's SM count (tune_splits.py), else a cost model's. */
int w4_split_choice(int64_t M, int64_t N, int64_t K, int group);

/* Number of kernels one call with these sizes launches on the current
 * device, for w4a8 = 0 (w4a16_gemm), 1 (w4a8_gemm) or 2
 * (w4a8_gemm_rowscale): 1 for a call on the cluster kernel (M <= 8, the
 * activations prepared and the split-K partials summed inside it);
 * otherwise a prologue (split-K counter reset; W4A8: also the activation
 * quantizer; W4A16 at M >= 9: the tensor-core operand layout), the main
 * kernel, and for W4A16 at M >= 9 with row groups split over several CTAs
 * the launch that sums their fp32 partials.  -1 when unsupported. */
int w4_kernel_launches(int64_t M, int64_t N, int64_t K, int group, int w4a8);

/* out = x . dequant(packed)^T, W4A16.
 *   x          device, bf16 [M,K] row-major
 *   packed     device, from w4_pack_weights(N, K)
 *   out        device, bf16 [M,N] row-major (written)
 *   workspace  device scratch of >= w4_workspace_bytes(M,N,K,group) bytes
 *              (may be NULL when that is 0); contents are clobbered.
 * Accumulates in fp32: for M <= 8 per group, sum_k (q - z) * x exactly in
 * the tensor core, then acc += s * sum (and, where K is split over the CTAs
 * of a cluster, the CTAs' sums added in rank order); for M >= 9 the dequantized weight
 * is rounded once to bf16 ((q - z) * s) and accumulated over all of K on
 * the tcgen05 tensor core.
 * out = bf16_RN(acc).  Defined by "test_int4_quantized_gemm.py", the
 * dequant + F.linear reference. */
int w4a16_gemm(const void *x_bf16, const void *packed, void *out_bf16,
               int64_t M, int64_t N, int64_t K, int group, void *workspace,
               size_t workspace_bytes, void *stream);

/* As w4a16_gemm with an explicit K partition: split_k = s >= 1 splits each
 * 16*8-row tile group's K range into s contiguous parts of whole 256-wide
 * super-blocks (legal iff s <= K/256, "test_int4_quantized_gemm.py",
 * Int4QuantizedGemmRulesTest: one 256-wide K tile per split), partials are
 * summed in fixed order; split_k = 0 is the balanced stream-K partition.
 * At M <= 8, s in 1..8 runs on the cluster kernel (s CTAs per cluster,
 * partials summed over distributed shared memory, no workspace) whenever
 * the CTA's slice of prepared activations fits its shared memory, and on
 * the stream-K kernel with a fixed split otherwise.  The library's own
 * choice is described at w4_split_choice; on the tensor-core path (M >= 9)
 * it is stream-K, or 1 (whole K per CTA, no partial-sum launch) with at
 * most 4 super-blocks and no more 256-row pairs than SMs.  Illegal s
 * returns W4Q_ERR_UNSUPPORTED. */
int w4a16_gemm_split(const void *x_bf16, const void *packed, void *out_bf16,
                     int64_t M, int64_t N, int64_t K, int group, int split_k,
                     void *workspace, size_t workspace_bytes, void *stream);

/* W4A16 for callers that cannot allocate device memory at all.  (The pages
 * have no counterpart; this is a property of this library's interface.)
 * Some callers may not call cudaMalloc on the path that runs a layer and
 * have no workspace to give: code running while a stream is captured into
 * a CUDA graph, hosts that plan all device memory ahead of time (embedded
 * or real-time loops that must not pause in an allocator), plug-ins whose
 * device memory belongs to a host framework.  This call computes exactly
 * what w4a16_gemm computes, with the same kernels, but takes its scratch
 * from one array of W4Q_NOALLOC_SCRATCH_BYTES (16 MiB) of device memory
 * that the library itself holds on every GPU that loads it, until exit.
 *   x, packed, out, M, N, K, group, stream: as w4a16_gemm.
 * Returns W4Q_ERR_UNSUPPORTED when the call would need more scratch than
 * the array holds (large M together with a wide split-K partition; see
 * w4_workspace_bytes for the amount), besides the w4a16_gemm errors.  It
 * calls no allocator of any kind.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress), so make that first
 * call before any stream capture.  Every call on a device shares the one
 * array: calls that may overlap on the GPU (other streams, other host
 * threads) race and give wrong results; serialize them.  Each call resets
 * the part of the array that must start at zero itself. */
#define W4Q_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int w4a16_gemm_noalloc(const void *x_bf16, const void *packed, void *out_bf16, int64_t M,
                       int64_t N, int64_t K, int group, void *stream);

/* out = x . dequant(packed)^T, W4A8: per row m and group g of 32 columns,
 * sx[m,g] = fp32(max_{k in g} |x| / 127), xq = clamp(rint(x / sx[m,g]),
 * -127, 127) in IEEE fp32 (xq = 0 when the group's max is 0); per group
 * D = sum_k (q - z) * xq, an exact integer (|D| <= 60960);
 * acc = sum_g sx[m,g] * s_g * D_g in fp32; out = bf16_RN(acc).  One scale
 * per group keeps an outlier channel from flattening its row: the outlier
 * case of Int4QuantizedGemmPrecisionTest ("test_int4_quantized_gemm.py")
 * fails with one scale per row.
 * Arguments as w4a16_gemm with 1 <= M <= 8 (the pages' W4A8 buckets are
 * 1..4); the workspace is needed only where w4_workspace_bytes says so (the
 * stream-K kernel keeps the prepared activations there; the cluster kernel
 * keeps them in shared memory). */
int w4a8_gemm(const void *x_bf16, const void *packed, void *out_bf16,
              int64_t M, int64_t N, int64_t K, int group, void *workspace,
              size_t workspace_bytes, void *stream);

int w4a8_gemm_split(const void *x_bf16, const void *packed, void *out_bf16,
                    int64_t M, int64_t N, int64_t K, int group, int split_k,
                    void *workspace, size_t workspace_bytes, void *stream);

/* out = x . dequant(packed)^T, W4A8 with one activation scale per row:
 * per row m, sx[m] = fp32(max_k |x[m,k]| / 127), xq = clamp(rint(x /
 * sx[m]), -127, 127) in IEEE fp32 (xq = 0 for an all-zero row); per group
 * D = sum_k (q - z) * xq, an exact integer; acc = sum_g (sx[m] * s_g) * D_g
 * in fp32; out = bf16_RN(acc).  Symmetric int8 activations with the scale
 * absmax / 127 per row, as the W4A8 bucket kernels of
 * "test_int4_quantized_gemm.py" are exercised on gaussian activations
 * (Int4QuantizedGemmPrecisionTest: mean |a8 - a16| / mean |a16| < 0.02).
 * A few large outlier channels flatten the rest of their row under this
 * rule; w4a8_gemm (one scale per group of 32) is the variant for them.
 * Arguments, limits and workspace as w4a8_gemm. */
int w4a8_gemm_rowscale(const void *x_bf16, const void *packed, void *out_bf16,
                       int64_t M, int64_t N, int64_t K, int group,
                       void *workspace, size_t workspace_bytes, void *stream);

int w4a8_gemm_rowscale_split(const void *x_bf16, const void *packed,
                             void *out_bf16, int64_t M, int64_t N, int64_t K,
                             int group, int split_k, void *workspace,
                             size_t workspace_bytes, void *stream);

/* The W4A8 activation quantizer alone (the rule w4a8_gemm applies).
 *   xq  device, int8 [M,K] (written);  sx  device, f32 [M][K/32] (written). */
int w4a8_quantize_act(const void *x_bf16, int64_t M, int64_t K, int8_t *xq,
                      float *sx, void *stream);

/* The per-row W4A8 activation quantizer alone (the rule w4a8_gemm_rowscale
 * applies).  xq  device, int8 [M,K] (written);  sx  device, f32 [M]. */
int w4a8_quantize_act_rowscale(const void *x_bf16, int64_t M, int64_t K,
                               int8_t *xq, float *sx, void *stream);

/* The exact W4A8 group dot products, for bit-exact checks (1 <= M <= 8).
 *   D          device, int32 [M][N][K/32] (written)
 *   workspace  device, >= w4_workspace_bytes(M,N,K,group) bytes
 * Uses the same activation quantizer and the same tensor-core group dot as
 * w4a8_gemm. */
int w4a8_group_dots(const void *x_bf16, const void *packed, int64_t M,
                    int64_t N, int64_t K, int group, int32_t *D,
                    void *workspace, size_t workspace_bytes, void *stream);

/* As w4a8_group_dots, with the per-row activation quantizer of
 * w4a8_gemm_rowscale. */
int w4a8_group_dots_rowscale(const void *x_bf16, const void *packed, int64_t M,
                             int64_t N, int64_t K, int group, int32_t *D,
                             void *workspace, size_t workspace_bytes,
                             void *stream);

/* ------------------------------------------------- compact W4 metadata --- */

/* The compact metadata of "test_int4_quantized_gemm.py"'s
 * CudaCoalescedInt4Tensor: per (row, group of 32) a uint8 scale code sc and
 * a uint8 zero code zc, per row two float16 steps ds and dz (the page's
 * scale / zero_point and scale_step / zero_point_step).  The page prints no
 * dequant formula; this library reads both as code x step:
 *   scale = sc * ds,  zero = zc * dz,  dequant(q) = (q - zero) * scale,
 * 2 bytes per group instead of the standard 3 (0.5625 bytes per weight).
 * Quantizer, per row n, in fp64 and in this order:
 *   s*_g = (max - min) / 15 (a constant group c: |c| / 15, or 1 if c == 0);
 *   ds = the smallest fp16 >= max_g s*_g / 255;
 *   sc_g = min(255, max(1, ceil(s*_g / ds)));  so scale >= s*_g;
 *   z*_g = clamp(-min / scale_g, 0, 15);
 *   dz = the smallest fp16 >= max_g z*_g / 255 (1.0 when every z*_g is 0);
 *   zc_g = min(255, rint(z*_g / dz));
 *   q = clamp(rint(w / scale_g + zero_g), 0, 15).
 * For groups with min <= 0 <= max, |w - dequant(q)| <= scale_g / 2.  Rows
 * whose group ranges overflow fp16 steps (max - min above ~1.2e8) or whose
 * steps fall below the fp16 subnormal range lose that bound.
 * Packed layout: tiles of 2304 bytes in the order of the standard layout
 * (offset (((t/8)*(K/256) + b)*8 + t%8)*2304), each
 *   [0, 2048)     the 4-bit codes, placed as in the standard layout;
 *   [2048, 2176)  scale codes: (sc[16t+r][8b+g], sc[16t+r+8][8b+g]) at
 *                 2048 + 16*r + 2*g;
 *   [2176, 2304)  zero codes, the same pairs at 2176 + 16*r + 2*g;
 * then, after all tiles, the fp16 pair (ds, dz) of every row n at 4*n (N
 * padded to a multiple of 128; padding rows all zero). */

/* Bytes of the compact packed buffer: ceil(N/128)*(8*(K/256)*2304 + 512);
 * 0 when unsupported. */
size_t w4_packed_bytes_compact(int64_t N, int64_t K, int group);

/* Quantize a bf16 weight [N,K] (device) into the compact format (device,
 * w4_packed_bytes_compact bytes, written fully).  Two launches. */
int w4_pack_weights_compact(const void *W_bf16, int64_t N, int64_t K, int group,
                            void *packed, void *stream);

/* Inverse view: q u8 [N,K], scale codes u8 [N,K/32], zero codes u8
 * [N,K/32], steps fp16 [N][2] (ds, dz), all device, written. */
int w4_unpack_weights_compact(const void *packed, int64_t N, int64_t K, int group,
                              uint8_t *q, uint8_t *scale_codes,
                              uint8_t *zero_codes, void *steps_fp16,
                              void *stream);

/* out = x . dequant(packed)^T with the compact metadata, W4A16, 1 <= M <= 8
 * (x, out as w4a16_gemm; packed from w4_pack_weights_compact).  Runs on the
 * cluster kernel: per group the scale sc*ds and the zero zc*dz are formed
 * exactly in fp32 and enter the fp32 update as in w4a16_gemm.  No
 * workspace; W4Q_ERR_UNSUPPORTED for M > 8 or when no K split fits the
 * kernel's shared memory (K above roughly 40960 at M <= 4). */
int w4a16_gemm_compact(const void *x_bf16, const void *packed, void *out_bf16,
                       int64_t M, int64_t N, int64_t K, int group, void *stream);

/* ---------------------------------------------------------------- W8 --- */

/* out[m,n] = bf16_RN(fp32(sum_k x[m,k] * W[n,k]) * scales[n]), one rounding
 * ("gpt-fast issue #114": WeightOnlyInt8Linear.forward and the fused
 * int8 -> fp32 reduction).
 *   x       device, bf16 [M,K] row-major, 1 <= M <= 4
 *   W       device, int8 [N,K] row-major, K a positive multiple of 16
 *   scales  device, bf16 [N]
 *   out     device, bf16 [M,N] (written)
 * No workspace. */
int w8_gemv(const void *x_bf16, const int8_t *W, const void *scales_bf16,
            void *out_bf16, int64_t M, int64_t N, int64_t K, void *stream);

/* The same operation for 1 <= M <= 64 ("gpt-fast issue #114": its open
 * question of batch sizes above one).  x, W, scales, out as w8_gemv; K a
 * positive multiple of 16 up to 2^20, N up to 2^24.
 *   workspace        device, >= w8_workspace_bytes(M, N, K) bytes, 16-byte
 *                    aligned, owned by the caller; may be NULL when that is 0
 * M = 1, and M = 2 with N <= 64 x (SM count), with K <= 16384 run on
 * w8_gemv's CUDA-core kernel (no workspace; measured faster there); the
 * other calls, M = 3..4 included (measured faster than w8_gemv), run on the
 * tcgen05 tensor core in fp16 with fp32 accumulation: every int8 weight is an
 * fp16 number exactly, and each row m of x is scaled by a power of two
 * 2^sigma_m (max |x[m]| 2^sigma in [2^14, 2^15)), which keeps every bf16
 * value down to 2^-28 of the row's max exact in fp16; the result is
 * bf16_RN((acc 2^-sigma_m) * scales[n]).  Two or three launches (see
 * w8_kernel_launches); W4Q_ERR_WORKSPACE when the workspace is missing or
 * too small. */
int w8_gemm(const void *x_bf16, const int8_t *W, const void *scales_bf16,
            void *out_bf16, int64_t M, int64_t N, int64_t K, void *workspace,
            size_t workspace_bytes, void *stream);

/* Workspace bytes w8_gemm needs for these sizes on the current device (0
 * when w8_gemv serves the call or the sizes are invalid). */
size_t w8_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* Kernel launches of one w8_gemm call (1 for the CUDA-core kernel; 2 or 3
 * on the tensor core: activation preparation, the main kernel and, when a
 * row pair's K is split between CTAs, the partial-sum launch); 0 for
 * invalid sizes. */
int w8_kernel_launches(int64_t M, int64_t N, int64_t K);

/* ------------------------------------------------------------ status --- */

/* Read and clear the device-side error word of the current device (set by
 * a kernel whose bounded wait on a barrier ran out).  Synchronizes the
 * device.  *code receives the word (0 = no error): bit 0 a consumer's wait
 * for a full stage, bit 1 the producer's wait for a free stage, bit 2 the
 * final wait for copies in flight.  Returns W4Q_ERR_DEVICE when the word
 * was not 0.  After such an error the outputs of the calls since the last
 * read are unspecified. */
int w4q_device_error(uint32_t *code);

/* Self-test of that protocol (the pages have no counterpart): launches one
 * kernel on `stream` whose single waiting thread waits, with the library's
 * bounded sleeping wait, on a shared-memory barrier phase that nothing
 * completes, gives up after limit_us microseconds (1..100000) and sets bit
 * 0 of the error word, as a kernel of the library does when its wait runs
 * out.  Nothing faults and the context stays usable.  For tests. */
int w4q_selftest_wait_expiry(unsigned limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4Q_H */
