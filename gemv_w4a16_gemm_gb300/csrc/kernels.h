// kernels.h -- host-side launchers of the CUDA kernels (internal; the public
// ABI is w4q.h).  Every launcher only launches: validation happens in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace w4q {

// The dynamic shared-memory opt-in of kernel fn, once per device: one bit
// per device in `done` (a device index of 64 or more opts in on every call).
// Setting the attribute on every call cost host time on each launch.
template <class F>
inline cudaError_t smem_opt_in_once(std::atomic<unsigned long long> &done, F fn, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0)
        done.fetch_or(bit, std::memory_order_release);
    return e;
}

// --- partial-sum launches of the tensor-core kernels

// Shape of a partial-sum launch over G2 row pairs of KB super-blocks whose
// U units are split into P contiguous ranges (split = 0) or `split` ranges
// per pair: rows of x per block (4 when the pairs alone would give few
// blocks, else 8) and contributors whose loads go out together (4, or 8
// when a pair can have more: under stream-K every range holds at least
// floor(U / P) units, so a pair meets at most ceil((KB - 1) / floor(U / P))
// ranges after its first).  Measured against a fixed (8, 4): 6656 x 19968
// M = 16 29.1 -> 27.1 us, W8 8192 x 8192 M = 64 22.0 -> 21.1 us.
struct FixShape {
    int rows, chunk;
};

inline FixShape fix_shape(int G2, int M, int KB, long long U, int P, int split, int sm_count)
{
    const long long minlen = P > 0 ? U / P : 1;
    const long long after = split > 0 ? split - 1
                                      : (minlen > 0 ? (KB - 1 + minlen - 1) / minlen : KB);
    FixShape fs;
    fs.chunk = after <= 4 ? 4 : 8;
    const long long blocks8 = (long long)G2 * ((M + 7) / 8);
    fs.rows = blocks8 <= 2LL * (sm_count > 0 ? sm_count : 1) ? 4 : 8;
    return fs;
}

// --- W4 pack / unpack (pack.cu)
cudaError_t launch_pack(const void *W, void *packed, int N, int K, cudaStream_t stream);
cudaError_t launch_unpack(const void *packed, uint8_t *q, void *scale, uint8_t *zero, int N, int K,
                          cudaStream_t stream);

// --- W4 GEMV / skinny GEMM (gemv_w4.cu)

// Work partition of the W4 kernel: the weight is cut into "tile groups" of
// 8 row tiles (128 rows) and 256-wide K super-blocks; unit u = g*KB + b.
// CTA c processes the contiguous units [begin(c), begin(c+1)).
struct W4Plan {
    int M, N, K;
    int KB;         // K / 256
    int T;          // ceil(N / 16) row tiles
    int G;          // ceil(T / 8) tile groups
    int P;          // CTAs
    int split;      // 0 = balanced (stream-K) ranges, s >= 1 = fixed split
    int NB;         // n8 blocks of the MMA: 1, 2, 4 or 8
    bool fold;      // dequantized weight rounded to bf16 (q - z) * s (the umma path)
    bool fixup;     // some tile group is split over CTAs
    size_t partial_bytes;  // fp32 partials [P][2][M][128] ([P][2][M][256] for umma)
    bool umma;      // tcgen05 kernel (W4A16, M >= 9): units are pairs of tile groups
    int NP;         // umma: M rounded up to 16 (the MMA's N)
    int G2;         // umma: ceil(G / 2) pairs of tile groups
    int cluster;    // > 0: the cluster kernel (M <= 8), this many CTAs split each group's K
    bool compact;   // the packed weight holds the compact metadata (cluster kernel only)
};

enum class W4Mode { A16, A8, A8_DOTS };

// Plan for these sizes (split: -1 = the library's choice, 0 = stream-K,
// s >= 1 = fixed).  Returns false when the sizes or split are unsupported.
// act_row: W4A8 with one activation scale per row (the split table keys it
// apart).  compact: the compact metadata, which only the cluster kernel reads.
bool w4_plan(int M, int N, int K, int split, int sm_count, W4Mode mode, W4Plan *plan,
             bool act_row = false, bool compact = false);

// Workspace bytes for a plan (partials + the W4A8 activation buffers).
size_t w4_workspace_for(const W4Plan &plan, W4Mode mode);

// act_row: W4A8 with one activation scale per row (else per group of 32).
cudaError_t launch_w4(const W4Plan &plan, W4Mode mode, const void *x, const void *packed,
                      void *out, int32_t *dots, void *workspace, unsigned *err,
                      cudaStream_t stream, bool act_row = false);

// --- W4A16 / W4A8 at M <= 8, one thread-block cluster per 128-row group
// (gemv_w4_cluster.cu).  w4_cluster_ring: the ring depth for a K split of C
// CTAs, 0 when the call does not fit the kernel's shared memory.
int w4_cluster_ring(int M, int KB, int C);
cudaError_t launch_w4_cluster(const W4Plan &plan, W4Mode mode, bool act_row, const void *x,
                              const void *packed, void *out, int32_t *dots, unsigned *err,
                              cudaStream_t stream);

// --- W4A16 on the tcgen05 tensor core, 9 <= M <= 64 (gemv_w4_umma.cu)
size_t w4_umma_workspace(const W4Plan &plan);
size_t w4_umma_partial_bytes(int P, int M);
cudaError_t launch_w4_umma(const W4Plan &plan, const void *x, const void *packed, void *out,
                           void *workspace, unsigned *err, cudaStream_t stream);

// --- compact metadata: packer and its inverse view (pack_compact.cu)
size_t packed_bytes_compact(int N, int K);
cudaError_t launch_pack_compact(const void *W, void *packed, int N, int K, cudaStream_t stream);
cudaError_t launch_unpack_compact(const void *packed, uint8_t *q, uint8_t *sc, uint8_t *zc,
                                  void *steps, int N, int K, cudaStream_t stream);

cudaError_t launch_act_quant_i8(const void *x, int M, int K, int8_t *xq, float *sx, bool row,
                                cudaStream_t stream);

// --- per-device state kept by api.cu
int device_sm_count(int dev);
unsigned *device_error_word(int dev);  // nullptr if the symbol lookup failed
unsigned long long current_context_id();  // 0 if no context is current

// --- W8 GEMV (w8.cu): CUDA cores, 1 <= M <= 4, K <= 16384, no workspace
cudaError_t launch_w8(const void *x, const int8_t *W, const void *scales, void *out, int M, int N,
                      int K, int sm_count, unsigned *err, cudaStream_t stream);
bool w8_supported(int M, int K);

// --- W8 on the tcgen05 tensor core, any 1 <= M <= 64 (gemv_w8_umma.cu)
size_t w8_tc_workspace(int M, int N, int K, int sm_count);
int w8_tc_launches(int M, int N, int K, int sm_count);
cudaError_t launch_w8_tc(const void *x, const int8_t *W, const void *scales, void *out, int M, int N,
                         int K, int sm_count, void *workspace, unsigned *err, cudaStream_t stream);

}  // namespace w4q
