// noalloc.cu -- w4a16_gemm_noalloc: the W4A16 call for callers that cannot
// allocate device memory and cannot hand the library a workspace.
//
// Some callers may not call cudaMalloc (or any allocator) on the path that
// runs a layer: code that runs while a stream is being captured into a CUDA
// graph, where an allocation is not allowed; hosts that plan every byte of
// device memory ahead of time (embedded and real-time inference loops, which
// must not pause in an allocator or fragment the heap); and plug-ins running
// inside a framework whose device memory belongs to the framework's own
// pool.  For them this file keeps the scratch memory the W4A16 kernels need
// (prepared activations, group sums, row factors, split-K counters and
// partial sums) in one fixed array in device memory that belongs to the
// library.  The kernels and the arithmetic are exactly those of w4a16_gemm;
// only the source of the scratch differs.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "w4q.h"

namespace {

// The library-owned scratch array.  Every GPU that loads the library holds
// these 16 MiB until the process exits.  In host code the name g_scratch
// stands for a host-side shadow, not a device address: its device address
// comes from cudaGetSymbolAddress (below) and only that is passed to kernels.
constexpr size_t STATIC_SCRATCH_BYTES = W4Q_NOALLOC_SCRATCH_BYTES;
static_assert(STATIC_SCRATCH_BYTES == (size_t(16) << 20), "16 MiB, as documented in w4q.h");
static __device__ __align__(256) unsigned char g_scratch[STATIC_SCRATCH_BYTES];

constexpr int MAX_DEV = 64;
std::mutex g_mu;
void *g_scratch_addr[MAX_DEV];               // device address of g_scratch, per device
unsigned long long g_scratch_ctx[MAX_DEV];    // the context that address belongs to

// Looks the array up with that device current, again whenever the current
// context is not the one the cached address came from (after a device reset).
void *scratch_address(int dev)
{
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = w4q::current_context_id();
    if (g_scratch_addr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = w4q::current_context_id();
    }
    return g_scratch_addr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int w4a16_gemm_noalloc(const void *x_bf16, const void *packed, void *out_bf16,
                                  int64_t M, int64_t N, int64_t K, int group, void *stream)
{
    if (x_bf16 == nullptr || packed == nullptr || out_bf16 == nullptr)
        return W4Q_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0)
        return W4Q_ERR_INVALID_ARG;
    if (M > 64 || N > (1 << 24) || K > (1 << 20) || K % 256 != 0 || group != 32)
        return W4Q_ERR_UNSUPPORTED;
    if (!aligned16(x_bf16) || !aligned16(packed) || !aligned16(out_bf16))
        return W4Q_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV)
        return W4Q_ERR_CUDA;
    w4q::W4Plan plan;
    if (!w4q::w4_plan((int)M, (int)N, (int)K, -1, w4q::device_sm_count(dev), w4q::W4Mode::A16,
                      &plan))
        return W4Q_ERR_UNSUPPORTED;
    if (w4q::w4_workspace_for(plan, w4q::W4Mode::A16) > STATIC_SCRATCH_BYTES)
        return W4Q_ERR_UNSUPPORTED;  // needs more scratch than the static array holds
    void *ws = scratch_address(dev);
    unsigned *err = w4q::device_error_word(dev);
    if (ws == nullptr || err == nullptr)
        return W4Q_ERR_CUDA;
    // The split-K counters, the only scratch that must start at zero, are
    // reset by the call's own first kernel; everything else is written
    // before it is read within the call.
    const cudaError_t e = w4q::launch_w4(plan, w4q::W4Mode::A16, x_bf16, packed, out_bf16,
                                         nullptr, ws, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}
