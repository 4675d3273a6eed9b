// api.cu -- the extern "C" entry points declared in include/w4q.h: host-side
// validation, per-device caches, and the launches.  Nothing here allocates
// device memory or synchronizes (except w4q_device_error).
#include <mutex>

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "w4q.h"

namespace w4q {

// The driver's unique id of the context current on this thread, 0 if there is
// none yet or the driver cannot say.  The two driver calls are resolved once
// through the runtime, so the library needs no link to libcuda.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static const GetCurrent get_current = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                           cudaSuccess && q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<GetCurrent>(f)
                   : nullptr;
    }();
    static const GetId get_id = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                           cudaSuccess && q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<GetId>(f)
                   : nullptr;
    }();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&c) != CUDA_SUCCESS || c == nullptr ||
        get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}
}  // namespace w4q

namespace {

// The device-side error word that bounded waits report into (one per device).
__device__ unsigned g_error_word;

constexpr int MAX_DEV = 64;
std::mutex g_mu;
int g_sm_count[MAX_DEV];
unsigned *g_err_ptr[MAX_DEV];
unsigned long long g_err_ctx[MAX_DEV];  // context the cached address belongs to

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV)
        return -1;
    return dev;
}

int sm_count(int dev)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

unsigned *error_word(int dev)
{
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long ctx = w4q::current_context_id();
    if (g_err_ptr[dev] == nullptr || ctx == 0 || ctx != g_err_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess)
            return nullptr;
        g_err_ptr[dev] = static_cast<unsigned *>(p);
        g_err_ctx[dev] = w4q::current_context_id();
    }
    return g_err_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sizes the kernels index with 32-bit ints (plus 64-bit products).
constexpr int64_t MAX_N = 1 << 24;
constexpr int64_t MAX_K = 1 << 20;

int check_w4_shape(int64_t M, int64_t N, int64_t K, int group)
{
    if (M <= 0 || N <= 0 || K <= 0)
        return W4Q_ERR_INVALID_ARG;
    if (M > 64 || N > MAX_N || K > MAX_K || K % 256 != 0 || group != 32)
        return W4Q_ERR_UNSUPPORTED;
    return W4Q_OK;
}

int gemm_common(w4q::W4Mode mode, const void *x, const void *packed, void *out, int64_t M,
                int64_t N, int64_t K, int group, int split, void *workspace,
                size_t workspace_bytes, int32_t *dots, void *stream, bool act_row = false,
                bool compact = false)
{
    if (x == nullptr || packed == nullptr || (out == nullptr && dots == nullptr))
        return W4Q_ERR_INVALID_ARG;
    int st = check_w4_shape(M, N, K, group);
    if (st != W4Q_OK)
        return st;
    if (split < -1)
        return W4Q_ERR_INVALID_ARG;
    if (split > (int)(K / 256))
        return W4Q_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(packed) || (out && !aligned16(out)) ||
        (dots && !aligned16(dots)) || (workspace && !aligned16(workspace)))
        return W4Q_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0)
        return W4Q_ERR_CUDA;
    w4q::W4Plan plan;
    if (!w4q::w4_plan((int)M, (int)N, (int)K, split, sm_count(dev), mode, &plan, act_row,
                      compact))
        return W4Q_ERR_UNSUPPORTED;
    const size_t need = w4q::w4_workspace_for(plan, mode);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return W4Q_ERR_WORKSPACE;
    unsigned *err = error_word(dev);
    if (err == nullptr)
        return W4Q_ERR_CUDA;
    cudaError_t e = w4q::launch_w4(plan, mode, x, packed, out, dots, workspace, err,
                                   static_cast<cudaStream_t>(stream), act_row);
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

int quantize_act_common(const void *x_bf16, int64_t M, int64_t K, int8_t *xq, float *sx,
                        bool row, void *stream)
{
    if (x_bf16 == nullptr || xq == nullptr || sx == nullptr)
        return W4Q_ERR_INVALID_ARG;
    int st = check_w4_shape(M, 1, K, 32);
    if (st != W4Q_OK)
        return st;
    if (!aligned16(x_bf16) || !aligned16(xq) || !aligned16(sx))
        return W4Q_ERR_MISALIGNED;
    cudaError_t e = w4q::launch_act_quant_i8(x_bf16, (int)M, (int)K, xq, sx, row,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

size_t workspace_common(int64_t M, int64_t N, int64_t K, int group, int split)
{
    if (check_w4_shape(M, N, K, group) != W4Q_OK || split < -1 || split > (int)(K / 256))
        return 0;
    const int dev = current_device();
    if (dev < 0)
        return 0;
    size_t best = 0;
    // W4A16, W4A8 with a scale per group, W4A8 with a scale per row
    const w4q::W4Mode modes[3] = {w4q::W4Mode::A16, w4q::W4Mode::A8, w4q::W4Mode::A8};
    for (int v = 0; v < 3; ++v) {
        const w4q::W4Mode mode = modes[v];
        w4q::W4Plan plan;
        if (w4q::w4_plan((int)M, (int)N, (int)K, split, sm_count(dev), mode, &plan, v == 2)) {
            const size_t b = w4q::w4_workspace_for(plan, mode);
            if (b > best)
                best = b;
        }
    }
    return best;
}

}  // namespace

namespace w4q {
// Internal accessors for other translation units of the library.
int device_sm_count(int dev) { return sm_count(dev); }
unsigned *device_error_word(int dev) { return error_word(dev); }
}  // namespace w4q

extern "C" {

const char *w4q_status_string(int status)
{
    switch (status) {
    case W4Q_OK: return "W4Q_OK";
    case W4Q_ERR_INVALID_ARG: return "W4Q_ERR_INVALID_ARG: null pointer or non-positive size";
    case W4Q_ERR_UNSUPPORTED: return "W4Q_ERR_UNSUPPORTED: M, K, group or split outside the supported ranges";
    case W4Q_ERR_MISALIGNED: return "W4Q_ERR_MISALIGNED: a device pointer is not 16-byte aligned";
    case W4Q_ERR_WORKSPACE: return "W4Q_ERR_WORKSPACE: workspace missing or too small";
    case W4Q_ERR_CUDA: return "W4Q_ERR_CUDA: a CUDA call or kernel launch failed";
    case W4Q_ERR_DEVICE: return "W4Q_ERR_DEVICE: a kernel's bounded wait ran out";
    default: return "W4Q_ERR_UNKNOWN";
    }
}

size_t w4_packed_bytes(int64_t N, int64_t K, int group)
{
    if (check_w4_shape(1, N, K, group) != W4Q_OK)
        return 0;
    return (size_t)((N + 127) / 128) * 8u * (size_t)(K / 256) * 2432u;
}

int w4_pack_weights(const void *W_bf16, int64_t N, int64_t K, int group, void *packed,
                    void *stream)
{
    if (W_bf16 == nullptr || packed == nullptr)
        return W4Q_ERR_INVALID_ARG;
    int st = check_w4_shape(1, N, K, group);
    if (st != W4Q_OK)
        return st;
    if (!aligned16(W_bf16) || !aligned16(packed))
        return W4Q_ERR_MISALIGNED;
    cudaError_t e = w4q::launch_pack(W_bf16, packed, (int)N, (int)K,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

int w4_unpack_weights(const void *packed, int64_t N, int64_t K, int group, uint8_t *q,
                      void *scale_bf16, uint8_t *zero, void *stream)
{
    if (packed == nullptr || q == nullptr || scale_bf16 == nullptr || zero == nullptr)
        return W4Q_ERR_INVALID_ARG;
    int st = check_w4_shape(1, N, K, group);
    if (st != W4Q_OK)
        return st;
    if (!aligned16(packed) || !aligned16(q) || !aligned16(scale_bf16) || !aligned16(zero))
        return W4Q_ERR_MISALIGNED;
    cudaError_t e = w4q::launch_unpack(packed, q, scale_bf16, zero, (int)N, (int)K,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

size_t w4_workspace_bytes(int64_t M, int64_t N, int64_t K, int group)
{
    return workspace_common(M, N, K, group, -1);
}

size_t w4_workspace_bytes_split(int64_t M, int64_t N, int64_t K, int group, int split_k)
{
    if (split_k < 0)
        return 0;
    return workspace_common(M, N, K, group, split_k);
}

int w4_split_choice(int64_t M, int64_t N, int64_t K, int group)
{
    if (check_w4_shape(M, N, K, group) != W4Q_OK)
        return -1;
    const int dev = current_device();
    if (dev < 0)
        return -1;
    w4q::W4Plan plan;
    if (!w4q::w4_plan((int)M, (int)N, (int)K, -1, sm_count(dev), w4q::W4Mode::A16, &plan))
        return -1;
    return plan.split;
}

int w4_kernel_launches(int64_t M, int64_t N, int64_t K, int group, int w4a8)
{
    if (check_w4_shape(M, N, K, group) != W4Q_OK)
        return -1;
    const int dev = current_device();
    if (dev < 0)
        return -1;
    if (w4a8 < 0 || w4a8 > 2)
        return -1;
    const w4q::W4Mode mode = w4a8 ? w4q::W4Mode::A8 : w4q::W4Mode::A16;
    w4q::W4Plan plan;
    if (!w4q::w4_plan((int)M, (int)N, (int)K, -1, sm_count(dev), mode, &plan, w4a8 == 2))
        return -1;
    // the cluster kernel alone; else the activation preparation (and counter
    // reset), the main kernel, and for the tensor-core kernel with split row
    // groups the partial-sum launch
    if (plan.cluster > 0)
        return 1;
    return (plan.umma && plan.fixup) ? 3 : 2;
}

int w4a16_gemm(const void *x_bf16, const void *packed, void *out_bf16, int64_t M, int64_t N,
               int64_t K, int group, void *workspace, size_t workspace_bytes, void *stream)
{
    return gemm_common(w4q::W4Mode::A16, x_bf16, packed, out_bf16, M, N, K, group, -1, workspace,
                       workspace_bytes, nullptr, stream);
}

int w4a16_gemm_split(const void *x_bf16, const void *packed, void *out_bf16, int64_t M,
                     int64_t N, int64_t K, int group, int split_k, void *workspace,
                     size_t workspace_bytes, void *stream)
{
    if (split_k < 0)
        return W4Q_ERR_INVALID_ARG;
    return gemm_common(w4q::W4Mode::A16, x_bf16, packed, out_bf16, M, N, K, group, split_k,
                       workspace, workspace_bytes, nullptr, stream);
}

int w4a8_gemm(const void *x_bf16, const void *packed, void *out_bf16, int64_t M, int64_t N,
              int64_t K, int group, void *workspace, size_t workspace_bytes, void *stream)
{
    return gemm_common(w4q::W4Mode::A8, x_bf16, packed, out_bf16, M, N, K, group, -1, workspace,
                       workspace_bytes, nullptr, stream);
}

int w4a8_gemm_split(const void *x_bf16, const void *packed, void *out_bf16, int64_t M,
                    int64_t N, int64_t K, int group, int split_k, void *workspace,
                    size_t workspace_bytes, void *stream)
{
    if (split_k < 0)
        return W4Q_ERR_INVALID_ARG;
    return gemm_common(w4q::W4Mode::A8, x_bf16, packed, out_bf16, M, N, K, group, split_k,
                       workspace, workspace_bytes, nullptr, stream);
}

int w4a8_quantize_act(const void *x_bf16, int64_t M, int64_t K, int8_t *xq, float *sx,
                      void *stream)
{
    return quantize_act_common(x_bf16, M, K, xq, sx, false, stream);
}

int w4a8_quantize_act_rowscale(const void *x_bf16, int64_t M, int64_t K, int8_t *xq, float *sx,
                               void *stream)
{
    return quantize_act_common(x_bf16, M, K, xq, sx, true, stream);
}

int w4a8_group_dots(const void *x_bf16, const void *packed, int64_t M, int64_t N, int64_t K,
                    int group, int32_t *D, void *workspace, size_t workspace_bytes, void *stream)
{
    if (D == nullptr)
        return W4Q_ERR_INVALID_ARG;
    return gemm_common(w4q::W4Mode::A8_DOTS, x_bf16, packed, nullptr, M, N, K, group, -1,
                       workspace, workspace_bytes, D, stream);
}

int w4a8_group_dots_rowscale(const void *x_bf16, const void *packed, int64_t M, int64_t N,
                             int64_t K, int group, int32_t *D, void *workspace,
                             size_t workspace_bytes, void *stream)
{
    if (D == nullptr)
        return W4Q_ERR_INVALID_ARG;
    return gemm_common(w4q::W4Mode::A8_DOTS, x_bf16, packed, nullptr, M, N, K, group, -1,
                       workspace, workspace_bytes, D, stream, true);
}

int w4a8_gemm_rowscale(const void *x_bf16, const void *packed, void *out_bf16, int64_t M,
                       int64_t N, int64_t K, int group, void *workspace, size_t workspace_bytes,
                       void *stream)
{
    return gemm_common(w4q::W4Mode::A8, x_bf16, packed, out_bf16, M, N, K, group, -1, workspace,
                       workspace_bytes, nullptr, stream, true);
}

int w4a8_gemm_rowscale_split(const void *x_bf16, const void *packed, void *out_bf16, int64_t M,
                             int64_t N, int64_t K, int group, int split_k, void *workspace,
                             size_t workspace_bytes, void *stream)
{
    if (split_k < 0)
        return W4Q_ERR_INVALID_ARG;
    return gemm_common(w4q::W4Mode::A8, x_bf16, packed, out_bf16, M, N, K, group, split_k,
                       workspace, workspace_bytes, nullptr, stream, true);
}

size_t w4_packed_bytes_compact(int64_t N, int64_t K, int group)
{
    if (check_w4_shape(1, N, K, group) != W4Q_OK)
        return 0;
    return w4q::packed_bytes_compact((int)N, (int)K);
}

int w4_pack_weights_compact(const void *W_bf16, int64_t N, int64_t K, int group, void *packed,
                            void *stream)
{
    if (W_bf16 == nullptr || packed == nullptr)
        return W4Q_ERR_INVALID_ARG;
    int st = check_w4_shape(1, N, K, group);
    if (st != W4Q_OK)
        return st;
    if (!aligned16(W_bf16) || !aligned16(packed))
        return W4Q_ERR_MISALIGNED;
    cudaError_t e = w4q::launch_pack_compact(W_bf16, packed, (int)N, (int)K,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

int w4_unpack_weights_compact(const void *packed, int64_t N, int64_t K, int group, uint8_t *q,
                              uint8_t *scale_codes, uint8_t *zero_codes, void *steps_fp16,
                              void *stream)
{
    if (packed == nullptr || q == nullptr || scale_codes == nullptr || zero_codes == nullptr ||
        steps_fp16 == nullptr)
        return W4Q_ERR_INVALID_ARG;
    int st = check_w4_shape(1, N, K, group);
    if (st != W4Q_OK)
        return st;
    if (!aligned16(packed) || !aligned16(q) || !aligned16(scale_codes) || !aligned16(zero_codes) ||
        !aligned16(steps_fp16))
        return W4Q_ERR_MISALIGNED;
    cudaError_t e = w4q::launch_unpack_compact(packed, q, scale_codes, zero_codes, steps_fp16,
                                               (int)N, (int)K, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

int w4a16_gemm_compact(const void *x_bf16, const void *packed, void *out_bf16, int64_t M,
                       int64_t N, int64_t K, int group, void *stream)
{
    if (M > 8)
        return W4Q_ERR_UNSUPPORTED;
    return gemm_common(w4q::W4Mode::A16, x_bf16, packed, out_bf16, M, N, K, group, -1, nullptr,
                       0, nullptr, stream, false, true);
}

int w8_gemv(const void *x_bf16, const int8_t *W, const void *scales_bf16, void *out_bf16,
            int64_t M, int64_t N, int64_t K, void *stream)
{
    if (x_bf16 == nullptr || W == nullptr || scales_bf16 == nullptr || out_bf16 == nullptr)
        return W4Q_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0)
        return W4Q_ERR_INVALID_ARG;
    if (N > MAX_N || !w4q::w8_supported((int)M, (int)(K > MAX_K ? MAX_K + 1 : K)))
        return W4Q_ERR_UNSUPPORTED;
    if (!aligned16(x_bf16) || !aligned16(W) || !aligned16(scales_bf16) || !aligned16(out_bf16))
        return W4Q_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0)
        return W4Q_ERR_CUDA;
    unsigned *err = error_word(dev);
    if (err == nullptr)
        return W4Q_ERR_CUDA;
    cudaError_t e = w4q::launch_w8(x_bf16, W, scales_bf16, out_bf16, (int)M, (int)N, (int)K,
                                   sm_count(dev), err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

// W8 calls up to this M (and K within its range) run on the CUDA-core
// kernel (w8.cu), the others on the tensor core (gemv_w8_umma.cu).
#ifndef W4Q_W8_CC_MAX_M
#define W4Q_W8_CC_MAX_M 2
#endif
// The CUDA-core kernel serves M = 1, and M = 2 when its rows fit one wave
// (at most 64 per CTA, one CTA per SM at M = 2); the tensor core the rest.
// Measured: 8192 x 8192 M = 2 16.2 us on the CUDA cores against 17.0 on the
// tensor core; 28672 x 8192 M = 2 53.2 against 41.3 us (three waves).
static bool w8_on_cuda_cores(int64_t M, int64_t N, int64_t K)
{
    if (M > W4Q_W8_CC_MAX_M || !w4q::w8_supported((int)M, (int)K))
        return false;
    if (M == 1)
        return true;
    const int dev = current_device();
    return dev >= 0 && N <= 64LL * sm_count(dev);
}

size_t w8_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0 || M > 64 || N > MAX_N || K > MAX_K || K % 16 != 0)
        return 0;
    if (w8_on_cuda_cores(M, N, K))
        return 0;  // the CUDA-core kernel: no workspace
    const int dev = current_device();
    if (dev < 0)
        return 0;
    return w4q::w8_tc_workspace((int)M, (int)N, (int)K, sm_count(dev));
}

int w8_kernel_launches(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0 || M > 64 || N > MAX_N || K > MAX_K || K % 16 != 0)
        return 0;
    if (w8_on_cuda_cores(M, N, K))
        return 1;
    const int dev = current_device();
    if (dev < 0)
        return 0;
    return w4q::w8_tc_launches((int)M, (int)N, (int)K, sm_count(dev));
}

int w8_gemm(const void *x_bf16, const int8_t *W, const void *scales_bf16, void *out_bf16, int64_t M,
            int64_t N, int64_t K, void *workspace, size_t workspace_bytes, void *stream)
{
    if (x_bf16 == nullptr || W == nullptr || scales_bf16 == nullptr || out_bf16 == nullptr)
        return W4Q_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || K % 16 != 0)
        return W4Q_ERR_INVALID_ARG;
    if (M > 64 || N > MAX_N || K > MAX_K)
        return W4Q_ERR_UNSUPPORTED;
    if (w8_on_cuda_cores(M, N, K))
        return w8_gemv(x_bf16, W, scales_bf16, out_bf16, M, N, K, stream);
    if (!aligned16(x_bf16) || !aligned16(W) || !aligned16(scales_bf16) || !aligned16(out_bf16) ||
        (workspace != nullptr && !aligned16(workspace)))
        return W4Q_ERR_MISALIGNED;
    const int dev = current_device();
    if (dev < 0)
        return W4Q_ERR_CUDA;
    const size_t need = w4q::w8_tc_workspace((int)M, (int)N, (int)K, sm_count(dev));
    if (workspace == nullptr || workspace_bytes < need)
        return W4Q_ERR_WORKSPACE;
    unsigned *err = error_word(dev);
    if (err == nullptr)
        return W4Q_ERR_CUDA;
    cudaError_t e = w4q::launch_w8_tc(x_bf16, W, scales_bf16, out_bf16, (int)M, (int)N, (int)K,
                                      sm_count(dev), workspace, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? W4Q_OK : W4Q_ERR_CUDA;
}

int w4q_device_error(uint32_t *code)
{
    if (code == nullptr)
        return W4Q_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return W4Q_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof v) != cudaSuccess)
        return W4Q_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero) != cudaSuccess)
        return W4Q_ERR_CUDA;
    *code = v;
    return v == 0 ? W4Q_OK : W4Q_ERR_DEVICE;
}

}  // extern "C"
