// timeline.cuh -- %globaltimer stamps for the profiling build only.
//
// Built with -DW4Q_TIMELINE (gemv_w4a16_gemm_gb300/timeline.py does this into
// a separate library), W4Q_STAMP(ev) appends (time in ns, ev << 32 | linear
// block index) to a device buffer of this translation unit, and
// W4Q_STAMP_READER(name) defines an extern "C" reader that copies the stamps
// out and empties the buffer.  In the ordinary build both expand to nothing.
#pragma once

#ifdef W4Q_TIMELINE
#include <cuda_runtime.h>

static __device__ unsigned long long g_w4q_stamps[2 << 18];
static __device__ unsigned g_w4q_nstamps;

#define W4Q_STAMP(ev)                                                                            \
    do {                                                                                         \
        unsigned long long t_;                                                                   \
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                   \
        const unsigned i_ = atomicAdd(&g_w4q_nstamps, 1u);                                       \
        if (i_ < (1u << 18)) {                                                                   \
            g_w4q_stamps[2 * i_] = t_;                                                           \
            g_w4q_stamps[2 * i_ + 1] =                                                           \
                ((unsigned long long)(ev) << 32) | (blockIdx.x + blockIdx.y * gridDim.x);        \
        }                                                                                        \
    } while (0)

#define W4Q_STAMP_READER(name)                                                                   \
    extern "C" int name(unsigned long long *host, unsigned *n)                                   \
    {                                                                                            \
        if (cudaDeviceSynchronize() != cudaSuccess)                                              \
            return 5;                                                                            \
        unsigned v = 0;                                                                          \
        if (cudaMemcpyFromSymbol(&v, g_w4q_nstamps, sizeof v) != cudaSuccess)                    \
            return 5;                                                                            \
        if (v > (1u << 18))                                                                      \
            v = 1u << 18;                                                                        \
        if (host && v && cudaMemcpyFromSymbol(host, g_w4q_stamps, (size_t)v * 16) != cudaSuccess) \
            return 5;                                                                            \
        *n = v;                                                                                  \
        const unsigned z = 0;                                                                    \
        return cudaMemcpyToSymbol(g_w4q_nstamps, &z, sizeof z) == cudaSuccess ? 0 : 5;           \
    }
#else
#define W4Q_STAMP(ev) ((void)0)
#define W4Q_STAMP_READER(name)
#endif
