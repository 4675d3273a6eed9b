// common.cuh -- inline-PTX helpers for the sm_103a kernels: mbarriers, 1-D
// bulk (TMA engine) copies, ldmatrix, the bf16 m16n8k16 MMA, bit tricks, and
// the bounded-wait error protocol.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4q {

// Error bits a kernel ORs into the device-side error word (passed to every
// kernel as a pointer): a consumer gave up waiting on a "full" barrier, the
// producer gave up waiting on an "empty" barrier, the final drain of
// in-flight copies ran out of time.

constexpr unsigned ERR_FULL_WAIT = 1u;
constexpr unsigned ERR_EMPTY_WAIT = 2u;
constexpr unsigned ERR_DRAIN_WAIT = 4u;

// A wait gives up after this many nanoseconds of %globaltimer (one second).
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete; false after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (global_timer() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

// As mbar_try_wait, but the thread may sleep up to `ns` nanoseconds in the
// instruction while the phase is incomplete (it resumes when the phase
// completes), so a long wait costs no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(ns)
                 : "memory");
    return ok != 0;
}

#ifndef W4Q_SLEEP_NS
#define W4Q_SLEEP_NS 20000u
#endif
// Wait for the phase of `parity`, the thread sleeping in the instruction
// (at most W4Q_SLEEP_NS per poll) instead of spinning, so waiting warps
// leave the issue slots to the others; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                unsigned long long limit_ns = WAIT_LIMIT_NS)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer();
    while (!mbar_try_wait_sleep(bar, parity, W4Q_SLEEP_NS))
        if (global_timer() - t0 > limit_ns)
            return false;
    return true;
}

__device__ __forceinline__ void report_error(unsigned *err, unsigned code)
{
    atomicOr(err, code);
}

// Device-scope atomic add with acquire-release ordering: writes made before
// it (by this thread, or by the warp through a preceding __syncwarp) are
// visible to whoever observes the increment, and reads after it see what
// the other incrementers wrote before theirs.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned *addr, unsigned v)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(addr), "r"(v)
                 : "memory");
    return old;
}

// ------------------------------------------------------------ bulk copies

// L2 eviction-priority policies for cp.async.bulk's cache hint.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on
// the mbarrier.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar), "l"(policy)
                 : "memory");
}

// 2-D tiled bulk copy global -> this CTA's shared memory through a tensor
// map (a __grid_constant__ kernel parameter), completing the box's bytes on
// the mbarrier.  (x, y): the box's first element (x innermost, its byte
// offset a multiple of 16); parts of the box outside the tensor read zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
                 : "memory");
}

// ------------------------------------------------- programmatic launches

// Let the next kernel in the stream (launched with programmatic stream
// serialization) start its prologue.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous kernel in the stream has completed and its memory
// is visible (a no-op when this kernel was launched without the attribute).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------------- fragments

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// D = A * B + C, bf16 inputs, fp32 accumulate, m16n8k16.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, const float (&c)[4])
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]),
                   "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// The W4A8 activation code of eight values: v[j] <- clamp(rint(fp32(v[j] /
// sx)), -127, 127), with sx = fp32(a / 127) for the max |v| a (> 0) of
// their group or row, so |v / sx| <= 127 (1 + 2^-23).  Computed as
// rint(v * r) with r = fp32(1 / sx): r and the product each round once,
// so |v * r - v / sx| < 2^-16 and |fp32(v / sx) - v / sx| < 2^-17, and
// the two round to the same integer unless v * r lies within 2^-15 of a
// half-integer.  There (|v * r - rint(v * r)| > 1/2 - 2^-14 is the test,
// with margin), and for a tiny sx whose reciprocal would overflow, the
// correctly rounded quotient decides.
__device__ __forceinline__ void act_code8(float (&v)[8], float sx)
{
    const float r = __frcp_rn(sx);
    const bool tiny = !(sx >= 0x1p-125f);
    constexpr float NEAR = 0.5f - 0x1p-14f;
    float q[8];
    bool near = tiny;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float y = v[j] * r;
        q[j] = rintf(y);
        near |= fabsf(y - q[j]) > NEAR;
    }
    if (near) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float y = v[j] * r;
            if (tiny || fabsf(y - rintf(y)) > NEAR)
                q[j] = rintf(__fdiv_rn(v[j], sx));
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
        v[j] = fminf(fmaxf(q[j], -127.f), 127.f);
}

}  // namespace w4q
