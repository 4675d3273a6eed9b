// tcgen05.cuh -- inline-PTX helpers for the 5th-generation tensor core of
// sm_100-family GPUs (sm_103a): tensor-memory (TMEM) allocation, loads and
// stores, the MMA with its A operand in TMEM and B in shared memory, the
// commit that signals MMA completion on an mbarrier, and the descriptors.
//
// TMEM addresses are 32 bits: lane in bits 31..16, column in bits 15..0.
// A warp may touch only the 32-lane quarter (warp id % 4) of the 128 lanes.
#pragma once

#include <stdint.h>

namespace w4q {

// ------------------------------------------------------------ allocation

// Warp-wide: allocate `ncols` TMEM columns (a power of two >= 32) and write
// the base address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Warp-wide (the allocating warp): free the columns again.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ----------------------------------------------------------------- fences

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Generic-proxy writes to shared memory made visible to the async proxy
// (the tensor core and the bulk-copy engine).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------- loads and stores

// 16 lanes x 256 bits, four repetitions along the columns: thread t holds,
// for repetition i, (lane t/4, columns 8i + 2(t%4), +1) in v[4i], v[4i+1]
// and (lane t/4 + 8, the same columns) in v[4i+2], v[4i+3].
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
                 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
                 "r"(v[14]), "r"(v[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_16x256b_x1(uint32_t taddr, uint32_t v0, uint32_t v1,
                                                   uint32_t v2, uint32_t v3)
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(v0), "r"(v1), "r"(v2), "r"(v3)
                 : "memory");
}

// 32 lanes x 32 bits, eight columns: thread t <-> lane (quarter base + t),
// v[j] <-> column j.
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&v)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------- MMA

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M rows (64 or 128) and N columns (a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4)                          // D format: f32
           | (1u << 7)                        // A format: bf16
           | (1u << 10)                       // B format: bf16
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// The same with fp16 A and B.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N)
{
    return (1u << 4)                          // D format: f32 (A, B format 0: f16)
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: 8-row x 128-byte atoms (the 16-byte chunk c of row r
// stored at chunk c ^ r), atoms of consecutive 8-row groups 1024 bytes
// apart.  `addr` is the shared address of the operand's first K step; the
// atom it lies in must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128_kmajor(uint32_t addr)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu)   // start address / 16
           | ((uint64_t)1u << 16)              // leading byte offset (unused when swizzled)
           | ((uint64_t)(1024u >> 4) << 32)    // stride byte offset: 8-row group pitch
           | ((uint64_t)1u << 46)              // descriptor version
           | ((uint64_t)2u << 61);             // layout: 128-byte swizzle
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.  accumulate = 0
// overwrites D.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// The mbarrier at `bar` receives one arrival once every tcgen05 operation
// this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

}  // namespace w4q
