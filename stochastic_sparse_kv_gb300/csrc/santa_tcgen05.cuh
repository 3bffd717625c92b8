// santa_tcgen05.cuh -- inline-PTX wrappers for the fifth-generation tensor cores
// (tcgen05: MMA from shared-memory descriptors into tensor memory, TMEM) and for tiled
// TMA loads (cp.async.bulk.tensor), sm_103a.
//
// Conventions used by the score kernel:
//  * operands are K-major bf16 tiles in the 128-byte swizzled layout that a TMA copy
//    with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128 bytes (64 elements), 16-byte
//    pieces of row y stored at piece index (i ^ (y % 8)), 8-row groups 1024 bytes apart,
//    every tile 1024-byte aligned;
//  * one MMA is M=128 x N x K=16, fp32 accumulation, issued by a single thread; its
//    accumulator row i sits in TMEM lane i, column j in TMEM column (base + j);
//  * a warp may read only the 32 TMEM lanes of its sub-partition, 32 * (warp % 4).
#pragma once

#include <cuda.h>  // CUtensorMap

#include "santa_common.cuh"

namespace santa {

// ---- tensor memory allocation (one whole warp; the address lands in shared memory)

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations across a thread synchronisation (barrier or mbarrier).
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Generic-proxy writes to shared memory made visible to the async proxy (TMA, MMA).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- MMA

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzled layout:
// start address >> 4 (bits 0-13), leading offset (unused by this layout: 16 bytes),
// stride between 8-row groups = 1024 bytes (bits 32-45), descriptor version 1
// (bits 46-47), layout 2 = 128-byte swizzle (bits 61-63).  Stepping K by 16 elements
// inside the 128-byte row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and fp32 D:
// D format (bits 4-5) = 1, A format (7-9) = 1, B format (10-12) = 1, N >> 3 (17-22),
// M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] = A * B^T (+ D when accumulate != 0); one thread issues it.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One arrival on `bar` once every MMA this thread has issued so far is complete.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---- TMEM -> registers: N consecutive 32-bit columns of the warp's 32 lanes (one lane
// per thread); the wait is in the same statement, so the values are ready on return.
template <int N>
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[N]);

template <>
__device__ __forceinline__ void tmem_ld32<1>(uint32_t taddr, uint32_t (&v)[1])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0])
        : "r"(taddr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld32<2>(uint32_t taddr, uint32_t (&v)[2])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1])
        : "r"(taddr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld32<4>(uint32_t taddr, uint32_t (&v)[4])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
        : "r"(taddr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld32<8>(uint32_t taddr, uint32_t (&v)[8])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
        : "r"(taddr)
        : "memory");
}

// ---- tiled TMA loads (2-D tensor map in kernel-parameter space)

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// Box at element coordinates (x, y) -> dst; x * 2 bytes must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_plain(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace santa
