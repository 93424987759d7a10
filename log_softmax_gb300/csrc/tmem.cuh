// Blackwell data movement shared by the kernels that park data in tensor memory:
// tcgen05 copies from shared memory into tensor memory, loads back to registers,
// their fences and completion, and the 2-D tensor (TMA) copy into shared memory.
//
// Tensor memory is 256 KB per SM: 128 lanes x 512 columns of 32 bits, allocated per
// CTA in columns (tcgen05.alloc).  The kernels here use it as a buffer, not as an
// MMA accumulator.  tcgen05.cp.128x256b with a no-swizzle shared-memory descriptor,
// 128 bytes between 8-row groups and 2048 bytes between the two 16-byte halves of a
// row, copies one 4 KB block of 1024 floats so that lane l holds floats [4l, 4l + 4)
// in its columns 0-3 and [512 + 4l, 512 + 4l + 4) in columns 4-7 (checked on GB300
// against the PTX description of the shape).  A warp reads the lanes of its quarter
// (warp index mod 4) with tcgen05.ld.32x32b.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace lse {

__device__ __forceinline__ uint64_t tmem_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tmem_cp_block(uint32_t taddr, const float* smem_block) {
    const uint64_t d = tmem_smem_desc(smem_u32(smem_block), 2048, 128);
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void tmem_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Whole warp: 32 consecutive columns of this warp's 32 lanes (four blocks).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Whole warp: 8 consecutive columns of this warp's 32 lanes (one block).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld_all() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Whole warp: allocates `cols` columns of tensor memory (a power of two, at least 32)
// and writes their base address to shared memory at `slot`; then gives up the right
// to allocate more, so that another CTA on the SM waiting to allocate can proceed.
__device__ __forceinline__ void tmem_alloc_warp(uint32_t* slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Whole warp: frees the columns that tmem_alloc_warp allocated.
__device__ __forceinline__ void tmem_dealloc_warp(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// 2-D tensor copy of the box at (x, row) of `map` into shared memory, completing on
// `bar` by transaction count; the source lines are marked evict-first (read once).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int row, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(row), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

}  // namespace lse
