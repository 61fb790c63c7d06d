// ak_tma.cuh -- sm_90+/sm_103a bulk tensor copies (TMA) and transaction
// barriers (mbarrier) in inline PTX, for kernels that stage whole tiles in
// shared memory without passing the bytes through registers.
//
// Every wait here is bounded: the caller passes an absolute global-timer
// deadline and gets false back when it passes, so a kernel can record an
// error and leave instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ak_common.cuh"

namespace ak {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --------------------------------------------------------------------------
// mbarrier (transaction-count barrier in shared memory)
// --------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` of incoming transactions.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// A plain arrival (no transactions): completes the phase of a count-1
// barrier on its own.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete; false once the
// global timer passes `deadline_ns`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t deadline_ns) {
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() > deadline_ns) return false;
    }
    return true;
}

// --------------------------------------------------------------------------
// bulk tensor copies (tile mode)
// --------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Global -> shared copy of the box at (c0, c1, c2); completion is signalled
// on `bar` as transaction bytes (the whole box, out-of-range parts
// zero-filled).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// --------------------------------------------------------------------------
// 128-byte swizzle (CU_TENSOR_MAP_SWIZZLE_128B) as seen from the threads
// --------------------------------------------------------------------------

// Byte offset of 16-byte chunk j of 128-byte row r in a buffer aligned to
// 1024 bytes: the chunk index is XOR-ed with the row's position within its
// group of 8 rows, so the 8 threads of a quarter-warp reading chunk j of 8
// consecutive rows touch 8 different bank quads.
__device__ __forceinline__ int swz128(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

}  // namespace ak
