// ak_common.cuh -- sm_103a building blocks shared by the reduce and scan
// kernels: streaming and L2-policy vector loads and stores, relaxed flag
// reads, the global timer, programmatic dependent launch, and ordered warp /
// block combines of partial results.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ak_types.cuh"

namespace ak {

constexpr int kWarp = 32;

// --------------------------------------------------------------------------
// raw vectors and streaming loads
// --------------------------------------------------------------------------

template <int BYTES>
struct alignas(BYTES) Raw {
    uint32_t w[BYTES / 4];
};

// Read-only streaming load of 16 bytes: no L1 allocation, 256-byte L2
// prefetch granule (the input is read exactly once).
__device__ __forceinline__ Raw<16> ld_stream16(const void* p) {
    Raw<16> r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
        : "l"(p));
    return r;
}

// 32-byte load (sm_100+ 256-bit vector access), same cache policy.
__device__ __forceinline__ Raw<32> ld_stream32(const void* p) {
    Raw<32> r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
          "=r"(r.w[6]), "=r"(r.w[7])
        : "l"(p));
    return r;
}

template <int BYTES>
__device__ __forceinline__ Raw<BYTES> ld_stream(const void* p) {
    if constexpr (BYTES == 32) return ld_stream32(p);
    else return ld_stream16(p);
}

// Element k of a raw vector viewed as T.
template <class T, int BYTES>
__device__ __forceinline__ T raw_get(const Raw<BYTES>& r, int k) {
    T v;
    memcpy(&v, reinterpret_cast<const char*>(r.w) + k * sizeof(T), sizeof(T));
    return v;
}

// L2 eviction-priority policies (createpolicy) and 16-byte accesses that
// carry them: evict_last keeps a tile in L2 until it is read again,
// evict_first marks a last use.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ Raw<16> ld_hint16(const void* p, uint64_t policy) {
    Raw<16> r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "l"(p), "l"(policy));
    return r;
}
__device__ __forceinline__ void st_hint16(void* p, const Raw<16>& r, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(r.w[0]),
                 "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "l"(policy)
                 : "memory");
}

// 32-byte (sm_100+ 256-bit) load / store with an L2 policy: one lane's
// access covers a whole 32-byte sector.
__device__ __forceinline__ Raw<32> ld_hint32(const void* p, uint64_t policy) {
    Raw<32> r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
                   "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p), "l"(policy));
    return r;
}
__device__ __forceinline__ void st_hint32(void* p, const Raw<32>& r, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p),
                 "r"(r.w[0]), "r"(r.w[1]), "r"(r.w[2]), "r"(r.w[3]), "r"(r.w[4]), "r"(r.w[5]), "r"(r.w[6]),
                 "r"(r.w[7]), "l"(policy)
                 : "memory");
}

// --------------------------------------------------------------------------
// inter-block communication
// --------------------------------------------------------------------------

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// a / b for a >= 0 and b > 0, in 32-bit arithmetic when both fit (a 64-bit
// division is a long emulated instruction sequence on the GPU).
__device__ __forceinline__ int64_t div_fast(int64_t a, int64_t b) {
    if (((uint64_t)a | (uint64_t)b) < (1ull << 32)) return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch (sm_90+): the dependent grid may be scheduled
// before this one ends; griddep_wait() blocks until the prerequisite grid has
// completed and its memory is visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// --------------------------------------------------------------------------
// shuffles of arbitrary word-sized values
// --------------------------------------------------------------------------

template <class T>
__device__ __forceinline__ T shfl_down_any(const T& v, int d) {
    static_assert(sizeof(T) % 4 == 0, "word-sized types only");
    T r;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(&v);
    uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); ++i) o[i] = __shfl_down_sync(0xffffffffu, s[i], d);
    return r;
}

// shfl_down within segments of `width` lanes (a power of two <= 32).
template <class T>
__device__ __forceinline__ T shfl_down_width(const T& v, int d, int width) {
    static_assert(sizeof(T) % 4 == 0, "word-sized types only");
    T r;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(&v);
    uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); ++i) o[i] = __shfl_down_sync(0xffffffffu, s[i], d, width);
    return r;
}

template <class T>
__device__ __forceinline__ T shfl_up_any(const T& v, int d) {
    T r;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(&v);
    uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); ++i) o[i] = __shfl_up_sync(0xffffffffu, s[i], d);
    return r;
}

template <class T>
__device__ __forceinline__ T shfl_idx_any(const T& v, int lane) {
    T r;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(&v);
    uint32_t* o = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(T) / 4); ++i) o[i] = __shfl_sync(0xffffffffu, s[i], lane);
    return r;
}

// --------------------------------------------------------------------------
// ordered warp / block combines (lane 0 / thread 0 is the leftmost operand)
// --------------------------------------------------------------------------

// Lane 0 receives combine(v_0, v_1, ..., v_31). Each step combines a lane
// with the lane d to its right, so the operand order is preserved and
// non-commutative operators are safe.
template <class M>
__device__ __forceinline__ typename M::P warp_reduce(typename M::P v) {
#pragma unroll
    for (int d = 1; d < kWarp; d <<= 1) {
        typename M::P o = shfl_down_any(v, d);
        v = M::combine(v, o);
    }
    return v;
}

// Inclusive warp scan: lane l receives combine(v_0, ..., v_l).
template <class M>
__device__ __forceinline__ typename M::P warp_inclusive_scan(typename M::P v, int lane) {
#pragma unroll
    for (int d = 1; d < kWarp; d <<= 1) {
        typename M::P o = shfl_up_any(v, d);
        if (lane >= d) v = M::combine(o, v);
    }
    return v;
}

// Thread 0 receives the ordered combine of all threads' values (thread index
// order). smem must hold BLOCK / 32 partials. Ends with the block in sync.
template <class M, int BLOCK>
__device__ __forceinline__ typename M::P block_reduce(typename M::P v, typename M::P* smem) {
    constexpr int W = BLOCK / kWarp;
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    v = warp_reduce<M>(v);
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    if (warp == 0) {
        typename M::P w = lane < W ? smem[lane] : M::empty();
        w = warp_reduce<M>(w);
        v = w;
    }
    __syncthreads();
    return v;
}

}  // namespace ak
