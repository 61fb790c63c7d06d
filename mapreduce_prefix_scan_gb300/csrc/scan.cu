// scan.cu -- inclusive scans (accumulate!, cumsum) on GB300.
//
// Contiguous lines (the whole array, or every line along dimension 0) take a
// single-pass tile scan; lines along a strided dimension take a
// column-parallel kernel.
//
// Tile scan (AcceleratedKernels.jl tile-scan PR #202, first two
// paragraphs): a tile is loaded striped (coalesced), each thread scans its
// own run of `items` consecutive elements, the run totals are scanned across
// the block, and the tile's prefix is applied. Runs sit in shared memory at
// an odd stride so that the threads of a warp reading their runs spread over
// the banks. GB300 version of that padding: the stride is odd in 16-byte
// units (one 16-byte pad after a run whose length is an even number of
// 16-byte chunks), which keeps every run 16-byte aligned, so runs of any
// element size are read and written with 128-bit shared accesses and 8
// consecutive threads hit 8 distinct bank quads.
//
// Tiles pass prefixes on in one pass with decoupled look-back (Merrill &
// Garland, "Single-pass Parallel Prefix Scan with Decoupled Look-back",
// 2016): a tile publishes its aggregate, a warp inspects up to 32
// predecessors at a time, folds aggregates back to the nearest published
// inclusive prefix, then publishes its own inclusive prefix. The grid is
// persistent and cooperative (all blocks co-resident) and each block takes
// its tiles in increasing order, so the lowest unfinished tile can always
// progress. Every tile-state word carries the call's epoch, so stale state
// from earlier calls is never mistaken for a publication and the workspace
// needs no clearing. Every wait is bounded by a global-timer deadline; a
// block that gives up records the epoch in the workspace's error word,
// which every other waiter also watches, and all blocks leave early.
#include <algorithm>

#include "ak_common.cuh"
#include "ak_internal.h"

namespace ak {

namespace {

constexpr int kMaxBlock = 512;
constexpr unsigned kFull = 0xffffffffu;
enum : uint64_t { kStatusAggregate = 1, kStatusPrefix = 2 };

template <class Acc>
constexpr int default_items() {
    return sizeof(Acc) >= 16 ? 8 : (sizeof(Acc) == 8 ? 8 : 16);
}

// Shared-memory run layout: run r starts at 16-byte chunk r * run_stride.
template <class Acc, int ITEMS>
struct RunLayout {
    static constexpr int chunks = ITEMS * (int)sizeof(Acc) / 16;
    static_assert(ITEMS * sizeof(Acc) % 16 == 0, "a run must be a whole number of 16-byte chunks");
    static constexpr int stride = chunks % 2 == 0 ? chunks + 1 : chunks;  // odd, in chunks
    static __device__ __forceinline__ char* run_ptr(char* base, int r) { return base + (size_t)r * stride * 16; }
    // byte offset of element e of the tile
    static __device__ __forceinline__ int elem_off(int e) {
        return (e / ITEMS) * stride * 16 + (e % ITEMS) * (int)sizeof(Acc);
    }
};

// Copies of whole 16-byte chunks through uint4, so shared-memory traffic is
// 128-bit (both pointers 16-byte aligned).
// Register side is assembled word by word with compile-time indices so
// that it stays in registers.
template <class T, int N>
__device__ __forceinline__ void smem_load(T (&dst)[N], const char* src) {
    static_assert(sizeof(T) * N % 16 == 0 && sizeof(T) % 4 == 0 && sizeof(T) <= 16, "whole chunks of words");
    constexpr int WPE = sizeof(T) / 4, E = 16 / sizeof(T);  // words per element, elements per chunk
#pragma unroll
    for (int c = 0; c < N / E; ++c) {
        const uint4 v = reinterpret_cast<const uint4*>(src)[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < E; ++k) {
            uint32_t e[WPE];
#pragma unroll
            for (int q = 0; q < WPE; ++q) e[q] = w[k * WPE + q];
            memcpy(&dst[c * E + k], e, sizeof(T));
        }
    }
}
template <class T, int N>
__device__ __forceinline__ void smem_store(char* dst, const T (&src)[N]) {
    static_assert(sizeof(T) * N % 16 == 0 && sizeof(T) % 4 == 0 && sizeof(T) <= 16, "whole chunks of words");
    constexpr int WPE = sizeof(T) / 4, E = 16 / sizeof(T);
#pragma unroll
    for (int c = 0; c < N / E; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < E; ++k) {
            uint32_t e[WPE];
            memcpy(e, &src[c * E + k], sizeof(T));
#pragma unroll
            for (int q = 0; q < WPE; ++q) w[k * WPE + q] = e[q];
        }
        reinterpret_cast<uint4*>(dst)[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <class P>
struct TileState {
    uint64_t* flags;
    P* aggs;
    P* incls;
};

struct ScanCtl {
    uint64_t epoch;
    uint64_t* error_word;
    int64_t wait_limit_ns;
    int64_t skip_tile;  // fault injection; -1 = off
};

__device__ __forceinline__ bool aborted(const ScanCtl& ctl) {
    return ld_relaxed_u64(ctl.error_word) == ctl.epoch;
}

// Ordered combine over the block (thread 0 leftmost) for a runtime block
// size; the result is valid in thread 0; ends with the block in sync.
template <class M>
__device__ __forceinline__ typename M::P block_reduce_rt(typename M::P v, typename M::P* red, int W) {
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    v = warp_reduce<M>(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        typename M::P w = lane < W ? red[lane] : M::empty();
        v = warp_reduce<M>(w);
    }
    __syncthreads();
    return v;
}

// Block-wide look-back: the exclusive prefix of tile g from its
// predecessors g_first..g-1, valid in thread 0. Thread t inspects tile
// hi - (B-1) + t, so one round covers B predecessors (a whole wave of the
// persistent grid); rounds repeat only while no inclusive prefix is found.
// Returns false (in every thread) when a wait ran out or another block gave
// up.
template <class M>
__device__ __forceinline__ bool block_look_back(int64_t g, int64_t g_first, const TileState<typename M::P>& ts,
                                                const ScanCtl& ctl, typename M::P* red, int* ints,
                                                typename M::P* excl0) {
    using P = typename M::P;
    const int B = blockDim.x, W = B / kWarp;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    P excl = M::empty();
    int64_t hi = g - 1;
    const uint64_t t_start = globaltimer_ns();
    while (true) {
        const int64_t idx = hi - (B - 1) + tid;
        const bool valid = idx >= g_first;
        uint64_t status = 0;
        bool fail = false;
        if (valid) {
            while (true) {
                const uint64_t f = ld_acquire_u64(ts.flags + idx);
                status = (f >> 2) == ctl.epoch ? (f & 3u) : 0u;
                if (status != 0) break;
                if (globaltimer_ns() - t_start > (uint64_t)ctl.wait_limit_ns || aborted(ctl)) {
                    fail = true;
                    break;
                }
                __nanosleep(64);
            }
        }
        if (__syncthreads_or(fail)) return false;
        // nearest inclusive prefix of the window: the highest thread holding one
        const unsigned pm = __ballot_sync(kFull, valid && status == kStatusPrefix);
        if (lane == 0) ints[warp] = pm ? warp * kWarp + (kWarp - 1 - __clz(pm)) : -1;
        __syncthreads();
        int stop = -1;
        for (int w = 0; w < W; ++w) stop = max(stop, ints[w]);
        P v = M::empty();
        if (valid && tid == stop) v = ld_coherent(ts.incls + idx);
        else if (valid && tid > stop) v = ld_coherent(ts.aggs + idx);
        v = block_reduce_rt<M>(v, red, W);  // tiles in increasing order
        if (tid == 0) excl = M::combine(v, excl);
        if (stop >= 0) break;
        hi -= B;
    }
    if (tid == 0) *excl0 = excl;
    return true;
}

// cp.async (LDGSTS) 16-byte global -> shared copy, cached in L2 only.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <class P>
__device__ __forceinline__ void publish(const TileState<P>& ts, int64_t g, uint64_t status, const P& v,
                                        uint64_t epoch) {
    if (status == kStatusAggregate) ts.aggs[g] = v;
    else ts.incls[g] = v;
    st_release_u64(ts.flags + g, (epoch << 2) | status);
}

template <class Acc>
constexpr int scan_max_threads() { return sizeof(Acc) >= 16 ? 256 : 512; }

// One tile scan over lines of `len` contiguous elements (lines follow each
// other in memory). Dynamic shared memory: one padded run tile (two when the
// next tile is prefetched), then the block-scan scratch. When the input and
// accumulator types coincide, the block prefetches its next tile with
// cp.async into the second buffer while it scans, looks back and stores
// the current one.
template <class In, class Acc, class Out, class M, int ITEMS>
__global__ void __launch_bounds__(scan_max_threads<Acc>(), 2)
    k_scan_tiles(const In* __restrict__ x, Out* __restrict__ y, int64_t len, int64_t tiles_per_line, int64_t ntiles,
                 TileState<typename M::P> ts, ScanCtl ctl, bool has_init, Acc init) {
    using P = typename M::P;
    using L = RunLayout<Acc, ITEMS>;
    constexpr bool kPrefetch = std::is_same_v<In, Acc>;
    extern __shared__ __align__(16) char smem_raw[];
    const int B = blockDim.x;
    const int W = B / kWarp;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const size_t tile_bytes = (size_t)B * L::stride * 16;
    // buffer k of the (one or two) run tiles
    auto buf_of = [&](int k) { return smem_raw + (kPrefetch ? (size_t)k * tile_bytes : 0); };
    P* warp_tot = reinterpret_cast<P*>(smem_raw + (kPrefetch ? 2 : 1) * tile_bytes);
    P* red = warp_tot + kWarp;
    P* bcast = red + kWarp;  // [0] tile aggregate, [1] tile prefix
    int* ints = reinterpret_cast<int*>(bcast + 2);  // [0..W) look-back scratch, [kWarp] stop flag

    const int tile_elems = B * ITEMS;
    constexpr int VIN = sizeof(In) < 16 ? 16 / (int)sizeof(In) : 1;   // input elements per 16-byte load
    constexpr int VOUT = sizeof(Out) < 16 ? 16 / (int)sizeof(Out) : 1;
    static_assert(ITEMS % VIN == 0 && ITEMS % VOUT == 0, "runs must hold whole vectors");

    // Starts the asynchronous copy of tile gg into buf; false when gg does not
    // exist or is ragged / unaligned (those are loaded synchronously).
    auto prefetch = [&](int64_t gg, char* buf) -> bool {
        if constexpr (!kPrefetch) {
            return false;
        } else {
            if (gg >= ntiles) return false;
            const int64_t t = gg % tiles_per_line;
            if (len - t * (int64_t)tile_elems < tile_elems) return false;
            const In* src = x + (gg / tiles_per_line) * len + t * tile_elems;
            if (reinterpret_cast<uintptr_t>(src) % 16 != 0) return false;
            for (int v = tid; v < tile_elems / VIN; v += B) cp_async16(buf + L::elem_off(v * VIN), src + (int64_t)v * VIN);
            return true;
        }
    };

    int cur = 0;
    bool have = prefetch(blockIdx.x, buf_of(0));
    if constexpr (kPrefetch) cp_async_commit();

    for (int64_t g = blockIdx.x; g < ntiles; g += gridDim.x) {
        const int64_t line = g / tiles_per_line, t = g % tiles_per_line;
        const int64_t start = line * len + t * tile_elems;
        const int cnt = (int)min((int64_t)tile_elems, len - t * (int64_t)tile_elems);
        const In* src = x + start;
        Out* dst = y + start;
        char* tile = buf_of(cur);

        bool have_next = false;
        if constexpr (kPrefetch) {
            have_next = prefetch(g + gridDim.x, buf_of(cur ^ 1));
            cp_async_commit();
            cp_async_wait<1>();  // this tile's group has landed (the newest may still fly)
        }
        // ---- striped load into the padded run layout (when not prefetched)
        if (!have) {
            const bool vec_in = cnt == tile_elems && (reinterpret_cast<uintptr_t>(src) % 16 == 0);
            if (vec_in) {
                for (int v = tid; v < tile_elems / VIN; v += B) {
                    In e[VIN];
                    if constexpr (VIN > 1) {
                        Raw<16> r = ld_stream16(src + (int64_t)v * VIN);
                        memcpy(e, &r, 16);
                    } else {
                        e[0] = src[v];
                    }
                    Acc a[VIN];
#pragma unroll
                    for (int q = 0; q < VIN; ++q) a[q] = convert<Acc>(e[q]);
                    smem_store(tile + L::elem_off(v * VIN), a);
                }
            } else {
                for (int e = tid; e < tile_elems; e += B) {
                    Acc a;
                    if (e < cnt) a = convert<Acc>(src[e]);
                    else memset(&a, 0, sizeof a);
                    *reinterpret_cast<Acc*>(tile + L::elem_off(e)) = a;
                }
            }
        }
        __syncthreads();

        // ---- each thread scans its run in registers
        Acc run[ITEMS];
        smem_load(run, L::run_ptr(tile, tid));
#pragma unroll
        for (int i = 1; i < ITEMS; ++i) run[i] = M::op::apply(run[i - 1], run[i]);
        // elements past the end of a ragged tile must not reach the aggregate
        const int valid_items = min(ITEMS, max(0, cnt - tid * ITEMS));
        P total = M::lift(run[ITEMS - 1]);
        if (valid_items < ITEMS) {
            // ragged run: predicated fold of the valid elements (still in smem)
            Acc orig[ITEMS];
            smem_load(orig, L::run_ptr(tile, tid));
            total = M::empty();
#pragma unroll
            for (int i = 0; i < ITEMS; ++i)
                if (i < valid_items) total = M::combine(total, M::lift(orig[i]));
        }

        // ---- block scan of run totals (thread order)
        P inc = warp_inclusive_scan<M>(total, lane);
        P lane_excl = shfl_up_any(inc, 1);
        if (lane == 0) lane_excl = M::empty();
        if (lane == kWarp - 1) warp_tot[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            P w = lane < W ? warp_tot[lane] : M::empty();
            P wi = warp_inclusive_scan<M>(w, lane);
            P we = shfl_up_any(wi, 1);
            if (lane == 0) we = M::empty();
            if (lane < W) warp_tot[lane] = we;  // exclusive base of each warp
            if (lane == 0) bcast[0] = shfl_idx_any(wi, W - 1);
            else shfl_idx_any(wi, W - 1);
        }
        __syncthreads();

        // ---- tile prefix: publish the aggregate, look back, publish the prefix
        const P agg = bcast[0];
        const bool first = (t == 0);
        const bool last = (t == tiles_per_line - 1);
        const bool skip = (g == ctl.skip_tile);
        P prefix = M::empty();
        if (first) {
            if (has_init) prefix = M::lift(init);
            if (tid == 0 && !last && !skip) publish(ts, g, kStatusPrefix, M::combine(prefix, agg), ctl.epoch);
        } else {
            if (tid == 0 && !last && !skip) publish(ts, g, kStatusAggregate, agg, ctl.epoch);
            if (!block_look_back<M>(g, g - t, ts, ctl, red, ints, &prefix)) {
                if (tid == 0)
                    atomicExch(reinterpret_cast<unsigned long long*>(ctl.error_word), (unsigned long long)ctl.epoch);
                if constexpr (kPrefetch) cp_async_wait<0>();  // no copy may outlive the block
                return;  // uniform: every thread got the same answer
            }
            if (tid == 0 && !last && !skip) publish(ts, g, kStatusPrefix, M::combine(prefix, agg), ctl.epoch);
        }
        if (tid == 0) bcast[1] = prefix;
        __syncthreads();

        // ---- apply prefixes to the run, write back
        const P base = M::combine(M::combine(bcast[1], warp_tot[warp]), lane_excl);
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) run[i] = M::value(M::combine(base, M::lift(run[i])));
        smem_store(L::run_ptr(tile, tid), run);
        __syncthreads();

        // ---- striped store
        const bool vec_out = cnt == tile_elems && (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
        if (vec_out) {
            for (int v = tid; v < tile_elems / VOUT; v += B) {
                Acc a[VOUT];
                smem_load(a, tile + L::elem_off(v * VOUT));
                Out o[VOUT];
#pragma unroll
                for (int q = 0; q < VOUT; ++q) o[q] = convert<Out>(a[q]);
                if constexpr (VOUT > 1) {
                    Raw<16> r;
                    memcpy(&r, o, 16);
                    st_global16(dst + (int64_t)v * VOUT, r);
                } else {
                    dst[v] = o[0];
                }
            }
        } else {
            for (int e = tid; e < cnt; e += B) {
                dst[e] = convert<Out>(*reinterpret_cast<const Acc*>(tile + L::elem_off(e)));
            }
        }
        __syncthreads();  // this buffer is refilled two tiles later
        have = have_next;
        cur ^= 1;
    }
    if constexpr (kPrefetch) cp_async_wait<0>();
}

// Lines along a strided dimension: y[i + I*(j + J*k)] over j, for every
// (i, k). One thread per column (i, k), walking j with rows prefetched.
template <class In, class Acc, class Out, class M>
__global__ void __launch_bounds__(256) k_scan_strided(const In* __restrict__ x, Out* __restrict__ y,
                                                      int64_t I, int64_t J, int64_t K, bool has_init,
                                                      Acc init) {
    using P = typename M::P;
    const int64_t col = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= I * K) return;
    const int64_t i = col % I, k = col / I;
    const In* src = x + i + I * J * k;
    Out* dst = y + i + I * J * k;
    P acc = has_init ? M::lift(init) : M::empty();
    constexpr int U = 4;
    int64_t j = 0;
    for (; j + U <= J; j += U) {
        In v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = src[I * (j + u)];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc = M::combine(acc, M::lift(convert<Acc>(v[u])));
            dst[I * (j + u)] = convert<Out>(M::value(acc));
        }
    }
    for (; j < J; ++j) {
        acc = M::combine(acc, M::lift(convert<Acc>(src[I * j])));
        dst[I * j] = convert<Out>(M::value(acc));
    }
}

template <class In, class Acc, class M>
size_t tile_smem_bytes(int block) {
    using L = RunLayout<Acc, default_items<Acc>()>;
    const size_t bufs = std::is_same_v<In, Acc> ? 2 : 1;
    return bufs * block * L::stride * 16 + (2 * kWarp + 2) * sizeof(typename M::P) + (kWarp + 4) * sizeof(int);
}

template <class In, class Acc, class Out, class M>
ak_status launch(const ScanCall& c, const ScanPlan& p) {
    using P = typename M::P;
    Acc init;
    memcpy(&init, c.init.b, sizeof(Acc));
    if (p.kind == 1) {
        const int64_t cols = c.inner * c.outer;
        const unsigned blocks = (unsigned)((cols + 255) / 256);
        k_scan_strided<In, Acc, Out, M><<<blocks, 256, 0, c.stream>>>(
            static_cast<const In*>(c.src), static_cast<Out*>(c.dst), c.inner, c.len, c.outer, c.has_init, init);
        ak_status s = check_launch();
        if (s == AK_OK) count_launches(1);
        return s;
    }
    constexpr int ITEMS = default_items<Acc>();
    if constexpr (!(ITEMS % (sizeof(In) < 16 ? 16 / sizeof(In) : 1) == 0 &&
                    ITEMS % (sizeof(Out) < 16 ? 16 / sizeof(Out) : 1) == 0)) {
        return AK_ERR_UNSUPPORTED;
    } else {
        auto kernel = k_scan_tiles<In, Acc, Out, M, ITEMS>;
        const size_t smem = tile_smem_bytes<In, Acc, M>(p.block);
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, p.block, smem);
        if (e != cudaSuccess) return cuda_fail(e);
        DeviceInfo dev;
        if (!current_device(&dev)) return AK_ERR_CUDA;
        int64_t grid = std::min<int64_t>(p.tiles, (int64_t)std::max(occ, 1) * dev.sm_count);
        if (c.target_blocks > 0) grid = std::min<int64_t>(grid, c.target_blocks);
        char* ws = static_cast<char*>(c.ws);
        TileState<P> ts;
        ts.flags = reinterpret_cast<uint64_t*>(ws + p.state_off);
        ts.aggs = reinterpret_cast<P*>(ws + p.state_off + align_up((size_t)p.tiles * 8, 16));
        ts.incls = ts.aggs + p.tiles;
        ScanCtl ctl;
        ctl.epoch = c.epoch;
        ctl.error_word = reinterpret_cast<uint64_t*>(ws);  // WsHeader::error_word
        ctl.wait_limit_ns = c.wait_limit_ns;
        ctl.skip_tile = c.skip_tile;
        const In* xs = static_cast<const In*>(c.src);
        Out* ys = static_cast<Out*>(c.dst);
        int64_t len = c.len, tpl = p.tiles_per_line, nt = p.tiles;
        bool hi = c.has_init;
        void* args[] = {(void*)&xs, (void*)&ys, (void*)&len, (void*)&tpl, (void*)&nt, (void*)&ts,
                        (void*)&ctl, (void*)&hi, (void*)&init};
        e = cudaLaunchCooperativeKernel((const void*)kernel, dim3((unsigned)grid), dim3(p.block), args, smem,
                                        c.stream);
        if (e != cudaSuccess) return cuda_fail(e);
        count_launches(1);
        return AK_OK;
    }
}

}  // namespace

ak_status plan_scan(int64_t inner, int64_t len, int64_t outer, ak_dtype in, ak_dtype acc, ak_op op,
                    bool no_neutral, int target_blocks, int items, const DeviceInfo& dev, ScanPlan* p) {
    (void)op;
    (void)target_blocks;
    (void)dev;
    const size_t psz = partial_size(acc, no_neutral);
    const size_t asz = ak_dtype_size(acc);
    if (!psz || !asz) return AK_ERR_UNSUPPORTED;
    p->state_off = kWsHeader;
    p->ws_bytes = kWsHeader;
    p->tiles = 0;
    p->tiles_per_line = 0;
    p->grid = 0;
    if (inner > 1) {
        p->kind = 1;
        p->block = 256;
        p->items = 1;
        return AK_OK;
    }
    p->kind = 0;
    const int it = asz >= 16 ? 8 : (asz == 8 ? 8 : 16);
    if (items != 0 && items != it) return AK_ERR_UNSUPPORTED;
    p->items = it;
    // Block size: the smallest of 128 / 256 / 512 threads whose tile holds a
    // whole line, else 512 (fewer, larger tiles for long lines).
    const int max_block = asz >= 16 ? 256 : kMaxBlock;
    int block = max_block;
    for (int b : {128, 256, 512}) {
        if (b <= max_block && (int64_t)b * it >= len) { block = b; break; }
    }
    p->block = block;
    const int64_t tile = (int64_t)block * it;
    p->tiles_per_line = (len + tile - 1) / tile;
    p->tiles = p->tiles_per_line * outer;
    if (p->tiles_per_line > 1)
        p->ws_bytes = align_up(kWsHeader + align_up((size_t)p->tiles * 8, 16) + 2 * (size_t)p->tiles * psz, 256);
    return AK_OK;
}

ak_status run_scan(const ScanCall& c, const ScanPlan& plan) {
    if (c.in == AK_BF16 || c.out == AK_BF16) return AK_ERR_UNSUPPORTED;
    return dispatch_types(c.in, c.acc, c.out, [&](auto ti, auto ta, auto to) -> ak_status {
        using In = typename decltype(ti)::type;
        using Acc = typename decltype(ta)::type;
        using Out = typename decltype(to)::type;
        if constexpr (std::is_same_v<In, bf16> || std::is_same_v<Out, bf16>) {
            return AK_ERR_UNSUPPORTED;
        } else {
            return dispatch_op<Acc>(c.op, [&](auto top) -> ak_status {
                using Op = typename decltype(top)::type;
                return dispatch_monoid<Op, Acc>(c.no_neutral, [&](auto tmo) -> ak_status {
                    using M = typename decltype(tmo)::type;
                    return launch<In, Acc, Out, M>(c, plan);
                });
            });
        }
    });
}

}  // namespace ak
