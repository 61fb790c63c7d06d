// scan.cuh -- inclusive and exclusive scans (accumulate!, cumsum) on GB300:
// the kernels and their launchers, as templates (compiled into libak for the
// built-in operators and into a caller's translation unit by include/ak.hpp).
//
// The kernels, chosen per call:
//
//  * k_scan_tma -- long contiguous lines of f32 / i32 / i64 with a neutral
//    element, and f64 sums: one persistent block per SM runs a ring of 32 KB
//    tiles copied by the TMA engine through producer, fold, look-back and
//    scan warps (described at the kernel). Every element is read once and
//    written once.
//  * k_scan3_fold / k_scan3_tiles / k_scan3_apply -- other single long
//    lines (f64 max / min / products, the matrix product, Optional
//    partials, mixed input and accumulator types): reduce-then-scan in
//    three launches, no block waiting on another.
//  * k_scan_tiles -- several such lines: persistent blocks claim
//    super-tiles, fold them (phase A) and scan them one round later from L2
//    (phase B).
//  * k_scan_lines -- lines that fit one tile (e.g. dims=1 of a matrix):
//    one block per line, no state shared between blocks.
//  * k_scan_strided -- lines along a strided dimension: a thread per column.
//
// Every kernel also writes the exclusive scan on request: element i then
// holds the fold of init and the elements before it (the store takes the
// running value before the element is combined instead of after).
//
// Tile scan (AcceleratedKernels.jl tile-scan PR #202, first two
// paragraphs): a tile is loaded, each thread scans its own run of
// consecutive elements, the run totals are scanned across the block, and
// the tile's prefix is applied. For lines that fit one tile the runs sit in
// shared memory at an odd stride, as there; the GB300 version of that
// padding is one 16-byte pad after a run whose length is an even number of
// 16-byte chunks, which keeps every run 16-byte aligned, so runs of any
// element size move with 128-bit shared accesses and 8 consecutive threads
// hit 8 distinct bank quads. The TMA path gets the same effect from the
// copy engine's 128-byte swizzle.
//
// Tile prefixes cross tiles in one pass from published tile records (after
// Merrill & Garland, "Single-pass Parallel Prefix Scan with Decoupled
// Look-back", 2016). Tile indices come from an atomic counter claimed by
// running blocks, so every tile a block waits for belongs to a block that
// is already running: progress never depends on the order in which the
// hardware dispatches blocks. Each call clears the counter and the tile
// records on its own stream before the kernel (so a call captured in a CUDA
// graph is correct on every replay), and every record also carries the
// call's epoch and a check word. Every wait is bounded by a global-timer
// deadline; a block that gives up records the epoch in the workspace's
// error word, which every other waiter also watches, and all blocks leave
// early.
#pragma once
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "ak_common.cuh"
#include "ak_internal.h"
#include "ak_tma.cuh"

namespace ak {
namespace scan {

constexpr unsigned kFull = 0xffffffffu;
enum : uint64_t { kStatusAggregate = 1, kStatusPrefix = 2 };

// Run length (items per thread) and block size per accumulator size: 128-byte
// runs, 32 KB tiles for 4- and 8-byte elements (16 KB for 16-byte ones).
template <class Acc>
constexpr int default_items() {
    return sizeof(Acc) >= 16 ? 8 : (sizeof(Acc) == 8 ? 16 : 32);
}
template <class Acc>
constexpr int default_block() {
    return sizeof(Acc) >= 16 ? 128 : 256;
}
// Elements of one thread's segment in the long-line scan: 128 bytes of
// 4-byte accumulators (32 KB super-tiles: the 4-byte types left on this path
// carry Optional partials, whose scans are short enough that more, smaller
// super-tiles keep every block busy), 512 bytes of 8-byte ones and 1 KB of
// 16-byte ones (128 KB super-tiles: more operator work per byte, so more
// bytes per look-back).
template <class Acc>
constexpr int default_seg() {
    return sizeof(Acc) >= 16 ? 64 : (sizeof(Acc) == 8 ? 64 : 32);
}
// Predecessor super-tiles one look-back round inspects, per thread.
constexpr int kLookSlots = 2;
// TMA tile scan: rows of 128 bytes per tile (32 KB tiles), warp roles of
// its one block per SM (warp 0 produces, then the look-back, fold and scan
// warps), and look-back records read per lane per batch.
constexpr int kWsRows = 256;
constexpr int kWsLookWarps = 2;                                   // warps 1..2 look back
constexpr int kWsFoldWarp0 = 1 + kWsLookWarps;                    // warps 3..10 fold
constexpr int kWsScanWarp0 = kWsFoldWarp0 + kWsRows / 32;         // warps 11..18 scan
constexpr int kWsThreads = (kWsScanWarp0 + kWsRows / 32) * 32;    // 608
constexpr int kWsLookQ = 4;
constexpr int kWsLookDefer = 1;  // a look-back also waits for this many later stages to be folded
// Resident blocks per SM the register budget is sized for: 3 blocks of 256
// threads (<= 80 registers a thread); 5 blocks of 128 for 16-byte elements
// (<= 96 registers: the matrix product's chains of dependent products need
// the extra warps to hide their latency more than they need registers).
template <int BLOCK, int ACC_BYTES>
constexpr int min_blocks_per_sm() {
    return ACC_BYTES >= 16 ? 5 : 3;
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

// Tile state without fences: one record per super-tile, rewritten when the
// aggregate is upgraded to the inclusive prefix. A record is written with
// relaxed stores and accepted by a reader only when its tag carries this
// call's epoch and its check word matches the tag and value read with it,
// so a record from an earlier call, arbitrary memory, or a half-visible
// rewrite is rejected and read again (a false acceptance needs a 64-bit
// check collision). Status and value arrive in one read.
template <class P>
struct alignas(16) TileRec {
    uint64_t tag;  // (epoch << 2) | status
    uint64_t chk;
    P v;
};

template <class P>
struct TileState {
    TileRec<P>* recs;
};

template <class P>
__device__ __forceinline__ uint64_t rec_check(uint64_t tag, const P& v) {
    uint64_t h = tag * 0x9E3779B97F4A7C15ull;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(P) / 4); ++i) {
        h = (h ^ w[i]) * 0xBF58476D1CE4E5B9ull;
        h ^= h >> 31;
    }
    return h ^ (h >> 29);
}


// A whole record as 64-bit words, moved with vector accesses: one 32-byte
// access for the 32-byte records (partials of up to 16 bytes), 16-byte
// accesses otherwise. One request per record instead of one per word; a
// read that races a rewrite may still mix old and new words, which the
// check word rejects.
template <class P>
constexpr int rec_words() {
    return (int)(sizeof(TileRec<P>) / 8);
}
template <class P>
__device__ __forceinline__ void rec_load(const TileRec<P>* r, uint64_t (&w)[rec_words<P>()]) {
    constexpr int NW = rec_words<P>();
    const uint64_t* p = reinterpret_cast<const uint64_t*>(r);
    if constexpr (NW == 4) {
        asm volatile("ld.relaxed.gpu.global.v4.u64 {%0,%1,%2,%3}, [%4];"
                     : "=l"(w[0]), "=l"(w[1]), "=l"(w[2]), "=l"(w[3])
                     : "l"(p)
                     : "memory");
    } else {
        static_assert(NW % 2 == 0, "records are whole 16-byte units");
#pragma unroll
        for (int i = 0; i < NW; i += 2)
            asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(w[i]), "=l"(w[i + 1]) : "l"(p + i) : "memory");
    }
}
template <class P>
__device__ __forceinline__ void rec_store(TileRec<P>* r, const uint64_t (&w)[rec_words<P>()]) {
    constexpr int NW = rec_words<P>();
    uint64_t* p = reinterpret_cast<uint64_t*>(r);
    if constexpr (NW == 4) {
        asm volatile("st.relaxed.gpu.global.v4.u64 [%0], {%1,%2,%3,%4};" ::"l"(p), "l"(w[0]), "l"(w[1]), "l"(w[2]),
                     "l"(w[3])
                     : "memory");
    } else {
#pragma unroll
        for (int i = 0; i < NW; i += 2)
            asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" ::"l"(p + i), "l"(w[i]), "l"(w[i + 1]) : "memory");
    }
}
// Status for this call (0 when not valid) and value of a record's words.
template <class P>
__device__ __forceinline__ uint64_t rec_decode(const uint64_t (&w)[rec_words<P>()], uint64_t epoch, P* v) {
    memcpy(v, &w[2], sizeof(P));
    const uint64_t tag = w[0];
    if ((tag >> 2) != epoch || w[1] != rec_check(tag, *v)) return 0;
    return tag & 3u;
}

// Reads a record: its status for this call (0 when not valid) and value.
template <class P>
__device__ __forceinline__ uint64_t read_rec(const TileRec<P>* r, uint64_t epoch, P* v) {
    uint64_t w[rec_words<P>()];
    rec_load(r, w);
    return rec_decode<P>(w, epoch, v);
}

struct ScanCtl {
    uint64_t epoch;
    uint64_t* error_word;
    unsigned long long* counter;  // next tile index (zeroed by the call before the kernel)
    int64_t wait_limit_ns;
    int64_t skip_tile;  // fault injection; -1 = off
};

__device__ __forceinline__ bool aborted(const ScanCtl& ctl) {
    return ld_relaxed_u64(ctl.error_word) == ctl.epoch;
}

// The next tile index of this call: the call zeroes the counter on its
// stream before the kernel (a memset node when the call is captured in a
// CUDA graph), so claims are plain atomic adds in claim order.
__device__ __forceinline__ int64_t claim_tile(const ScanCtl& ctl, int64_t ntiles) {
    (void)ntiles;
    return (int64_t)atomicAdd(ctl.counter, 1ull);
}

// Position of tile k in its line (t = k mod tiles_per_line, line = k div
// tiles_per_line): no 64-bit division (a long emulated sequence on the GPU)
// when the array is one line, one division otherwise.
__device__ __forceinline__ void tile_pos(int64_t k, int64_t tiles_per_line, int64_t ntiles, int64_t* t,
                                         int64_t* line) {
    if (tiles_per_line >= ntiles) {
        *t = k;
        *line = 0;
    } else {
        const int64_t q = k / tiles_per_line;
        *line = q;
        *t = k - q * tiles_per_line;
    }
}

// Ordered combine over the block (thread 0 leftmost); result in thread 0;
// ends with the block in sync.
template <class M, int BLOCK>
__device__ __forceinline__ typename M::P block_reduce_ordered(typename M::P v, typename M::P* red) {
    constexpr int W = BLOCK / kWarp;
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

// Whole block: exclusive prefix of tile g from its predecessors
// g_first..g-1, valid in thread 0. One round inspects the window of
// kLookSlots * BLOCK tiles ending at hi (thread t holds the kLookSlots
// consecutive tiles at 2t, 2t+1 of the window). A round first reads every
// flag once and finds the nearest inclusive prefix, then waits only for the
// tiles newer than it that have not published yet; with none in the window,
// it waits for all of them, folds their aggregates and moves one window
// back. The window is wide enough that the published-prefix frontier keeps
// up with the rate at which tiles start. Returns false (in every thread)
// when a wait ran out or another block gave up.
template <class M, int BLOCK>
__device__ __forceinline__ bool look_back(int64_t g, int64_t g_first, const TileState<typename M::P>& ts,
                                          const ScanCtl& ctl, typename M::P* red, int* ints,
                                          typename M::P* excl0) {
    using P = typename M::P;
    constexpr int W = BLOCK / kWarp, S = kLookSlots, WIN = S * BLOCK;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    // Fast path: warp 0 reads the 32 nearest records once; when an inclusive
    // prefix is among them and every newer one has published, that decides.
    if (warp == 0) {
        const int64_t idx = g - kWarp + lane;
        const bool valid = idx >= g_first;
        P val = M::empty();
        const uint64_t st = valid ? read_rec(ts.recs + idx, ctl.epoch, &val) : 0;
        const unsigned pm = __ballot_sync(kFull, valid && st == kStatusPrefix);
        const int stop = pm ? (kWarp - 1 - __clz(pm)) : -1;
        const bool ok = stop >= 0 && __ballot_sync(kFull, valid && lane > stop && st == 0) == 0;
        if (ok) {
            P v = (valid && lane >= stop) ? val : M::empty();
            v = warp_reduce<M>(v);
            if (lane == 0) *excl0 = v;
        }
        if (lane == 0) ints[2 * kWarp] = ok;
    }
    __syncthreads();
    if (ints[2 * kWarp]) return true;

    P excl = M::empty();
    int64_t hi = g - 1;
    const uint64_t t_start = globaltimer_ns();
    while (true) {
        const int64_t base = hi - (WIN - 1) + (int64_t)S * tid;  // this thread's first slot
        uint64_t st[S];
        P val[S];
#pragma unroll
        for (int k = 0; k < S; ++k) {
            st[k] = 0;
            val[k] = M::empty();
            if (base + k >= g_first) st[k] = read_rec(ts.recs + base + k, ctl.epoch, &val[k]);
        }
        // nearest inclusive prefix seen so far: the highest window position
        int mine = -1;
#pragma unroll
        for (int k = 0; k < S; ++k)
            if (base + k >= g_first && st[k] == kStatusPrefix) mine = S * tid + k;
        for (int d = kWarp / 2; d > 0; d >>= 1) mine = max(mine, __shfl_xor_sync(kFull, mine, d));
        if (lane == 0) ints[warp] = mine;
        __syncthreads();
        int stop0 = -1;
#pragma unroll
        for (int w = 0; w < W; ++w) stop0 = max(stop0, ints[w]);
        // wait for the unpublished tiles newer than it
        bool fail = false;
#pragma unroll
        for (int k = 0; k < S; ++k) {
            const int pos = S * tid + k;
            if (base + k >= g_first && pos > stop0 && st[k] == 0) {
                while (true) {
                    st[k] = read_rec(ts.recs + base + k, ctl.epoch, &val[k]);
                    if (st[k] != 0) break;
                    if (globaltimer_ns() - t_start > (uint64_t)ctl.wait_limit_ns || aborted(ctl)) {
                        fail = true;
                        break;
                    }
                    __nanosleep(32);
                }
            }
        }
        if (__syncthreads_or(fail)) return false;
        // a newer tile may have published its prefix meanwhile: use the nearest
        mine = -1;
#pragma unroll
        for (int k = 0; k < S; ++k)
            if (base + k >= g_first && S * tid + k >= stop0 && st[k] == kStatusPrefix) mine = S * tid + k;
        for (int d = kWarp / 2; d > 0; d >>= 1) mine = max(mine, __shfl_xor_sync(kFull, mine, d));
        if (lane == 0) ints[kWarp + warp] = mine;
        __syncthreads();
        int stop = -1;
#pragma unroll
        for (int w = 0; w < W; ++w) stop = max(stop, ints[kWarp + w]);
        // fold the window from the prefix (or its start) to its end, in order
        P v = M::empty();
#pragma unroll
        for (int k = 0; k < S; ++k) {
            const int pos = S * tid + k;
            if (base + k < g_first || pos < stop) continue;
            v = M::combine(v, val[k]);
        }
        v = block_reduce_ordered<M, BLOCK>(v, red);
        if (tid == 0) excl = M::combine(v, excl);
        if (stop >= 0 || hi - WIN < g_first) break;
        hi -= WIN;
    }
    if (tid == 0) *excl0 = excl;
    return true;
}

template <class P>
__device__ __forceinline__ void publish(const TileState<P>& ts, int64_t g, uint64_t status, const P& v,
                                        uint64_t epoch) {
    const uint64_t tag = (epoch << 2) | status;
    uint64_t w[rec_words<P>()];
#pragma unroll
    for (int i = 0; i < rec_words<P>(); ++i) w[i] = 0;
    w[0] = tag;
    w[1] = rec_check(tag, v);
    memcpy(&w[2], &v, sizeof(P));
    rec_store(ts.recs + g, w);
}

// ---------------------------------------------------------------------------
// tile building blocks
// ---------------------------------------------------------------------------

// Striped (coalesced) load of one tile into the padded run layout, with the
// given L2 policy; a ragged or unaligned tile is loaded element by element
// and padded with zero bytes.
template <class In, class Acc, int ITEMS, int BLOCK>
__device__ __forceinline__ void load_tile(char* tile, const In* src, int cnt, uint64_t policy) {
    using L = RunLayout<Acc, ITEMS>;
    constexpr int TILE = BLOCK * ITEMS;
    constexpr int VIN = sizeof(In) < 16 ? 16 / (int)sizeof(In) : 1;
    static_assert(ITEMS % VIN == 0, "runs must hold whole vectors");
    const int tid = threadIdx.x;
    if (cnt == TILE && reinterpret_cast<uintptr_t>(src) % 16 == 0) {
#pragma unroll
        for (int k = 0; k < TILE / VIN / BLOCK; ++k) {
            const int v = tid + k * BLOCK;
            In e[VIN];
            Raw<16> r = ld_hint16(src + (int64_t)v * VIN, policy);
            memcpy(e, &r, sizeof e);
            Acc a[VIN];
#pragma unroll
            for (int q = 0; q < VIN; ++q) a[q] = convert<Acc>(e[q]);
            smem_store(tile + L::elem_off(v * VIN), a);
        }
    } else {
        for (int e = tid; e < TILE; e += BLOCK) {
            Acc a;
            if (e < cnt) a = convert<Acc>(src[e]);
            else memset(&a, 0, sizeof a);
            *reinterpret_cast<Acc*>(tile + L::elem_off(e)) = a;
        }
    }
}

// Scan of the tile in shared memory with the tile's exclusive prefix
// (`*prefix`, shared), then the coalesced store of the result; `*prefix`
// then becomes the inclusive prefix of the tile (the next tile's carry).
template <class Acc, class Out, class M, int ITEMS, int BLOCK>
__device__ __forceinline__ void scan_apply_store(char* tile, Out* dst, int cnt, typename M::P* prefix,
                                                 typename M::P* warp_tot, uint64_t policy, bool excl) {
    using P = typename M::P;
    using L = RunLayout<Acc, ITEMS>;
    constexpr int W = BLOCK / kWarp;
    constexpr int TILE = BLOCK * ITEMS;
    constexpr int VOUT = sizeof(Out) < 16 ? 16 / (int)sizeof(Out) : 1;
    static_assert(ITEMS % VOUT == 0, "runs must hold whole vectors");
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;

    // each thread scans its run in registers
    Acc run[ITEMS];
    smem_load(run, L::run_ptr(tile, tid));
#pragma unroll
    for (int i = 1; i < ITEMS; ++i) run[i] = M::op::apply(run[i - 1], run[i]);
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
    // block scan of run totals (thread order)
    P inc = warp_inclusive_scan<M>(total, lane);
    P lane_excl = shfl_up_any(inc, 1);
    if (lane == 0) lane_excl = M::empty();
    if (lane == kWarp - 1) warp_tot[warp] = inc;
    __syncthreads();
    P block_total = M::empty();  // meaningful in warp 0
    if (warp == 0) {
        P w = lane < W ? warp_tot[lane] : M::empty();
        P wi = warp_inclusive_scan<M>(w, lane);
        P we = shfl_up_any(wi, 1);
        if (lane == 0) we = M::empty();
        if (lane < W) warp_tot[lane] = M::combine(*prefix, we);  // tile prefix + exclusive base of each warp
        block_total = shfl_idx_any(wi, W - 1);
    }
    __syncthreads();
    // apply the prefixes to the run, write back (exclusive: element i takes
    // the inclusive value of element i - 1, the first one the run's prefix,
    // which is present: an exclusive scan always starts from init)
    const P base = M::combine(warp_tot[warp], lane_excl);
    if (excl) {
        Acc prev = M::value(base);
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const Acc cur = M::value(M::combine(base, M::lift(run[i])));
            run[i] = prev;
            prev = cur;
        }
    } else {
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) run[i] = M::value(M::combine(base, M::lift(run[i])));
    }
    smem_store(L::run_ptr(tile, tid), run);
    __syncthreads();
    // striped (coalesced) store
    if (cnt == TILE && reinterpret_cast<uintptr_t>(dst) % 16 == 0) {
#pragma unroll
        for (int k = 0; k < TILE / VOUT / BLOCK; ++k) {
            const int v = tid + k * BLOCK;
            Acc a[VOUT];
            smem_load(a, tile + L::elem_off(v * VOUT));
            Out o[VOUT];
#pragma unroll
            for (int q = 0; q < VOUT; ++q) o[q] = convert<Out>(a[q]);
            Raw<16> r;
            memcpy(&r, o, 16);
            st_hint16(dst + (int64_t)v * VOUT, r, policy);
        }
    } else {
        for (int e = tid; e < cnt; e += BLOCK) dst[e] = convert<Out>(*reinterpret_cast<const Acc*>(tile + L::elem_off(e)));
    }
    if (tid == 0) *prefix = M::combine(*prefix, block_total);  // carry into the next sub-tile
    __syncthreads();  // the tile buffer and the carry are used next
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// register-resident segments
// ---------------------------------------------------------------------------

// Each thread of a super-tile owns one contiguous segment of SEG elements,
// read and written with 32-byte (256-bit) per-lane accesses: every access
// is a whole sector, so a warp's blocked accesses use each DRAM / L2 sector
// fully and no shared-memory transpose is needed.
template <class In>
__host__ __device__ constexpr int chunk_elems() {
    return 32 / (int)sizeof(In);
}

// Sum of a row of doubles in 64-bit fixed point, off the FP64 pipe (GB300
// issues two FP64 additions per clock per SM, so a scan that adds every
// element twice in FP64 is bound by that pipe, not by HBM). Every element is
// aligned to the row's largest exponent with 6 guard bits below that
// element's last mantissa bit (16 aligned values of at most 59 bits cannot
// overflow 63 bits), negated by its sign and added exactly; bits shifted out
// are truncated, an error below 16 * 2^-6 units in the last place of the
// largest element, far inside the f64 scan tolerance. The integer sum is
// rounded to double once. Rows holding an infinity or NaN (exponent field all
// ones) or only zeros and subnormals (field all zeros) take the plain FP64
// fold, which keeps IEEE specials and the sign of zero exact.
template <int R>
__device__ __forceinline__ double row_sum_fixed(const double (&run)[R]) {
    uint32_t e[R];
    uint32_t emax = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        e[i] = ((uint32_t)__double2hiint(run[i]) >> 20) & 0x7FFu;
        emax = max(emax, e[i]);
    }
    if (emax == 0x7FFu || emax == 0u) {
        double a = run[0];
#pragma unroll
        for (int i = 1; i < R; ++i) a += run[i];
        return a;
    }
    int64_t sum = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const uint64_t bits = (uint64_t)__double_as_longlong(run[i]);
        const uint64_t m = (bits & 0x000FFFFFFFFFFFFFull) | (e[i] != 0u ? (1ull << 52) : 0ull);
        const uint32_t sh = emax - max(e[i], 1u);
        const int64_t q = sh >= 64u ? 0 : (int64_t)((m << 6) >> sh);
        sum += (bits >> 63) ? -q : q;
    }
    // sum * 2^(emax - 1075 - 6): one rounding in the conversion, the scaling by
    // a power of two is exact unless the result is subnormal
    return scalbn((double)sum, (int)emax - 1081);
}

// Wide fixed point for f64 sums on the integer pipes (GB300 runs FP64 at a
// small fraction of its integer rate, so the TMA scan of f64 sums keeps
// FP64 off the per-element path). A partial is (a, e): the value
// a * 2^(e - kFxK), a a signed 64-bit integer, e >= 1 a biased binary
// exponent. A finite double enters exactly, at its own exponent with kFxG
// guard bits; two partials add at the larger exponent (the other one's bits
// below it are truncated, an error under one unit there); a partial is
// renormalised to at most L significant bits before headroom runs out. Every
// truncation is below 2^-53 of a magnitude that the sum of |x| over the
// elements involved bounds, far inside the f64 scan tolerance.
struct Fx {
    int64_t a;
    int32_t e;
    int32_t pad;
};
constexpr int kFxG = 3;
constexpr int kFxK = 1075 + kFxG;
constexpr uint64_t kF64Frac = 0x000FFFFFFFFFFFFFull;
constexpr uint64_t kF64NegZero = 0x8000000000000000ull;

__device__ __forceinline__ Fx fx_zero() { return Fx{0, 1, 0}; }

// a >> d for d >= 0 (arithmetic; d >= 64 leaves the sign)
__device__ __forceinline__ int64_t fx_shr(int64_t a, int d) { return a >> min(d, 63); }

__device__ __forceinline__ Fx fx_add(const Fx& x, const Fx& y) {
    const int e = max(x.e, y.e);
    return Fx{fx_shr(x.a, e - x.e) + fx_shr(y.a, e - y.e), e, 0};
}

// |a| < 2^L afterwards
__device__ __forceinline__ Fx fx_norm(Fx x, int L) {
    const uint64_t m = (uint64_t)(x.a < 0 ? -x.a : x.a);
    const int s = max(0, 64 - __clzll((long long)m) - L);
    x.a >>= s;
    x.e += s;
    return x;
}

// A finite double, exactly (|a| < 2^56).
__device__ __forceinline__ Fx fx_of(double v) {
    const uint64_t b = (uint64_t)__double_as_longlong(v);
    const int f = (int)((b >> 52) & 0x7FFu);
    const int64_t m = (int64_t)(((b & kF64Frac) | (f != 0 ? 1ull << 52 : 0ull)) << kFxG);
    return Fx{(b >> 63) ? -m : m, max(f, 1), 0};
}

// Rounded to the nearest double (ties away from zero); zero gives +0. A
// result below the normal range or above the largest double takes the
// library scaling (rare).
__device__ __forceinline__ double fx_to_double(const Fx& x) {
    if (x.a == 0) return 0.0;
    const uint64_t mag = (uint64_t)(x.a < 0 ? -x.a : x.a);
    const int lz = __clzll((long long)mag);
    const uint64_t nm = mag << lz;  // leading one at bit 63
    // nm >> 11 is the 53-bit significand, the value nm * 2^(e - kFxK - lz)
    const int B = x.e - kFxG - lz + 11;
    if (B < 1 || B > 2046) return scalbn((double)x.a, x.e - kFxK);
    // a carry out of the significand moves into the exponent field
    const uint64_t bits = ((uint64_t)(B - 1) << 52) + (nm >> 11) + ((nm >> 10) & 1u);
    return __longlong_as_double((long long)(bits | (x.a < 0 ? kF64NegZero : 0ull)));
}

__device__ __forceinline__ Fx fx_shfl_up(const Fx& v, int d) {
    return Fx{(int64_t)__shfl_up_sync(0xffffffffu, (long long)v.a, d), __shfl_up_sync(0xffffffffu, v.e, d), 0};
}
__device__ __forceinline__ Fx fx_shfl_idx(const Fx& v, int lane) {
    return Fx{(int64_t)__shfl_sync(0xffffffffu, (long long)v.a, lane), __shfl_sync(0xffffffffu, v.e, lane), 0};
}

// Sum of a row of doubles at the row's largest exponent: the 53-bit
// significands are aligned there without guard bits (each truncation is
// under one unit in the last place of the row's largest element) and the
// guard scale goes into the exponent (|a| < 2^57). *fmax is the largest
// exponent field: 0x7FF when the row holds an infinity or a NaN, 0 when it
// holds only zeros and subnormals (the caller then takes the FP64 path,
// which keeps IEEE specials and signed zeros).
template <int R>
__device__ __forceinline__ Fx row_total_fx(const double (&run)[R], int* fmax) {
    int f[R];
    int fm = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        f[i] = (int)(((uint32_t)__double2hiint(run[i]) >> 20) & 0x7FFu);
        fm = max(fm, f[i]);
    }
    const int emax = max(fm, 1);
    int64_t sum = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const uint64_t b = (uint64_t)__double_as_longlong(run[i]);
        const uint64_t m = (b & kF64Frac) | (f[i] != 0 ? 1ull << 52 : 0ull);
        const int64_t q = (int64_t)(m >> min(emax - max(f[i], 1), 63));
        sum += (b >> 63) ? -q : q;
    }
    *fmax = fm;
    return Fx{sum, emax + kFxG, 0};
}

// Fold of one segment (n <= SEG valid elements) in element order.
template <class In, class M, int SEG>
__device__ __forceinline__ typename M::P segment_fold(const In* src, int n, uint64_t policy) {
    using P = typename M::P;
    using Acc = typename M::acc;
    constexpr int CH = chunk_elems<In>();
    constexpr int NC = SEG / CH;
    constexpr int U = NC < 8 ? NC : 8;
    static_assert(SEG % CH == 0 && NC % U == 0, "whole chunks per segment");
    if (n == SEG && reinterpret_cast<uintptr_t>(src) % 32 == 0) {
        if constexpr (std::is_same_v<In, double> && std::is_same_v<typename M::P, double> &&
                      std::is_same_v<typename M::op, OpAdd> && SEG % 16 == 0 && 16 % CH == 0) {
            // groups of 16 summed in fixed point, the group sums added in FP64
            // (16 elements = 4 loads in flight at a time: room for the integer work)
            P a = M::empty();
            constexpr int U4 = 16 / CH;
#pragma unroll 1
            for (int c0 = 0; c0 < NC; c0 += U4) {
                Raw<32> r[U4];
#pragma unroll
                for (int u = 0; u < U4; ++u) r[u] = ld_hint32(src + (c0 + u) * CH, policy);
#pragma unroll
                for (int g = 0; g < U4 * CH / 16; ++g) {
                    double grp[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) grp[e] = raw_get<double>(r[(g * 16 + e) / CH], (g * 16 + e) % CH);
                    a += row_sum_fixed(grp);
                }
            }
            return a;
        } else if constexpr (M::commutative) {
            // one accumulator per chunk position: short dependency chains
            P acc[CH];
#pragma unroll
            for (int q = 0; q < CH; ++q) acc[q] = M::empty();
#pragma unroll 1
            for (int c0 = 0; c0 < NC; c0 += U) {
                Raw<32> r[U];
#pragma unroll
                for (int u = 0; u < U; ++u) r[u] = ld_hint32(src + (c0 + u) * CH, policy);
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int q = 0; q < CH; ++q)
                        acc[q] = M::combine(acc[q], M::lift(convert<Acc>(raw_get<In>(r[u], q))));
            }
            P a = acc[0];
#pragma unroll
            for (int q = 1; q < CH; ++q) a = M::combine(a, acc[q]);
            return a;
        } else {
            P a = M::empty();
#pragma unroll 1
            for (int c0 = 0; c0 < NC; c0 += U) {
                Raw<32> r[U];
#pragma unroll
                for (int u = 0; u < U; ++u) r[u] = ld_hint32(src + (c0 + u) * CH, policy);
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int q = 0; q < CH; ++q) a = M::combine(a, M::lift(convert<Acc>(raw_get<In>(r[u], q))));
            }
            return a;
        }
    }
    P a = M::empty();
    for (int i = 0; i < n; ++i) a = M::combine(a, M::lift(convert<Acc>(src[i])));
    return a;
}

// Stores the CH outputs of one chunk (CH * sizeof(Out) bytes: 16, 32 or 64).
template <class Out, int CH>
__device__ __forceinline__ void store_chunk(Out* dst, const Out (&o)[CH], uint64_t policy) {
    constexpr int NB = CH * (int)sizeof(Out);
    if constexpr (NB == 16) {
        Raw<16> r;
        memcpy(&r, o, 16);
        st_hint16(dst, r, policy);
    } else {
        static_assert(NB % 32 == 0, "chunk of whole sectors");
#pragma unroll
        for (int h = 0; h < NB / 32; ++h) {
            Raw<32> r;
            memcpy(&r, reinterpret_cast<const char*>(o) + 32 * h, 32);
            st_hint32(reinterpret_cast<char*>(dst) + 32 * h, r, policy);
        }
    }
}

// Inclusive scan of one segment starting from the exclusive prefix `acc`,
// stored to dst.
template <class In, class Out, class M, int SEG>
__device__ __forceinline__ void segment_scan_store(const In* src, Out* dst, int n, typename M::P acc,
                                                   uint64_t pol_in, uint64_t pol_out, bool excl) {
    using Acc = typename M::acc;
    constexpr int CH = chunk_elems<In>();
    constexpr int NC = SEG / CH;
    constexpr int U = NC < 8 ? NC : 8;
    constexpr int OB = CH * (int)sizeof(Out);
    if (n == SEG && reinterpret_cast<uintptr_t>(src) % 32 == 0 &&
        reinterpret_cast<uintptr_t>(dst) % (OB < 32 ? OB : 32) == 0) {
#pragma unroll 1
        for (int c0 = 0; c0 < NC; c0 += U) {
            Raw<32> r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) r[u] = ld_hint32(src + (c0 + u) * CH, pol_in);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                Out o[CH];
#pragma unroll
                for (int q = 0; q < CH; ++q) {
                    const typename M::P before = acc;
                    acc = M::combine(acc, M::lift(convert<Acc>(raw_get<In>(r[u], q))));
                    o[q] = convert<Out>(M::value(excl ? before : acc));
                }
                store_chunk<Out, CH>(dst + (c0 + u) * CH, o, pol_out);
            }
        }
        return;
    }
    for (int i = 0; i < n; ++i) {
        const typename M::P before = acc;
        acc = M::combine(acc, M::lift(convert<Acc>(src[i])));
        dst[i] = convert<Out>(M::value(excl ? before : acc));
    }
}

// Lines that span several super-tiles of BLOCK x SEG elements. A persistent
// block repeats: claim the next super-tile k; phase A of k -- every thread
// streams its segment from HBM with an L2 evict-last hint and folds it, the
// block keeps the segment totals in shared memory, reduces them in order
// and publishes the super-tile's aggregate (for a line's first super-tile,
// its inclusive prefix); then phase B of the super-tile it claimed one round
// earlier -- look back to its exclusive prefix, publish its inclusive
// prefix, scan the kept segment totals across the block, and every thread
// walks its segment again (now from L2) from its own exclusive prefix,
// storing as it goes. Phase A never waits, so every claimed super-tile's
// aggregate appears promptly, and by the time a block looks back its
// predecessors have long published: the waiting that a one-pass tile scan
// does with the tile held in shared memory is done here with the data
// parked in the 129 MB L2. HBM traffic stays one read and one write per
// element; the operator is applied twice per element.
template <class In, class Acc, class Out, class M, int BLOCK, int SEG>
__global__ void __launch_bounds__(BLOCK, min_blocks_per_sm<BLOCK, (int)sizeof(Acc)>())
    k_scan_tiles(const In* __restrict__ x, Out* __restrict__ y, int64_t len, int64_t tiles_per_line, int64_t ntiles,
                 TileState<typename M::P> ts, ScanCtl ctl, bool has_init, Acc init, bool excl) {
    using P = typename M::P;
    constexpr int W = BLOCK / kWarp;
    constexpr int64_t SUPER = (int64_t)BLOCK * SEG;
    __shared__ P seg_tot[2][BLOCK];  // segment totals of the two open super-tiles
    __shared__ P warp_tot[W];
    __shared__ P red[W];
    __shared__ int ints[2 * kWarp + 1];
    __shared__ P s_bc;
    __shared__ int64_t s_k;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t last_use = l2_policy_evict_first();

    int64_t prev = -1;
    P prev_agg = M::empty();
    int slot = 0;
    while (true) {
        if (tid == 0) s_k = claim_tile(ctl, ntiles);
        __syncthreads();
        const int64_t k = s_k;
        P agg = M::empty();
        if (k < ntiles) {
            // ---- phase A of super-tile k
            int64_t t, line;
            tile_pos(k, tiles_per_line, ntiles, &t, &line);
            const int64_t start = line * len + t * SUPER;
            const int64_t cnt = min(SUPER, len - t * SUPER);
            const int n = (int)max((int64_t)0, min((int64_t)SEG, cnt - (int64_t)tid * SEG));
            const P tot = n > 0 ? segment_fold<In, M, SEG>(x + start + (int64_t)tid * SEG, n, keep) : M::empty();
            seg_tot[slot][tid] = tot;
            if (tiles_per_line > 1) {
                agg = block_reduce_ordered<M, BLOCK>(tot, red);
                const bool last = (t == tiles_per_line - 1);
                if (tid == 0 && !last && k != ctl.skip_tile) {
                    if (t == 0) publish(ts, k, kStatusPrefix, M::combine(has_init ? M::lift(init) : M::empty(), agg), ctl.epoch);
                    else publish(ts, k, kStatusAggregate, agg, ctl.epoch);
                }
            }
        }
        if (prev >= 0) {
            // ---- phase B of super-tile prev
            const int pslot = slot ^ 1;
            int64_t t, line;
            tile_pos(prev, tiles_per_line, ntiles, &t, &line);
            const int64_t start = line * len + t * SUPER;
            const int64_t cnt = min(SUPER, len - t * SUPER);
            P prefix = has_init ? M::lift(init) : M::empty();
            if (t != 0) {
                if (!look_back<M, BLOCK>(prev, prev - t, ts, ctl, red, ints, &prefix)) {
                    if (tid == 0)
                        atomicExch(reinterpret_cast<unsigned long long*>(ctl.error_word), (unsigned long long)ctl.epoch);
                    return;  // uniform: every thread got the same answer
                }
                if (tid == 0 && t != tiles_per_line - 1 && prev != ctl.skip_tile)
                    publish(ts, prev, kStatusPrefix, M::combine(prefix, prev_agg), ctl.epoch);
                if (tid == 0) s_bc = prefix;
                __syncthreads();
                prefix = s_bc;
            }
            // exclusive prefix of this thread's segment: prefix + earlier segments
            const P tot = seg_tot[pslot][tid];
            const P inc = warp_inclusive_scan<M>(tot, lane);
            P lane_excl = shfl_up_any(inc, 1);
            if (lane == 0) lane_excl = M::empty();
            if (lane == kWarp - 1) warp_tot[warp] = inc;
            __syncthreads();
            if (warp == 0) {
                const P w = lane < W ? warp_tot[lane] : M::empty();
                const P wi = warp_inclusive_scan<M>(w, lane);
                P we = shfl_up_any(wi, 1);
                if (lane == 0) we = M::empty();
                if (lane < W) warp_tot[lane] = we;
            }
            __syncthreads();
            const P mine = M::combine(M::combine(prefix, warp_tot[warp]), lane_excl);
            const int n = (int)max((int64_t)0, min((int64_t)SEG, cnt - (int64_t)tid * SEG));
            if (n > 0)
                segment_scan_store<In, Out, M, SEG>(x + start + (int64_t)tid * SEG, y + start + (int64_t)tid * SEG, n,
                                                    mine, last_use, last_use, excl);
            __syncthreads();  // warp_tot and the slot are reused next
        }
        if (k >= ntiles) break;
        prev = k;
        prev_agg = agg;
        slot ^= 1;
    }
}

// ---------------------------------------------------------------------------
// Reduce-then-scan in three launches, for single long lines
// ---------------------------------------------------------------------------
//
// A single long line outside the TMA scan (matrices, Optional partials,
// mixed types, f64 operators other than the sum) is scanned by three
// launches chained with
// programmatic dependent launch, without any wait between blocks:
//   fold   block t folds super-tile t: its segment totals and its aggregate
//          go to the workspace, the tile is kept in L2 (evict_last);
//   tiles  one block scans the aggregates into each tile's exclusive prefix
//          (init at the front) -- or, for up to kFusedPrefixTiles tiles, each
//          apply block folds the aggregates before it itself;
//   apply  block t scans its segment totals from its prefix and every thread
//          walks its segment again, storing as it goes.
// A line that fits L2 is read from HBM once (the second read hits); a longer
// one pays part of the second read, but on GB300 the single-pass super-tile
// scan, whose blocks wait on each other's look-backs, is slower at every
// length measured. The operator is applied twice per element either way.

constexpr int kTilesBlock = 1024;  // threads of the one-block tile-prefix scan
// Up to this many tiles the apply blocks fold the aggregates before them
// themselves (at most this many reads per block, from L2).
constexpr int64_t kFusedPrefixTiles = 2048;

template <class In, class M, int BLOCK, int SEG>
__global__ void __launch_bounds__(BLOCK) k_scan3_fold(const In* __restrict__ x, int64_t len,
                                                      typename M::P* __restrict__ seg_out,
                                                      typename M::P* __restrict__ agg_out, uint64_t* error_word) {
    using P = typename M::P;
    constexpr int W = BLOCK / kWarp;
    constexpr int64_t SUPER = (int64_t)BLOCK * SEG;
    __shared__ P red[W];
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    if (t == 0 && tid == 0) *error_word = 0;  // no waits in this scan: the call's status is ok
    const int64_t start = t * SUPER + (int64_t)tid * SEG;
    const int n = (int)max((int64_t)0, min((int64_t)SEG, len - start));
    const P tot = n > 0 ? segment_fold<In, M, SEG>(x + start, n, l2_policy_evict_last()) : M::empty();
    seg_out[t * BLOCK + tid] = tot;
    griddep_launch_dependents();
    const P agg = block_reduce_ordered<M, BLOCK>(tot, red);
    if (tid == 0) agg_out[t] = agg;
}

// One block: pre[t] = init (or empty) combined with agg[0 .. t-1]. Thread r
// folds a contiguous run of tiles, the runs are scanned across the block in
// order, then every thread writes its tiles' prefixes.
template <class M>
__global__ void __launch_bounds__(kTilesBlock) k_scan3_tiles(const typename M::P* __restrict__ agg,
                                                             typename M::P* __restrict__ pre, int64_t ntiles,
                                                             bool has_init, typename M::acc init) {
    using P = typename M::P;
    constexpr int W = kTilesBlock / kWarp;
    __shared__ P wt[W];
    griddep_wait();
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int64_t per = (ntiles + kTilesBlock - 1) / kTilesBlock;
    const int64_t t0 = min(ntiles, (int64_t)tid * per), t1 = min(ntiles, t0 + per);
    P run = M::empty();
    for (int64_t t = t0; t < t1; ++t) run = M::combine(run, agg[t]);
    const P inc = warp_inclusive_scan<M>(run, lane);
    P lane_excl = shfl_up_any(inc, 1);
    if (lane == 0) lane_excl = M::empty();
    if (lane == kWarp - 1) wt[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const P w = lane < W ? wt[lane] : M::empty();
        const P wi = warp_inclusive_scan<M>(w, lane);
        P we = shfl_up_any(wi, 1);
        if (lane == 0) we = M::empty();
        wt[lane] = we;
    }
    __syncthreads();
    griddep_launch_dependents();
    P a = M::combine(M::combine(has_init ? M::lift(init) : M::empty(), wt[warp]), lane_excl);
    for (int64_t t = t0; t < t1; ++t) {
        pre[t] = a;
        a = M::combine(a, agg[t]);
    }
}

// Block t scans tile t. Its exclusive prefix comes from k_scan3_tiles
// (pre != nullptr), or (pre == nullptr) the block folds it itself: init (or
// the neutral element) combined with the aggregates of tiles 0 .. t-1, the
// threads taking consecutive runs that are combined in order.
template <class In, class Acc, class Out, class M, int BLOCK, int SEG>
__global__ void __launch_bounds__(BLOCK, min_blocks_per_sm<BLOCK, (int)sizeof(Acc)>())
    k_scan3_apply(const In* __restrict__ x, Out* __restrict__ y, int64_t len,
                  const typename M::P* __restrict__ seg_tot, const typename M::P* __restrict__ pre,
                  const typename M::P* __restrict__ agg, bool has_init, Acc init, bool excl) {
    using P = typename M::P;
    constexpr int W = BLOCK / kWarp;
    constexpr int64_t SUPER = (int64_t)BLOCK * SEG;
    __shared__ P warp_tot[W];
    __shared__ P red[W];
    __shared__ P s_pre;
    griddep_wait();
    // last tile first: the fold went first to last, so the end of a line
    // longer than L2 is what its evict_last reads left there
    const int64_t t = (int64_t)gridDim.x - 1 - blockIdx.x;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    if (pre == nullptr) {
        const int64_t per = (t + BLOCK - 1) / BLOCK;
        const int64_t a0 = min(t, (int64_t)tid * per), a1 = min(t, a0 + per);
        P f = M::empty();
#pragma unroll 4
        for (int64_t q = a0; q < a1; ++q) f = M::combine(f, agg[q]);
        f = block_reduce_ordered<M, BLOCK>(f, red);
        if (tid == 0) s_pre = M::combine(has_init ? M::lift(init) : M::empty(), f);
        __syncthreads();
    }
    const P tile_pre = pre == nullptr ? s_pre : pre[t];
    const P tot = seg_tot[t * BLOCK + tid];
    const P inc = warp_inclusive_scan<M>(tot, lane);
    P lane_excl = shfl_up_any(inc, 1);
    if (lane == 0) lane_excl = M::empty();
    if (lane == kWarp - 1) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const P w = lane < W ? warp_tot[lane] : M::empty();
        const P wi = warp_inclusive_scan<M>(w, lane);
        P we = shfl_up_any(wi, 1);
        if (lane == 0) we = M::empty();
        if (lane < W) warp_tot[lane] = we;
    }
    __syncthreads();
    const P mine = M::combine(M::combine(tile_pre, warp_tot[warp]), lane_excl);
    const int64_t start = t * SUPER + (int64_t)tid * SEG;
    const int n = (int)max((int64_t)0, min((int64_t)SEG, len - start));
    const uint64_t last_use = l2_policy_evict_first();
    if (n > 0) segment_scan_store<In, Out, M, SEG>(x + start, y + start, n, mine, last_use, last_use, excl);
}

// ---------------------------------------------------------------------------
// TMA tile scan: one read and one write of every element
// ---------------------------------------------------------------------------

// Stages of the ring and the block's dynamic shared memory: each stage
// holds a tile and its rows' in-tile prefixes; plus slack to align the
// tiles to the 1024 bytes that the 128-byte swizzle pattern repeats over.
template <class P>
constexpr int ws_stages() {
    return sizeof(P) <= 16 ? 6 : 5;
}
// f64 sums keep their in-tile row prefixes as wide fixed-point partials.
template <class T, class M>
constexpr bool ws_fx() {
    return std::is_same_v<T, double> && std::is_same_v<typename M::op, OpAdd>;
}
template <class T, class M>
constexpr int ws_rowpre_bytes() {
    return ws_fx<T, M>() ? (int)sizeof(Fx) : (int)sizeof(typename M::P);
}
template <class T, class M>
constexpr int ws_smem_bytes() {
    return ws_stages<typename M::P>() * (kWsRows * 128 + kWsRows * ws_rowpre_bytes<T, M>()) + 1024;
}

// Row r of a swizzled tile <-> the R elements of a thread, 16 bytes at a time.
template <class T, int R>
__device__ __forceinline__ void row_load(T (&run)[R], const unsigned char* buf, int r) {
    static_assert(R * sizeof(T) == 128 && sizeof(T) % 4 == 0 && sizeof(T) <= 16, "128-byte rows of word-sized elements");
    constexpr int WPE = sizeof(T) / 4, E = 16 / sizeof(T);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = *reinterpret_cast<const uint4*>(buf + swz128(r, j));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < E; ++k) {
            uint32_t e[WPE];
#pragma unroll
            for (int q = 0; q < WPE; ++q) e[q] = w[k * WPE + q];
            memcpy(&run[j * E + k], e, sizeof(T));
        }
    }
}

// A thread's row straight to global memory: 32-byte stores when the row is
// 32-byte aligned, else 16-byte ones; the L2 is told this is a last use.
template <class T, int R>
__device__ __forceinline__ void row_store_global(T* dst, const T (&run)[R], uint64_t policy) {
    static_assert(R * sizeof(T) == 128, "128-byte rows");
    const uint32_t* w = reinterpret_cast<const uint32_t*>(run);
    if (reinterpret_cast<uintptr_t>(dst) % 32 == 0) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            Raw<32> r;
#pragma unroll
            for (int q = 0; q < 8; ++q) r.w[q] = w[8 * h + q];
            st_hint32(reinterpret_cast<char*>(dst) + 32 * h, r, policy);
        }
    } else {
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            Raw<16> r;
#pragma unroll
            for (int q = 0; q < 4; ++q) r.w[q] = w[4 * h + q];
            st_hint16(reinterpret_cast<char*>(dst) + 16 * h, r, policy);
        }
    }
}

// Fold of a whole row: in element order, or for a commutative operator as
// four interleaved chains combined at the end (independent operations in
// flight; a reordering that only rounding can tell apart).
template <class M, class T, int R>
__device__ __forceinline__ T row_fold(const T (&run)[R]) {
    if constexpr (M::commutative && R % 4 == 0) {
        T c[4] = {run[0], run[1], run[2], run[3]};
#pragma unroll
        for (int i = 4; i < R; i += 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q) c[q] = M::op::apply(c[q], run[i + q]);
        }
        return M::op::apply(M::op::apply(c[0], c[1]), M::op::apply(c[2], c[3]));
    } else {
        T a = run[0];
#pragma unroll
        for (int i = 1; i < R; ++i) a = M::op::apply(a, run[i]);
        return a;
    }
}

// Inclusive scan of a row in place, starting from the exclusive prefix
// `mine` (absent only for the very first row of a line without init).
// Exclusive: element i takes the fold before it, the first one `mine`
// itself (always present: an exclusive scan starts from init).
template <class M, class T, int R>
__device__ __forceinline__ void row_scan_from(T (&run)[R], const typename M::P& mine, bool excl) {
    if (excl) {
        T a = M::value(mine);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const T x = run[i];
            run[i] = a;
            a = M::op::apply(a, x);
        }
        return;
    }
    T a = M::present(mine) ? M::op::apply(M::value(mine), run[0]) : run[0];
    run[0] = a;
#pragma unroll
    for (int i = 1; i < R; ++i) {
        a = M::op::apply(a, run[i]);
        run[i] = a;
    }
}

// Named barrier over `n` threads; returns whether `v` held in any of them.
__device__ __forceinline__ bool group_any(bool v, int id, int n) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void group_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Bounded wait for a ring barrier's phase; false when the wait limit passes
// or another block gave up.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, const ScanCtl& ctl) {
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > (uint64_t)ctl.wait_limit_ns) return false;
        if ((i & 63) == 63 && aborted(ctl)) return false;
    }
}

__device__ __forceinline__ void give_up(const ScanCtl& ctl) {
    atomicExch(reinterpret_cast<unsigned long long*>(ctl.error_word), (unsigned long long)ctl.epoch);
}

// Long contiguous lines, element type = accumulator type = output type,
// viewed as rows of 128 bytes (R elements); a tile is 256 rows (32 KB). One
// persistent block per SM runs a ring of STAGES tiles through four warp
// roles, handing each stage on with transaction barriers in shared memory:
//
//  producer (warp 0, one thread): claims tile indices from the call's
//    counter in order (one claim in flight ahead of its use) and, once the
//    scan warps have released a stage, has the next tile copied into it by
//    one bulk tensor load, swizzled so that every thread reads its own row
//    without bank conflicts;
//  fold warps (8): thread r folds row r, the row totals are scanned across
//    the group, each row's exclusive in-tile prefix goes to shared memory and
//    the tile's aggregate is published at once (the fold never waits on
//    another block);
//  look-back warps (kWsLookWarps, taking the stages in turn): compute each
//    tile's exclusive prefix from the previous tile of this block -- that
//    tile's inclusive prefix, then the aggregates of the tiles claimed in
//    between by other blocks (about one per block, read in one batch of
//    vector loads and folded in order). The warps fold their batches in
//    parallel and hand the running inclusive prefix on in tile order through
//    shared memory. Only aggregates are ever waited for, and those are
//    published as soon as a tile lands, so no prefix has to travel from
//    block to block and look-backs do not chain;
//  scan warps (8): thread r reads row r again, scans it from the tile's
//    exclusive prefix combined with the row's in-tile prefix and stores it
//    straight to global memory, then the stage goes back to the producer.
//
// HBM traffic is one read and one write of every element; the operator is
// applied twice per element (fold and scan), as in any single-pass scan
// whose tiles cannot wait for their prefix before starting. Rows past a
// line's end are zero-filled by the copy and ignored; the partial row of a
// single ragged line is read and written directly by its thread. Every wait
// is bounded and watches the call's error word; a role that gives up
// records the call's epoch there, and the producer lets its copies land
// before it leaves.
template <class T, class M>
__global__ void __launch_bounds__(kWsThreads, 1)
    k_scan_tma(const __grid_constant__ CUtensorMap tin, const T* __restrict__ x, T* __restrict__ y, int64_t len,
               int64_t rows_full, int64_t tiles_per_line, int64_t ntiles, TileState<typename M::P> ts, ScanCtl ctl,
               bool has_init, T init, bool excl) {
    using P = typename M::P;
    constexpr int S = ws_stages<P>();
    constexpr int R = 128 / (int)sizeof(T);
    constexpr int ROWS = kWsRows;
    constexpr uint32_t TILE_BYTES = ROWS * 128;
    constexpr int NW = rec_words<P>();
    constexpr int Q = kWsLookQ;
    extern __shared__ unsigned char dyn_smem[];
    unsigned char* const bufs =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    constexpr bool FX = ws_fx<T, M>();
    constexpr int RPB = ws_rowpre_bytes<T, M>();
    unsigned char* const rowpre = bufs + (size_t)S * TILE_BYTES;  // [S][ROWS] slots of RPB bytes
    auto rowpre_at = [&](int s, int r) { return rowpre + ((size_t)s * ROWS + r) * RPB; };
    __shared__ __align__(8) uint64_t full[S], folded[S], ready[S], empty[S];
    __shared__ int64_t s_k[S];
    __shared__ int64_t s_kprev[S];  // the block's tile before s_k[s] (-1: none)
    __shared__ int64_t s_t[S];      // position of s_k[s] in its line
    __shared__ int64_t s_base[S];   // element offset of the tile's first row
    __shared__ P s_agg[S];
    __shared__ P s_pre[S];
    __shared__ P fwt[ROWS / 32];
    // f64 sums: warp totals and flags of the fold, double-buffered by tile
    // parity (no warp gets a whole tile ahead of another), and whether the
    // tile took the FP64 path
    __shared__ Fx fwt_fx[2][ROWS / 32];
    __shared__ int s_wsp[2][ROWS / 32];
    __shared__ int s_special[S];
    // hand-off between the look-back warps, in tile order: after ring slot
    // s_chain - 1, the inclusive prefix of that slot's tile is s_incl;
    // s_end is the slot of the end-of-claims sentinel once it is known
    __shared__ P s_incl;
    __shared__ volatile int s_chain;
    __shared__ volatile int s_end;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const int64_t rem = len - rows_full * R;  // elements of the partial last row (a single line only)

    // valid elements of row r of the tile in stage s, and the row's element
    // offset (tile positions are worked out once, by the producer)
    auto row_count = [&](int s, int r) -> int {
        const int64_t row = s_t[s] * ROWS + r;
        return row < rows_full ? R : (row == rows_full ? (int)rem : 0);
    };
    auto row_off = [&](int s, int r) -> int64_t { return s_base[s] + (int64_t)r * R; };

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&folded[s], FX ? ROWS / 32 : 1);  // f64 sums: every fold warp arrives
            mbar_init(&ready[s], 1);
            mbar_init(&empty[s], ROWS / 32);
        }
        fence_barrier_init();
        s_chain = 0;
        s_end = 1 << 30;
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------- producer
        if (lane != 0) return;
        tma_prefetch_map(&tin);
        unsigned long long next = atomicAdd(ctl.counter, 1ull);
        int64_t kprev = -1;
        int j = 0;
        for (;; ++j) {
            const int s = j % S;
            if (j >= S && !ring_wait(&empty[s], (uint32_t)(j / S - 1) & 1u, ctl)) {
                give_up(ctl);
                break;
            }
            const int64_t k = (int64_t)next;
            s_k[s] = k;
            s_kprev[s] = kprev;
            kprev = k;
            if (k >= ntiles) {  // end of the claims: pass the sentinel down the ring
                mbar_arrive(&full[s]);
                ++j;
                break;
            }
            next = atomicAdd(ctl.counter, 1ull);
            int64_t t, line;
            tile_pos(k, tiles_per_line, ntiles, &t, &line);
            const int64_t row0 = t * ROWS;
            s_t[s] = t;
            s_base[s] = line * len + row0 * R;
            if (row0 < rows_full) {
                mbar_arrive_expect_tx(&full[s], TILE_BYTES);
                tma_load_3d(bufs + (size_t)s * TILE_BYTES, &tin, 0, (int)row0, (int)line, &full[s]);
            } else {
                mbar_arrive(&full[s]);  // only the partial row: nothing to copy
            }
        }
        // the block's shared memory must outlive every copy started into it
        const uint64_t until = globaltimer_ns() + (uint64_t)ctl.wait_limit_ns;
        for (int q = (j > S ? j - S : 0); q < j; ++q) mbar_wait(&full[q % S], (uint32_t)(q / S) & 1u, until);
        return;
    }

    if (warp <= kWsLookWarps) {
        // ---------------- look-back (this warp takes ring slots lw, lw + L, ...)
        const int lw = warp - 1;
        for (int j = lw;; j += kWsLookWarps) {
            const int s = j % S;
            bool ok = true;
            {
                const uint64_t t0 = globaltimer_ns();
                for (int i = 0;; ++i) {
                    if (mbar_try_wait(&folded[s], (uint32_t)(j / S) & 1u)) break;
                    if (s_end < j) return;  // the claims ended in an earlier slot
                    if (globaltimer_ns() - t0 > (uint64_t)ctl.wait_limit_ns || ((i & 63) == 63 && aborted(ctl))) {
                        ok = false;
                        break;
                    }
                }
            }
            if (__any_sync(kFull, !ok)) {
                if (lane == 0) give_up(ctl);
                return;
            }
            const int64_t k = s_k[s];
            if (k >= ntiles) {
                if (lane == 0) {
                    s_end = j;
                    mbar_arrive(&ready[s]);
                }
                return;
            }

            // Give the other blocks time to publish the tiles they claimed
            // just before this one: wait until the next kWsLookDefer stages
            // of this block are folded too (their copies were started after
            // this tile's, so by then the in-between tiles have landed
            // elsewhere as well). A stage past the end of the claims is
            // folded as a sentinel; the ring is deep enough that this never
            // waits on a stage that needs this look-back to make progress.
            for (int d = 1; d <= kWsLookDefer && ok; ++d) {
                const int jd = j + d, sd = jd % S;
                const uint64_t t0 = globaltimer_ns();
                for (int i = 0;; ++i) {
                    if (mbar_try_wait(&folded[sd], (uint32_t)(jd / S) & 1u)) break;
                    if (globaltimer_ns() - t0 > (uint64_t)ctl.wait_limit_ns || ((i & 63) == 63 && aborted(ctl))) {
                        ok = false;
                        break;
                    }
                }
                if (s_k[sd] >= ntiles) break;  // the sentinel: nothing after it
            }
            if (__any_sync(kFull, !ok)) {
                if (lane == 0) give_up(ctl);
                return;
            }
            const int64_t t = s_t[s], first = k - t, kp = s_kprev[s];
            const bool chained = t != 0 && kp >= first;  // prefix continues from the block's previous tile
            const int64_t lo = t == 0 ? k : (chained ? kp + 1 : first);
            // fold the aggregates of tiles lo .. k-1 in order
            P f = M::empty();
            bool good = true;
            for (int64_t base = lo; base < k; base += (int64_t)kWarp * Q) {
                const int64_t mine = base + (int64_t)lane * Q;  // this lane's Q consecutive tiles
                uint64_t w[Q][NW];
#pragma unroll
                for (int q = 0; q < Q; ++q)
                    if (mine + q < k) rec_load(ts.recs + mine + q, w[q]);
                P vals[Q];
                unsigned pend = 0;  // records of this lane not published yet
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    vals[q] = M::empty();
                    if (mine + q < k && rec_decode<P>(w[q], ctl.epoch, &vals[q]) == 0) pend |= 1u << q;
                }
                const uint64_t t0 = globaltimer_ns();
                while (pend != 0) {  // read every pending record again, all at once
                    if (globaltimer_ns() - t0 > (uint64_t)ctl.wait_limit_ns || aborted(ctl)) {
                        good = false;
                        break;
                    }
                    __nanosleep(100);
#pragma unroll
                    for (int q = 0; q < Q; ++q)
                        if (pend & (1u << q)) rec_load(ts.recs + mine + q, w[q]);
#pragma unroll
                    for (int q = 0; q < Q; ++q)
                        if ((pend & (1u << q)) && rec_decode<P>(w[q], ctl.epoch, &vals[q]) != 0) pend &= ~(1u << q);
                }
                if (__any_sync(kFull, !good)) {
                    good = false;
                    break;
                }
                P v = M::empty();
#pragma unroll
                for (int q = 0; q < Q; ++q)
                    if (mine + q < k) v = M::combine(v, vals[q]);
                v = warp_reduce<M>(v);  // lane 0 holds the ordered fold of the batch
                f = M::combine(f, shfl_idx_any(v, 0));
            }
            if (!good) {
                if (lane == 0) give_up(ctl);
                return;
            }
            // wait for this slot's turn in the hand-off
            {
                const uint64_t t0 = globaltimer_ns();
                for (int i = 0; s_chain != j; ++i) {
                    __nanosleep(64);  // leave the issue slots to the other roles
                    if (globaltimer_ns() - t0 > (uint64_t)ctl.wait_limit_ns || ((i & 63) == 63 && aborted(ctl))) {
                        ok = false;
                        break;
                    }
                }
            }
            if (__any_sync(kFull, !ok)) {
                if (lane == 0) give_up(ctl);
                return;
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                const P start = chained ? s_incl : (has_init ? M::lift(init) : M::empty());
                const P excl = M::combine(start, f);
                s_pre[s] = excl;
                s_incl = M::combine(excl, s_agg[s]);
                __threadfence_block();
                s_chain = j + 1;
                mbar_arrive(&ready[s]);
            }
            __syncwarp();
        }
    }

    if (warp < kWsScanWarp0) {
        // ---------------- fold
        const int r = tid - kWsFoldWarp0 * kWarp, fw = r / kWarp;
        for (int j = 0;; ++j) {
            const int s = j % S;
            const bool ok = ring_wait(&full[s], (uint32_t)(j / S) & 1u, ctl);
            if (group_any(!ok, 1, ROWS)) {
                if (r == 0) give_up(ctl);
                return;
            }
            const int64_t k = s_k[s];
            if (k >= ntiles) {
                if (FX ? lane == 0 : r == 0) mbar_arrive(&folded[s]);
                return;
            }
            const int nt = row_count(s, r);
            T run[R];
            if (nt == R) row_load(run, bufs + (size_t)s * TILE_BYTES, r);
            P tot = M::empty();
            if (nt != R && nt > 0) {
                const T* src = x + row_off(s, r);
                for (int i = 0; i < nt; ++i) tot = M::combine(tot, M::lift(src[i]));
            }
            if constexpr (FX) {
                // Row totals in wide fixed point; their warp scans go ahead,
                // and the flags written beside the warp totals decide after
                // the one barrier whether the tile takes the FP64 path
                // instead (a row with an infinity or a NaN, or with only
                // zeros and subnormals).
                const int pb = j & 1;
                int fm = 1;
                Fx rt = fx_zero();
                if (nt == R) {
                    rt = row_total_fx(run, &fm);
                } else if (nt > 0) {
                    const uint64_t tb = (uint64_t)__double_as_longlong(tot);
                    fm = ((tb >> 52) & 0x7FFu) == 0x7FFu ? 0x7FF : 1;
                    if (fm == 1) rt = fx_of(tot);
                }
                const bool sp = fm == 0 || fm == 0x7FF;
                rt = fx_norm(rt, 54);
                Fx inc = rt;
#pragma unroll
                for (int d = 1; d < kWarp; d <<= 1) {
                    const Fx o = fx_shfl_up(inc, d);
                    if (lane >= d) inc = fx_add(o, inc);
                }
                Fx lane_excl = fx_shfl_up(inc, 1);
                if (lane == 0) lane_excl = fx_zero();
                const bool wsp = __any_sync(kFull, sp);
                if (lane == kWarp - 1) {
                    fwt_fx[pb][fw] = inc;
                    s_wsp[pb][fw] = wsp;
                }
                group_sync(1, ROWS);
                bool tsp = false;
#pragma unroll
                for (int w = 0; w < ROWS / 32; ++w) tsp |= s_wsp[pb][w] != 0;
                if (!tsp) {
                    // the warp totals scanned across lanes 0..7
                    Fx wv = lane < ROWS / 32 ? fwt_fx[pb][lane] : fx_zero();
#pragma unroll
                    for (int d = 1; d < ROWS / 32; d <<= 1) {
                        const Fx o = fx_shfl_up(wv, d);
                        if (lane >= d) wv = fx_add(o, wv);
                    }
                    const Fx base = fx_shfl_idx(wv, fw == 0 ? 0 : fw - 1);
                    const Fx agg = fx_shfl_idx(wv, ROWS / 32 - 1);
                    *reinterpret_cast<Fx*>(rowpre_at(s, r)) = fw == 0 ? lane_excl : fx_add(base, lane_excl);  // |a| < 2^62
                    if (r == 0) {
                        // published at once: other blocks' look-backs wait for it
                        const P aggd = fx_to_double(agg);
                        s_agg[s] = aggd;
                        s_special[s] = 0;
                        if (s_t[s] != tiles_per_line - 1 && k != ctl.skip_tile)
                            publish(ts, k, kStatusAggregate, aggd, ctl.epoch);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&folded[s]);
                    continue;
                }
                if (r == 0) s_special[s] = 1;
            }
            if (nt == R) tot = M::lift(row_fold<M>(run));
            const P inc = warp_inclusive_scan<M>(tot, lane);
            P lane_excl = shfl_up_any(inc, 1);
            if (lane == 0) lane_excl = M::empty();
            if (lane == kWarp - 1) fwt[fw] = inc;
            group_sync(1, ROWS);
            // every warp folds the warp totals before its own (at most 7
            // combines), the first thread all of them: no second hand-off
            P base = M::empty();
#pragma unroll
            for (int w = 0; w < ROWS / 32; ++w)
                if (w < fw) base = M::combine(base, fwt[w]);
            if (r == 0) {
                P agg = base;
#pragma unroll
                for (int w = 0; w < ROWS / 32; ++w) agg = M::combine(agg, fwt[w]);
                s_agg[s] = agg;
                if (s_t[s] != tiles_per_line - 1 && k != ctl.skip_tile) publish(ts, k, kStatusAggregate, agg, ctl.epoch);
            }
            *reinterpret_cast<P*>(rowpre_at(s, r)) = M::combine(base, lane_excl);
            group_sync(1, ROWS);  // every row prefix written; fwt free again
            if (FX ? lane == 0 : r == 0) mbar_arrive(&folded[s]);
        }
    }

    {
        // ---------------- scan
        const int r = tid - kWsScanWarp0 * kWarp;
        const uint64_t last_use = l2_policy_evict_first();
        for (int j = 0;; ++j) {
            const int s = j % S;
            const bool ok = ring_wait(&ready[s], (uint32_t)(j / S) & 1u, ctl);
            if (__any_sync(kFull, !ok)) {
                if (lane == 0) give_up(ctl);
                return;
            }
            const int64_t k = s_k[s];
            if (k >= ntiles) return;
            const int nt = row_count(s, r);
            P rp;
            if constexpr (FX) {
                const Fx rpx = *reinterpret_cast<const Fx*>(rowpre_at(s, r));
                // (row 0: nothing before it in the tile, the identity -0)
                rp = s_special[s] ? *reinterpret_cast<const P*>(rowpre_at(s, r))
                                  : (r == 0 ? M::empty() : fx_to_double(rpx));
            } else {
                rp = *reinterpret_cast<const P*>(rowpre_at(s, r));
            }
            const P from = M::combine(s_pre[s], rp);
            if (nt == R) {
                T run[R];
                row_load(run, bufs + (size_t)s * TILE_BYTES, r);
                row_scan_from<M>(run, from, excl);
                row_store_global(y + row_off(s, r), run, last_use);
            } else if (nt > 0) {
                const T* src = x + row_off(s, r);
                T* dst = y + row_off(s, r);
                P a = from;
                for (int i = 0; i < nt; ++i) {
                    const P before = a;
                    a = M::combine(a, M::lift(src[i]));
                    dst[i] = M::value(excl ? before : a);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
}

// Lines that fit one tile: block b scans line b with the init prefix; no
// state is shared between blocks.
template <class In, class Acc, class Out, class M, int ITEMS, int BLOCK>
__global__ void __launch_bounds__(BLOCK, min_blocks_per_sm<BLOCK, (int)sizeof(Acc)>())
    k_scan_lines(const In* __restrict__ x, Out* __restrict__ y, int64_t len, bool has_init, Acc init, bool excl,
                 uint64_t* error_word) {
    using P = typename M::P;
    using L = RunLayout<Acc, ITEMS>;
    constexpr int W = BLOCK / kWarp;
    __shared__ __align__(16) char tile[BLOCK * L::stride * 16];
    __shared__ P warp_tot[W];
    __shared__ P s_prefix;
    const int64_t start = (int64_t)blockIdx.x * len;
    const int cnt = (int)len;
    if (threadIdx.x == 0) s_prefix = has_init ? M::lift(init) : M::empty();
    if (blockIdx.x == 0 && threadIdx.x == 0) *error_word = 0;  // no waits here: the call's status is ok
    load_tile<In, Acc, ITEMS, BLOCK>(tile, x + start, cnt, l2_policy_evict_first());
    __syncthreads();
    scan_apply_store<Acc, Out, M, ITEMS, BLOCK>(tile, y + start, cnt, &s_prefix, warp_tot, l2_policy_evict_first(),
                                                excl);
}

// Lines along a strided dimension: y[i + I*(j + J*k)] over j, for every
// (i, k). One thread per column (i, k), walking j with rows prefetched.
template <class In, class Acc, class Out, class M>
__global__ void __launch_bounds__(256) k_scan_strided(const In* __restrict__ x, Out* __restrict__ y,
                                                      int64_t I, int64_t J, int64_t K, bool has_init,
                                                      Acc init, bool excl, uint64_t* error_word) {
    using P = typename M::P;
    const int64_t col = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (col == 0) *error_word = 0;  // no waits here: the call's status is ok
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
            const P before = acc;
            acc = M::combine(acc, M::lift(convert<Acc>(v[u])));
            dst[I * (j + u)] = convert<Out>(M::value(excl ? before : acc));
        }
    }
    for (; j < J; ++j) {
        const P before = acc;
        acc = M::combine(acc, M::lift(convert<Acc>(src[I * j])));
        dst[I * j] = convert<Out>(M::value(excl ? before : acc));
    }
}

// Lines along a strided dimension with too few columns to fill the GPU:
// the scanned dimension is cut into `chunks` chunks of CH rows. The fold
// (block (column tile, chunk)) folds each column's chunk into part[chunk][col];
// the apply, chained with programmatic dependent launch, starts each column's
// chunk from init and the totals of the chunks before it (in order) and
// scans the chunk again, now from L2, storing as it goes.
constexpr int64_t kStridedTarget = 1 << 18;  // columns x chunks to aim for (about the resident threads)
constexpr int64_t kStridedMaxChunks = 1024;
constexpr int64_t kStridedMinRows = 16;       // rows per chunk at least

template <class In, class M>
__global__ void __launch_bounds__(256) k_scan_strided_fold(const In* __restrict__ x, int64_t I, int64_t J,
                                                           int64_t K, int64_t CH, typename M::P* __restrict__ part,
                                                           uint64_t* error_word) {
    using P = typename M::P;
    using Acc = typename M::acc;
    const int64_t cols = I * K;
    const int64_t col = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t ch = blockIdx.y;
    if (col == 0 && ch == 0) *error_word = 0;  // no waits here: the call's status is ok
    if (col < cols) {
        const int64_t i = col % I, k = col / I;
        const In* src = x + i + I * J * k;
        const int64_t j0 = ch * CH, j1 = min(J, j0 + CH);
        P a = M::empty();
        constexpr int U = 4;
        int64_t j = j0;
        for (; j + U <= j1; j += U) {
            In v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) v[u] = src[I * (j + u)];
#pragma unroll
            for (int u = 0; u < U; ++u) a = M::combine(a, M::lift(convert<Acc>(v[u])));
        }
        for (; j < j1; ++j) a = M::combine(a, M::lift(convert<Acc>(src[I * j])));
        part[ch * cols + col] = a;
    }
    griddep_launch_dependents();
}

template <class In, class Acc, class Out, class M>
__global__ void __launch_bounds__(256) k_scan_strided_apply(const In* __restrict__ x, Out* __restrict__ y, int64_t I,
                                                            int64_t J, int64_t K, int64_t CH,
                                                            const typename M::P* __restrict__ part, bool has_init,
                                                            Acc init, bool excl) {
    using P = typename M::P;
    griddep_wait();
    const int64_t cols = I * K;
    const int64_t col = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t ch = blockIdx.y;
    if (col >= cols) return;
    P acc = has_init ? M::lift(init) : M::empty();
#pragma unroll 8
    for (int64_t q = 0; q < ch; ++q) acc = M::combine(acc, part[q * cols + col]);
    const int64_t i = col % I, k = col / I;
    const In* src = x + i + I * J * k;
    Out* dst = y + i + I * J * k;
    const int64_t j0 = ch * CH, j1 = min(J, j0 + CH);
    constexpr int U = 4;
    int64_t j = j0;
    for (; j + U <= j1; j += U) {
        In v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = src[I * (j + u)];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const P before = acc;
            acc = M::combine(acc, M::lift(convert<Acc>(v[u])));
            dst[I * (j + u)] = convert<Out>(M::value(excl ? before : acc));
        }
    }
    for (; j < j1; ++j) {
        const P before = acc;
        acc = M::combine(acc, M::lift(convert<Acc>(src[I * j])));
        dst[I * j] = convert<Out>(M::value(excl ? before : acc));
    }
}

// cuTensorMapEncodeTiled from the driver the runtime is using (no link-time
// dependency on libcuda); null when the driver does not provide it.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// Lines of `rows` 128-byte rows (32 words), `lines` of them `line_bytes`
// apart, copied in boxes of box_rows rows with the 128-byte swizzle.
inline bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const void* base, int64_t rows,
                 int64_t lines, uint64_t line_bytes, int box_rows) {
    const cuuint64_t dims[3] = {32, (cuuint64_t)rows, (cuuint64_t)lines};
    const cuuint64_t strides[2] = {128, (cuuint64_t)line_bytes};
    const cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per device: the kernel's shared-memory opt-in done and its resident
// blocks per SM (0 = not yet known).
template <class T, class M>
int tma_blocks_per_sm(int device) {
    static std::atomic<int> cache[64];
    auto kernel = k_scan_tma<T, M>;
    constexpr int smem = ws_smem_bytes<T, M>();
    if (device >= 0 && device < 64) {
        const int v = cache[device].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kWsThreads, smem) != cudaSuccess) return -1;
    if (occ < 1) return 0;
    if (device >= 0 && device < 64) cache[device].store(occ, std::memory_order_relaxed);
    return occ;
}

// The TMA tile scan; AK_ERR_UNSUPPORTED (nothing launched) when the
// pointers are not 16-byte aligned or the driver has no tensor-map encoder.
template <class T, class M>
ak_status launch_tma(const ScanCall& c, const ScanPlan& p) {
    constexpr int64_t R = 128 / (int64_t)sizeof(T);
    if (reinterpret_cast<uintptr_t>(c.src) % 16 != 0 || reinterpret_cast<uintptr_t>(c.dst) % 16 != 0)
        return AK_ERR_UNSUPPORTED;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return AK_ERR_UNSUPPORTED;
    const int64_t rows_full = c.len / R;
    const uint64_t line_bytes = c.outer > 1 ? (uint64_t)c.len * sizeof(T) : (uint64_t)rows_full * 128;
    alignas(64) CUtensorMap tin;
    if (!encode_rows(enc, &tin, c.src, rows_full, c.outer, line_bytes, kWsRows)) return AK_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    const int occ = tma_blocks_per_sm<T, M>(dev.device);
    if (occ < 0) return cuda_fail(cudaGetLastError());
    if (occ == 0) return AK_ERR_UNSUPPORTED;
    int64_t grid = std::min<int64_t>(p.tma_tiles, (int64_t)occ * dev.sm_count);
    if (c.target_blocks > 0) grid = std::min<int64_t>(grid, c.target_blocks);
    char* ws = static_cast<char*>(c.ws);
    TileState<typename M::P> ts;
    ts.recs = reinterpret_cast<TileRec<typename M::P>*>(ws + p.state_off);
    ScanCtl ctl;
    ctl.epoch = c.epoch;
    ctl.error_word = reinterpret_cast<uint64_t*>(ws);  // WsHeader::error_word
    ctl.counter = reinterpret_cast<unsigned long long*>(ws + 64);
    ctl.wait_limit_ns = c.wait_limit_ns;
    ctl.skip_tile = c.skip_tile;
    T init;
    memcpy(&init, c.init.b, sizeof(T));
    // fresh counter, error word and records (correct under CUDA graph replay)
    cudaError_t e = cudaMemsetAsync(ws, 0, p.tma_ws_bytes, c.stream);
    if (e != cudaSuccess) return cuda_fail(e);
    k_scan_tma<T, M><<<(unsigned)grid, kWsThreads, ws_smem_bytes<T, M>(), c.stream>>>(
        tin, static_cast<const T*>(c.src), static_cast<T*>(c.dst), c.len, rows_full, p.tma_tiles_per_line,
        p.tma_tiles, ts, ctl, c.has_init, init, c.exclusive);
    ak_status s = check_launch();
    if (s == AK_OK) count_launches(1);
    return s;
}

template <class In, class Acc, class Out, class M>
ak_status launch(const ScanCall& c, const ScanPlan& p) {
    using P = typename M::P;
    Acc init;
    memcpy(&init, c.init.b, sizeof(Acc));
    if (p.kind == 1) {
        const int64_t cols = c.inner * c.outer;
        const unsigned blocks = (unsigned)((cols + 255) / 256);
        if (p.chunks <= 1) {
            k_scan_strided<In, Acc, Out, M><<<blocks, 256, 0, c.stream>>>(
                static_cast<const In*>(c.src), static_cast<Out*>(c.dst), c.inner, c.len, c.outer, c.has_init, init,
                c.exclusive, static_cast<uint64_t*>(c.ws));
            ak_status s = check_launch();
            if (s == AK_OK) count_launches(1);
            return s;
        }
        P* part = reinterpret_cast<P*>(static_cast<char*>(c.ws) + p.seg_off);
        const dim3 grid(blocks, (unsigned)p.chunks);
        k_scan_strided_fold<In, M><<<grid, 256, 0, c.stream>>>(static_cast<const In*>(c.src), c.inner, c.len,
                                                               c.outer, p.chunk_rows, part,
                                                               static_cast<uint64_t*>(c.ws));
        ak_status s = check_launch();
        if (s != AK_OK) return s;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.stream = c.stream;
        cfg.gridDim = grid;
        cfg.blockDim = dim3(256);
        const cudaError_t e = cudaLaunchKernelEx(&cfg, k_scan_strided_apply<In, Acc, Out, M>,
                                                 static_cast<const In*>(c.src), static_cast<Out*>(c.dst), c.inner,
                                                 c.len, c.outer, p.chunk_rows, (const P*)part, c.has_init, init,
                                                 c.exclusive);
        if (e != cudaSuccess) return cuda_fail(e);
        count_launches(2);
        return AK_OK;
    }
    constexpr int ITEMS = default_items<Acc>();
    constexpr int BLOCK = default_block<Acc>();
    constexpr int SEG = default_seg<Acc>();
    if constexpr (!(ITEMS % (sizeof(In) < 16 ? 16 / sizeof(In) : 1) == 0 &&
                    ITEMS % (sizeof(Out) < 16 ? 16 / sizeof(Out) : 1) == 0)) {
        return AK_ERR_UNSUPPORTED;
    } else {
        if (p.block != BLOCK || p.items != ITEMS) return AK_ERR_UNSUPPORTED;
        if constexpr (std::is_same_v<In, Acc> && std::is_same_v<Acc, Out> && std::is_same_v<typename M::P, Acc> &&
                      (std::is_same_v<Acc, float> || std::is_same_v<Acc, int32_t> || std::is_same_v<Acc, int64_t> ||
                       (std::is_same_v<Acc, double> && std::is_same_v<typename M::op, OpAdd>))) {
            if (p.kind == 0 && p.tma) {
                const ak_status st = launch_tma<Acc, M>(c, p);
                if (st != AK_ERR_UNSUPPORTED) return st;
            }
        }
        char* ws = static_cast<char*>(c.ws);
        TileState<P> ts;
        ts.recs = reinterpret_cast<TileRec<P>*>(ws + p.state_off);
        ScanCtl ctl;
        ctl.epoch = c.epoch;
        ctl.error_word = reinterpret_cast<uint64_t*>(ws);  // WsHeader::error_word
        ctl.counter = reinterpret_cast<unsigned long long*>(ws + 64);
        ctl.wait_limit_ns = c.wait_limit_ns;
        ctl.skip_tile = c.skip_tile;
        if (p.kind == 2) {
            // the smallest block whose tile holds a whole line
            auto lines = [&](auto blk) {
                constexpr int B = decltype(blk)::value;
                k_scan_lines<In, Acc, Out, M, ITEMS, B><<<(unsigned)p.tiles, B, 0, c.stream>>>(
                    static_cast<const In*>(c.src), static_cast<Out*>(c.dst), c.len, c.has_init, init, c.exclusive,
                    reinterpret_cast<uint64_t*>(ws));
            };
            if (c.len <= 64 * ITEMS) lines(std::integral_constant<int, 64>{});
            else if (c.len <= 128 * ITEMS || BLOCK == 128) lines(std::integral_constant<int, 128>{});
            else lines(std::integral_constant<int, BLOCK>{});
        } else if (p.three) {
            // reduce-then-scan: fold, tile prefixes, apply (PDL-chained)
            P* seg = reinterpret_cast<P*>(ws + p.seg_off);
            P* agg = reinterpret_cast<P*>(ws + p.agg_off);
            P* pre = reinterpret_cast<P*>(ws + p.pre_off);
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            cfg.stream = c.stream;
            const In* xs = static_cast<const In*>(c.src);
            Out* ys = static_cast<Out*>(c.dst);
            uint64_t* err = reinterpret_cast<uint64_t*>(ws);
            k_scan3_fold<In, M, BLOCK, SEG><<<(unsigned)p.tiles, BLOCK, 0, c.stream>>>(xs, c.len, seg, agg, err);
            ak_status s = check_launch();
            if (s != AK_OK) return s;
            // few tiles: the apply blocks fold the aggregates before them
            // themselves; many: one block scans them first
            const bool fused = p.tiles <= kFusedPrefixTiles;
            if (!fused) {
                cfg.gridDim = dim3(1);
                cfg.blockDim = dim3(kTilesBlock);
                const cudaError_t e =
                    cudaLaunchKernelEx(&cfg, k_scan3_tiles<M>, (const P*)agg, pre, p.tiles, c.has_init, init);
                if (e != cudaSuccess) return cuda_fail(e);
            }
            cfg.gridDim = dim3((unsigned)p.tiles);
            cfg.blockDim = dim3(BLOCK);
            const cudaError_t e = cudaLaunchKernelEx(
                &cfg, k_scan3_apply<In, Acc, Out, M, BLOCK, SEG>, xs, ys, c.len, (const P*)seg,
                fused ? (const P*)nullptr : (const P*)pre, (const P*)agg, c.has_init, init, c.exclusive);
            if (e != cudaSuccess) return cuda_fail(e);
            count_launches(fused ? 2 : 3);
            return AK_OK;
        } else {
            DeviceInfo dev;
            if (!current_device(&dev)) return AK_ERR_CUDA;
            int occ = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &occ, k_scan_tiles<In, Acc, Out, M, BLOCK, SEG>, BLOCK, 0);
            if (e != cudaSuccess) return cuda_fail(e);
            int64_t grid = std::min<int64_t>(p.tiles, (int64_t)std::max(occ, 1) * dev.sm_count);
            if (c.target_blocks > 0) grid = std::min<int64_t>(grid, c.target_blocks);
            // Fresh claim counter, error word and tile records for this call. The
            // records also carry the call's epoch; zeroing them makes a call
            // captured in a CUDA graph (whose epoch is fixed at capture) correct
            // on every replay.
            e = cudaMemsetAsync(ws, 0, p.ws_bytes, c.stream);
            if (e != cudaSuccess) return cuda_fail(e);
            k_scan_tiles<In, Acc, Out, M, BLOCK, SEG><<<(unsigned)grid, BLOCK, 0, c.stream>>>(
                static_cast<const In*>(c.src), static_cast<Out*>(c.dst), c.len, p.tiles_per_line, p.tiles, ts, ctl,
                c.has_init, init, c.exclusive);
        }
        ak_status s = check_launch();
        if (s == AK_OK) count_launches(1);
        return s;
    }
}

// The scan plan from the accumulator and partial sizes: kernel kind, run
// length and block, tile counts and workspace. tma_type: the element type
// may take the TMA tile scan (one 4- or 8-byte type throughout: f32 / i32 /
// i64 with a neutral element, and f64 sums, whose folds run in fixed point;
// the matrix product spends more operator work per byte and Optional
// partials more per combine, and those run faster on kernels whose blocks
// carry more warps per SM); it then also needs rows of 128 bytes, several
// tiles per line, and lines that start on a row boundary unless there is
// only one.
// Single lines not on the TMA scan take the reduce-then-scan in three
// launches at any length: on GB300 it beat the single-pass super-tile scan
// at every size measured, even where the second read misses L2 (1e8 f64:
// 418 against 444 us; 1e8 f32 max under Optional partials: 231 against 332
// us; 1e7 mod-p products: level), because no block ever waits on another.
constexpr uint64_t kThreePassMaxBytes = ~0ull;

inline ak_status plan_sizes(int64_t inner, int64_t len, int64_t outer, size_t asz, size_t psz, bool tma_type,
                            int items, ScanPlan* p, size_t in_bytes = 0, bool single_pass = false) {
    p->three = false;
    p->seg_off = p->agg_off = p->pre_off = 0;
    p->state_off = kWsHeader;
    p->ws_bytes = kWsHeader;
    p->tiles = 0;
    p->tiles_per_line = 0;
    p->grid = 0;
    p->tma = false;
    p->tma_tiles_per_line = 0;
    p->tma_tiles = 0;
    p->tma_ws_bytes = 0;
    p->chunks = 1;
    p->chunk_rows = len;
    if (inner > 1) {
        p->kind = 1;
        p->block = 256;
        p->items = 1;
        // few columns: cut the scanned dimension into chunks (fold, then apply)
        const int64_t cols = inner * outer;
        const int64_t chunks = cols < 1 ? 1
                                        : std::min<int64_t>((kStridedTarget + cols - 1) / cols,
                                                            std::min<int64_t>(kStridedMaxChunks, len / kStridedMinRows));
        if (chunks > 1) {
            p->chunk_rows = (len + chunks - 1) / chunks;
            p->chunks = (len + p->chunk_rows - 1) / p->chunk_rows;
            p->seg_off = kWsHeader;
            p->ws_bytes = std::max(p->ws_bytes, align_up(kWsHeader + (size_t)p->chunks * (size_t)cols * psz, 256));
        }
        return AK_OK;
    }
    p->kind = 0;
    const int it = asz >= 16 ? 8 : (asz == 8 ? 16 : 32);
    if (items != 0 && items != it) return AK_ERR_UNSUPPORTED;
    p->items = it;
    const int block = asz >= 16 ? 128 : 256;
    const int seg = asz >= 16 ? 64 : (asz == 8 ? 64 : 32);
    p->block = block;
    const int64_t tile = (int64_t)block * it;
    if (len <= tile) {
        p->kind = 2;  // every line fits one tile: no state shared between blocks
        p->tiles_per_line = 1;
        p->tiles = outer;
        return AK_OK;
    }
    const int64_t super = (int64_t)block * seg;
    p->tiles_per_line = (len + super - 1) / super;
    p->tiles = p->tiles_per_line * outer;
    p->ws_bytes = align_up(kWsHeader + (size_t)p->tiles * (16 + align_up(psz, 16)), 256);  // TileRec per super-tile
    const int64_t rl = 128 / (int64_t)asz;
    if (items == 0 && tma_type && (asz == 4 || asz == 8) && len > kWsRows * rl && (outer == 1 || len % rl == 0) &&
        len / rl < ((int64_t)1 << 31) && outer < ((int64_t)1 << 31)) {
        const int64_t rows = (len + rl - 1) / rl;
        p->tma = true;
        p->tma_tiles_per_line = (rows + kWsRows - 1) / kWsRows;
        p->tma_tiles = p->tma_tiles_per_line * outer;
        p->tma_ws_bytes = align_up(kWsHeader + (size_t)p->tma_tiles * (16 + align_up(psz, 16)), 256);
        p->ws_bytes = std::max(p->ws_bytes, p->tma_ws_bytes);
    }
    // one line outside the TMA scan: reduce-then-scan in three launches
    // (in_bytes = 0: unknown, not taken; single_pass: the caller wants the
    // single-pass kernel, e.g. to exercise its bounded waits)
    const uint64_t in_total = (uint64_t)in_bytes * (uint64_t)len;
    if (!p->tma && outer == 1 && in_bytes != 0 && !single_pass && in_total <= kThreePassMaxBytes) {
        p->three = true;
        p->seg_off = kWsHeader;
        p->agg_off = align_up(p->seg_off + (size_t)p->tiles * block * psz, 256);
        p->pre_off = align_up(p->agg_off + (size_t)p->tiles * psz, 256);
        p->ws_bytes = std::max(p->ws_bytes, align_up(p->pre_off + (size_t)p->tiles * psz, 256));
    }
    return AK_OK;
}

// Runs a scan whose input type is In: dispatches the accumulator / output
// types, operator and monoid. Each scan_*.cu instantiates it for one input
// type, so the scan kernels compile in parallel translation units.
template <class In>
ak_status run_for_input(const ScanCall& c, const ScanPlan& plan) {
    return dispatch_types(c.in, c.acc, c.out, [&](auto ti, auto ta, auto to) -> ak_status {
        using In2 = typename decltype(ti)::type;
        using Acc = typename decltype(ta)::type;
        using Out = typename decltype(to)::type;
        if constexpr (!std::is_same_v<In, In2> || std::is_same_v<In2, bf16> || std::is_same_v<Out, bf16>) {
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

}  // namespace scan
}  // namespace ak
