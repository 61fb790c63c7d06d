// findall.cu -- stream compaction on GB300: the indices of the nonzero
// elements of an array (Julia's findall over a Bool array, or over x .!= 0),
// written in increasing order, and their count.
//
// findall is a scan in disguise: the output position of a selected element
// is the exclusive prefix count of the selected elements before it
// (AcceleratedKernels.jl tile-scan PR #202 counts findall's byte tiles among
// its scans: ratio table, and the paragraph on its tests). One pass over the
// input, on the tile machinery of the long-line scans (scan.cuh):
//
//   persistent blocks of 256 threads claim tiles of 256 x E elements (E = 64
//   bytes, 32 four-byte or 16 eight-byte elements a thread; 16 K / 8 K / 4 K
//   elements a tile). Phase A of tile k: every thread reads its E
//   consecutive elements with 32-byte loads, turns them into an E-bit mask
//   (kept in shared memory) and a count; the block sums the counts and
//   publishes the tile's aggregate (a line's first tile publishes its
//   inclusive prefix). Phase B of the tile claimed one round earlier: look
//   back to the tile's exclusive count (decoupled look-back over the
//   published records, bounded waits), publish its inclusive count, scan the
//   thread counts, expand every thread's mask into tile-relative positions in
//   shared memory, and store the tile's indices with consecutive threads on
//   consecutive output slots (every warp store covers 256 contiguous bytes).
//
// The input is read once and never re-read (phase B works from the masks);
// the output is written once: HBM traffic is n * sizeof(T) + 8 * count bytes.
#include <algorithm>

#include "scan.cuh"

namespace ak {
namespace fa {

using scan::ScanCtl;
using scan::TileRec;
using scan::TileState;

constexpr int kBlock = 256;
using Count = Plain<OpAdd, int64_t>;  // the monoid of the tile counts

// Elements per thread: 64 bytes of flags, 128 bytes of wider elements.
template <class T>
constexpr int elems_per_thread() {
    return sizeof(T) == 1 ? 64 : 128 / (int)sizeof(T);
}
template <class T>
constexpr int tile_elems() {
    return kBlock * elems_per_thread<T>();
}

// Nonzero test of one element: bytes and integers against 0, floats against
// 0.0 (so -0.0 is zero and NaN is not).
template <class T>
__device__ __forceinline__ bool nonzero(T v) {
    if constexpr (std::is_same_v<T, float>) return (__float_as_uint(v) & 0x7FFFFFFFu) != 0u;
    else if constexpr (std::is_same_v<T, double>) return ((uint64_t)__double_as_longlong(v) & 0x7FFFFFFFFFFFFFFFull) != 0ull;
    else return v != 0;
}

// Mask bits of the 32 bytes of one load: bit b set when byte b is nonzero.
__device__ __forceinline__ uint32_t byte_mask32(const Raw<32>& r) {
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        // 0xFF in every nonzero byte lane; pick bit b of byte b, gather to 4 bits
        const uint32_t t = __vcmpne4(r.w[w], 0u) & 0x08040201u;
        m |= ((t | (t >> 8) | (t >> 16) | (t >> 24)) & 0xFu) << (4 * w);
    }
    return m;
}

// Mask bits of one 32-byte load of 4- or 8-byte elements.
template <class T>
__device__ __forceinline__ uint32_t elem_mask32(const Raw<32>& r) {
    constexpr int K = 32 / (int)sizeof(T);
    uint32_t m = 0;
#pragma unroll
    for (int q = 0; q < K; ++q) m |= (uint32_t)nonzero(raw_get<T>(r, q)) << q;
    return m;
}

// The E-bit mask of a thread's elements [e0, e0 + E) (bits past n are 0).
template <class T>
__device__ __forceinline__ uint64_t thread_mask(const T* x, int64_t n, int64_t e0, uint64_t policy) {
    constexpr int E = elems_per_thread<T>();
    constexpr int PER = 32 / (int)sizeof(T);  // elements per 32-byte load
    constexpr int L = E / PER;                // loads per thread
    const T* p = x + e0;
    uint64_t m = 0;
    if (e0 + E <= n && reinterpret_cast<uintptr_t>(p) % 32 == 0) {
        Raw<32> r[L];
#pragma unroll
        for (int u = 0; u < L; ++u) r[u] = ld_hint32(p + u * PER, policy);
#pragma unroll
        for (int u = 0; u < L; ++u) {
            uint64_t part;
            if constexpr (sizeof(T) == 1) part = byte_mask32(r[u]);
            else part = elem_mask32<T>(r[u]);
            m |= part << (u * PER);
        }
    } else {
        const int cnt = (int)max((int64_t)0, min((int64_t)E, n - e0));
        for (int i = 0; i < cnt; ++i) m |= (uint64_t)nonzero(p[i]) << i;
    }
    return m;
}

template <class T>
__global__ void __launch_bounds__(kBlock, 3)
    k_findall(const T* __restrict__ x, int64_t n, int64_t ntiles, int64_t* __restrict__ idx, int64_t* count,
              TileState<int64_t> ts, ScanCtl ctl) {
    constexpr int E = elems_per_thread<T>();
    constexpr int TILE = tile_elems<T>();
    constexpr int W = kBlock / kWarp;
    __shared__ uint64_t s_mask[2][kBlock];  // the masks of the two open tiles
    __shared__ int s_cnt[2][kBlock];
    __shared__ uint16_t s_pos[TILE];        // tile-relative positions, in order
    __shared__ int64_t red[W];
    __shared__ int ints[2 * kWarp + 1];
    __shared__ int s_wsum[W];
    __shared__ int64_t s_k;
    __shared__ int64_t s_bc;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const uint64_t once = l2_policy_evict_first();

    int64_t prev = -1, prev_agg = 0;
    int slot = 0;
    while (true) {
        if (tid == 0) s_k = (int64_t)atomicAdd(ctl.counter, 1ull);
        __syncthreads();
        const int64_t k = s_k;
        int64_t agg = 0;
        if (k < ntiles) {
            // ---- phase A of tile k: masks, counts, the tile's aggregate
            const uint64_t m = thread_mask<T>(x, n, k * TILE + (int64_t)tid * E, once);
            s_mask[slot][tid] = m;
            const int c = __popcll(m);
            s_cnt[slot][tid] = c;
            agg = scan::block_reduce_ordered<Count, kBlock>((int64_t)c, red);
            if (tid == 0) {  // thread 0 holds the block total
                if (k != ctl.skip_tile) scan::publish(ts, k, k == 0 ? scan::kStatusPrefix : scan::kStatusAggregate,
                                                      agg, ctl.epoch);
                s_bc = agg;
            }
            __syncthreads();
            agg = s_bc;
        }
        if (prev >= 0) {
            // ---- phase B of tile prev: its exclusive count, then the indices
            const int pslot = slot ^ 1;
            int64_t base = 0;
            if (prev != 0) {
                if (!scan::look_back<Count, kBlock>(prev, 0, ts, ctl, red, ints, &base)) {
                    if (tid == 0) scan::give_up(ctl);
                    return;  // uniform: every thread got the same answer
                }
                if (tid == 0) {
                    if (prev != ctl.skip_tile) scan::publish(ts, prev, scan::kStatusPrefix, base + prev_agg, ctl.epoch);
                    s_bc = base;
                }
                __syncthreads();
                base = s_bc;
            }
            // exclusive scan of the thread counts
            const int c = s_cnt[pslot][tid];
            int inc = c;
#pragma unroll
            for (int d = 1; d < kWarp; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, inc, d);
                if (lane >= d) inc += o;
            }
            if (lane == kWarp - 1) s_wsum[warp] = inc;
            __syncthreads();
            int woff = 0;
#pragma unroll
            for (int w = 0; w < W; ++w) woff += w < warp ? s_wsum[w] : 0;
            int off = woff + inc - c;
            uint64_t m = s_mask[pslot][tid];
            while (m) {
                const int b = __ffsll((long long)m) - 1;
                s_pos[off++] = (uint16_t)(tid * E + b);
                m &= m - 1;
            }
            __syncthreads();
            const int total = (int)prev_agg;
            int64_t* out = idx + base;
            const int64_t first = prev * TILE;
            for (int j = tid; j < total; j += kBlock) out[j] = first + s_pos[j];
            if (prev == ntiles - 1 && tid == 0) *count = base + prev_agg;
            __syncthreads();  // s_pos, s_wsum and the slot are reused next
        }
        if (k >= ntiles) break;
        prev = k;
        prev_agg = agg;
        slot ^= 1;
    }
}

template <class T>
ak_status launch(const void* src, int64_t n, int64_t* idx, int64_t* count, void* ws, int64_t ntiles,
                 size_t ws_bytes, uint64_t epoch, int64_t wait_limit_ns, int64_t skip_tile, int target_blocks,
                 cudaStream_t stream) {
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_findall<T>, kBlock, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    int64_t grid = std::min<int64_t>(ntiles, (int64_t)std::max(occ, 1) * dev.sm_count);
    if (target_blocks > 0) grid = std::min<int64_t>(grid, target_blocks);
    char* w = static_cast<char*>(ws);
    TileState<int64_t> ts;
    ts.recs = reinterpret_cast<TileRec<int64_t>*>(w + kWsHeader);
    ScanCtl ctl;
    ctl.epoch = epoch;
    ctl.error_word = reinterpret_cast<uint64_t*>(w);
    ctl.counter = reinterpret_cast<unsigned long long*>(w + 64);
    ctl.wait_limit_ns = wait_limit_ns;
    ctl.skip_tile = skip_tile;
    // fresh claim counter, error word and tile records (correct under graph replay)
    e = cudaMemsetAsync(ws, 0, ws_bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    k_findall<T><<<(unsigned)grid, kBlock, 0, stream>>>(static_cast<const T*>(src), n, ntiles, idx, count, ts, ctl);
    ak_status s = check_launch();
    if (s == AK_OK) count_launches(1);
    return s;
}

}  // namespace fa

// Tiles and workspace of a findall: header, one 32-byte record per tile,
// then the count slot used when the caller gives no device count.
ak_status plan_findall(int64_t n, ak_dtype in, int64_t* ntiles, size_t* ws_bytes, size_t* count_off) {
    int64_t tile = 0;
    switch (in) {
    case AK_U8: tile = fa::tile_elems<uint8_t>(); break;
    case AK_I32: case AK_F32: tile = fa::tile_elems<float>(); break;
    case AK_I64: case AK_F64: tile = fa::tile_elems<double>(); break;
    default: return AK_ERR_UNSUPPORTED;
    }
    *ntiles = (std::max<int64_t>(n, 1) + tile - 1) / tile;
    *count_off = align_up(kWsHeader + (size_t)*ntiles * sizeof(scan::TileRec<int64_t>), 64);
    *ws_bytes = align_up(*count_off + 8, 256);
    return AK_OK;
}

ak_status run_findall(const void* src, int64_t n, ak_dtype in, int64_t* idx, int64_t* count, void* ws,
                      int64_t ntiles, size_t ws_bytes, uint64_t epoch, int64_t wait_limit_ns, int64_t skip_tile,
                      int target_blocks, cudaStream_t stream) {
    switch (in) {
    case AK_U8:
        return fa::launch<uint8_t>(src, n, idx, count, ws, ntiles, ws_bytes, epoch, wait_limit_ns, skip_tile,
                                   target_blocks, stream);
    case AK_I32:
        return fa::launch<int32_t>(src, n, idx, count, ws, ntiles, ws_bytes, epoch, wait_limit_ns, skip_tile,
                                   target_blocks, stream);
    case AK_F32:
        return fa::launch<float>(src, n, idx, count, ws, ntiles, ws_bytes, epoch, wait_limit_ns, skip_tile,
                                 target_blocks, stream);
    case AK_I64:
        return fa::launch<int64_t>(src, n, idx, count, ws, ntiles, ws_bytes, epoch, wait_limit_ns, skip_tile,
                                   target_blocks, stream);
    case AK_F64:
        return fa::launch<double>(src, n, idx, count, ws, ntiles, ws_bytes, epoch, wait_limit_ns, skip_tile,
                                  target_blocks, stream);
    default: return AK_ERR_UNSUPPORTED;
    }
}

}  // namespace ak
