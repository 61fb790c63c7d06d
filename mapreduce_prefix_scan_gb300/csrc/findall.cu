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
//   consecutive elements with 32-byte loads and turns them into an E-bit
//   mask and a count, kept in registers; a warp scan and one barrier give
//   every thread its offset in the tile and the tile's aggregate, which is
//   published at once (the first tile publishes its inclusive prefix).
//   Phase B of the tile claimed one round earlier: look back to the tile's
//   exclusive count (decoupled look-back over the published records,
//   bounded waits), publish its inclusive count, expand every thread's mask
//   into tile-relative positions in shared memory, and store the tile's
//   indices with consecutive threads on consecutive pairs of output slots
//   (16-byte stores: every warp store covers 512 contiguous bytes).
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
// Per word: the top bit of every nonzero byte (the low seven bits plus 0x7F
// carry into it without crossing bytes, or the byte's own top bit is set),
// then one multiply gathers the four top bits into bits 28..31 (the partial
// products land on distinct bits, so nothing carries).
__device__ __forceinline__ uint32_t byte_mask32(const Raw<32>& r) {
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t v = r.w[w];
        const uint32_t top = (((v & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | v) & 0x80808080u;
        m |= (((top >> 7) * 0x10204080u) >> 28) << (4 * w);
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
    __shared__ uint16_t s_pos[TILE];  // tile-relative positions, in order
    __shared__ int64_t red[W];
    __shared__ int ints[2 * kWarp + 1];
    __shared__ int s_wsum[W];
    __shared__ int64_t s_k;
    __shared__ int64_t s_bc;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const uint64_t once = l2_policy_evict_first();

    // the tile claimed one round earlier: its count, and this thread's mask
    // and offset in it
    int64_t prev = -1, prev_agg = 0;
    uint64_t prev_mask = 0;
    int prev_off = 0;
    while (true) {
        if (tid == 0) s_k = (int64_t)atomicAdd(ctl.counter, 1ull);
        __syncthreads();  // s_k; the last round's reads of s_pos and s_wsum are done
        const int64_t k = s_k;
        uint64_t m = 0;
        int off = 0;
        if (k < ntiles) {
            // ---- phase A of tile k: mask, offset, the tile's aggregate
            m = thread_mask<T>(x, n, k * TILE + (int64_t)tid * E, once);
            const int c = __popcll(m);
            int inc = c;
#pragma unroll
            for (int d = 1; d < kWarp; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, inc, d);
                if (lane >= d) inc += o;
            }
            if (lane == kWarp - 1) s_wsum[warp] = inc;
            off = inc - c;
        }
        __syncthreads();  // the warp totals
        int64_t agg = 0;
        if (k < ntiles) {
            int tot = 0;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const int v = s_wsum[w];
                off += w < warp ? v : 0;
                tot += v;
            }
            agg = tot;
            if (tid == 0 && k != ctl.skip_tile)
                scan::publish(ts, k, k == 0 ? scan::kStatusPrefix : scan::kStatusAggregate, agg, ctl.epoch);
        }
        if (prev >= 0) {
            // ---- phase B of tile prev: its exclusive count, then the indices
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
            }
            // the set bits of this thread's mask, as positions in the tile
            {
                int o = prev_off;
                const int p0 = tid * E;
                uint32_t lo = (uint32_t)prev_mask;
                while (lo) {
                    s_pos[o++] = (uint16_t)(p0 + __ffs((int)lo) - 1);
                    lo &= lo - 1;
                }
                if constexpr (E > 32) {
                    uint32_t hi = (uint32_t)(prev_mask >> 32);
                    while (hi) {
                        s_pos[o++] = (uint16_t)(p0 + 31 + __ffs((int)hi));
                        hi &= hi - 1;
                    }
                }
            }
            __syncthreads();  // positions written; s_bc
            if (prev != 0) base = s_bc;
            const int total = (int)prev_agg;
            int64_t* out = idx + base;
            const int64_t first = prev * TILE;
            // pairs of slots on 16-byte boundaries; a leading or trailing
            // single slot takes an 8-byte store
            const int lead = (int)((reinterpret_cast<uintptr_t>(out) >> 3) & 1u) < total
                                 ? (int)((reinterpret_cast<uintptr_t>(out) >> 3) & 1u)
                                 : total;
            const int pairs = (total - lead) / 2;
            if (tid == 0 && lead) out[0] = first + s_pos[0];
            for (int q = tid; q < pairs; q += kBlock) {
                const int j = lead + 2 * q;
                longlong2 v;
                v.x = first + s_pos[j];
                v.y = first + s_pos[j + 1];
                *reinterpret_cast<longlong2*>(out + j) = v;
            }
            if (tid == kBlock - 1 && lead + 2 * pairs < total) out[total - 1] = first + s_pos[total - 1];
            if (prev == ntiles - 1 && tid == 0) *count = base + prev_agg;
        }
        if (k >= ntiles) break;
        prev = k;
        prev_agg = agg;
        prev_mask = m;
        prev_off = off;
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
