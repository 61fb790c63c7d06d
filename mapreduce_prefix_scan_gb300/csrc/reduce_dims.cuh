// reduce_dims.cuh -- kernels of the reductions over a set of dimensions of a
// column-major array (dense, or a strided view) on GB300.
//
// After merging dimensions (api.cu), most problems take one of two canonical
// forms (ldj, ldk: source strides in elements; a dense array has ldj = I,
// ldk = I*J):
//   strided  out[i + I*k] = fold_j x[i + ldj*j + ldk*k]   (I > 1: outputs are
//            contiguous in the source, the reduction walks rows: sum(x;
//            dims=2) of a matrix, the middle dimension of a 3-d array)
//   rows     out[k]       = fold_j x[j + ldk*k]           (contiguous reduction)
// anything else (a kept dimension without unit stride, several reduced
// blocks that do not merge) goes to a general kernel.
//
// Strided kernel (strided-reduction PR #176, "This PR" item 1 and the
// paragraph after it: a fixed 2-d block of outputs by reduction rows, split
// across blocks only when the outputs alone cannot fill the device; item 2:
// a 3-d reduction over the middle dimension becomes one run of contiguous
// outputs per outer index k, handled by the same kernel). A block owns a
// tile of `tile_out` consecutive outputs of one run k and a range of
// reduction rows. Its threads form `row_groups` groups of `tpr` threads; a
// group covers the tile's row segment with 16-byte vector loads and walks a
// contiguous sub-range of rows with all of its rows' loads in flight. Groups
// are combined in row order (a few threads per output and an ordered shuffle
// tree), so non-commutative operators keep their order. The reduction is
// split across blocks when the outputs alone do not fill the device: the
// blocks of one output tile either form a thread-block cluster and push
// their partials into the owning block's shared memory (small inputs: one
// launch, one cluster barrier), or write per-split partials that a second
// pass (programmatic dependent launch) folds in split order.
//
// The three shapes of the pages are parameter regimes of this one kernel:
// "thread" = one group (each thread owns vec outputs and walks all rows),
// "tiled" = several groups, no split, "columns" = several groups and a split.
#pragma once
#include <algorithm>
#include <atomic>
#include <cooperative_groups.h>

#include "ak_common.cuh"
#include "ak_internal.h"

namespace ak {
namespace dims {

constexpr int kBlock = 256;
constexpr int kUnroll = 8;          // rows in flight per thread (at most)
constexpr int kMaxClusterSplit = 16;  // blocks of an output tile combined in one cluster
constexpr int kMinRowsPerGroup = 8; // the selector splits no further than this many rows per group

template <class Acc, class Out, class M>
struct DimsStore {
    int mode;
    Acc init;
    Out* dst;
};

template <class Acc, class Out, class M>
__device__ __forceinline__ void dims_store(const typename M::P& r, const DimsStore<Acc, Out, M>& st,
                                           int64_t o) {
    using Op = typename M::op;
    Acc v = M::value(r);
    if (st.mode == AK_STORE_INIT) v = Op::apply(st.init, v);
    else if (st.mode == AK_STORE_FOLD) v = Op::apply(convert<Acc>(st.dst[o]), v);
    st.dst[o] = convert<Out>(v);
}

template <class In, class Acc, class Map, class M>
__device__ __forceinline__ typename M::P lift_elem(In x) {
    return M::lift(Map::apply(convert<Acc>(x)));
}

// One row segment of VB bytes, kept as raw words until its elements are
// used (8 bf16 stay in 4 registers): a 16-byte streaming vector load, or a
// single element.
template <class In, int VB>
struct RowSeg {
    static constexpr bool kVec = VB == 16 && sizeof(In) < 16;
    Raw<kVec ? 16 : (sizeof(In) < 4 ? 4 : (int)sizeof(In))> raw;
    __device__ __forceinline__ void load(const In* p) {
        if constexpr (kVec) raw = ld_stream16(p);
        else memcpy(&raw, p, sizeof(In));
    }
    __device__ __forceinline__ In get(int q) const { return raw_get<In>(raw, q); }
};

// VB = bytes per load: 16 (vector of 16/sizeof(In) outputs) or sizeof(In).
// CLUSTER: the `split` blocks of one output tile form a thread-block
// cluster (split = cluster size); each keeps its partial outputs in shared
// memory and, after a cluster barrier, rank r folds the partials of its
// share of the outputs from every rank's shared memory (distributed shared
// memory), in rank (= row) order, and stores them: no workspace, no second
// pass. Otherwise blockIdx.y is the split index and split > 1 writes
// partials for k_dims_finish.
template <class In, class Acc, class Out, class Map, class M, int VB, bool CLUSTER>
__global__ void __launch_bounds__(kBlock, 4) k_dims_strided(const In* __restrict__ x, int64_t I, int64_t J,
                                                         int64_t K, int64_t ldj, int64_t ldk, int tile_out, int tpr,
                                                         int R,
                                                         int split, typename M::P* __restrict__ partials,
                                                         DimsStore<Acc, Out, M> st) {
    using P = typename M::P;
    constexpr int V = VB / (int)sizeof(In);
    // row-group partials, row groups tile_out + 1 apart (an odd pitch: the
    // stores of a warp's row groups and the fold's reads spread over banks)
    __shared__ P smem[kBlock * V + kBlock];
    const int pitch = tile_out + 1;

    const int64_t tiles_i = div_fast(I + tile_out - 1, tile_out);
    const int64_t tile_id = CLUSTER ? blockIdx.x / split : blockIdx.x;
    const int64_t k = div_fast(tile_id, tiles_i), ct = tile_id - k * tiles_i;
    const int s = CLUSTER ? (int)(blockIdx.x % split) : (int)blockIdx.y;
    const int tid = threadIdx.x, c = tid % tpr, rg = tid / tpr;
    const int64_t i0 = ct * tile_out + (int64_t)c * V;

    const int64_t jper = div_fast(J + split - 1, split);
    const int64_t js = (int64_t)s * jper, je = min(J, js + jper);
    const int64_t rper = div_fast(max(je - js, (int64_t)0) + R - 1, R);
    const int64_t jr = min(je, js + rg * rper), jre = min(je, jr + rper);

    P acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = M::empty();

    if (rg < R && i0 < I) {
        const In* base = x + i0 + ldk * k;
        if (i0 + V <= I) {
            // ROWS rows per round, all loads issued before any is used; a
            // short last round is predicated, not walked row by row
            constexpr int ROWS = kUnroll;
            const In* p = base + ldj * jr;     // walks the rows by pointer
            int left = (int)(jre - jr);        // rows of this group (< 2^31)
            for (; left >= ROWS; left -= ROWS, p += ldj * ROWS) {
                RowSeg<In, VB> r[ROWS];
#pragma unroll
                for (int u = 0; u < ROWS; ++u) r[u].load(p + ldj * u);
#pragma unroll
                for (int u = 0; u < ROWS; ++u)
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        acc[q] = M::combine(acc[q], lift_elem<In, Acc, Map, M>(r[u].get(q)));
            }
            if (left > 0) {
                RowSeg<In, VB> r[ROWS];
#pragma unroll
                for (int u = 0; u < ROWS; ++u)
                    if (u < left) r[u].load(p + ldj * u);
#pragma unroll
                for (int u = 0; u < ROWS; ++u)
                    if (u < left)
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            acc[q] = M::combine(acc[q], lift_elem<In, Acc, Map, M>(r[u].get(q)));
            }
        } else {
            // ragged last vector of the row: scalar loads of the valid columns
            for (int64_t j = jr; j < jre; ++j)
#pragma unroll
                for (int q = 0; q < V; ++q)
                    if (i0 + q < I) acc[q] = M::combine(acc[q], lift_elem<In, Acc, Map, M>(base[ldj * j + q]));
        }
    }
    griddep_launch_dependents();

    // smem[rg][c*V + q]; group rows are contiguous ranges, combined in order
    if (rg < R) {
#pragma unroll
        for (int q = 0; q < V; ++q) smem[rg * pitch + c * V + q] = acc[q];
    }
    __syncthreads();
    if (kBlock % tile_out != 0) {
        // wide tiles (one row group; a tile of more than kBlock outputs or of
        // a width that does not divide the block): a thread per output
        for (int o = tid; o < tile_out; o += kBlock) {
            const int64_t i = ct * tile_out + o;
            if (i >= I) continue;
            P a = smem[o];
            for (int g = 1; g < R; ++g) a = M::combine(a, smem[g * pitch + o]);
            if (split == 1) dims_store<Acc, Out, M>(a, st, i + I * k);
            else if constexpr (!CLUSTER) partials[((int64_t)s * K + k) * I + i] = a;
        }
        return;
    }
    // The R row groups of output e are folded by G consecutive threads (each
    // folds `per_t` consecutive groups, then an ordered shuffle tree within
    // the G lanes): a short dependency chain instead of R serial combines.
    // tile_out divides kBlock here, so G = kBlock / tile_out = R / V is a
    // power of two (capped at a warp and at the number of row groups).
    const int G0 = kBlock / tile_out;
    const int G = min(min(G0, kWarp), R);  // powers of two; the thread shape has R = 1
    const int per_t = R / G;
    const int e = tid / G, h = tid % G;
    P a = M::empty();
    if (e < tile_out) {
        a = smem[(h * per_t) * pitch + e];
        for (int g = 1; g < per_t; ++g) a = M::combine(a, smem[(h * per_t + g) * pitch + e]);
    }
    for (int d = 1; d < G; d <<= 1) {
        const P o = shfl_down_width(a, d, G);
        if (h + d < G) a = M::combine(a, o);
    }
    // lane h == 0 of each group now holds output e's partial of this block
    if constexpr (CLUSTER) {
        // push: the owner rank of output e folds it; every block stores its
        // partial straight into the owner's inbox (distributed shared
        // memory), then one cluster barrier (release / acquire) makes the
        // stores visible. Nothing reads another block's shared memory after
        // the barrier, so blocks may leave as soon as they are done.
        namespace cg = cooperative_groups;
        cg::cluster_group cluster = cg::this_cluster();
        __shared__ P inbox[kBlock + kMaxClusterSplit];
        const int per = (tile_out + split - 1) / split;
        if (h == 0 && e < tile_out) {
            P* box = cluster.map_shared_rank(inbox, e / per);
            box[s * per + e % per] = a;
        }
        cluster.sync();
        const int eo = s * per + tid;
        if (tid < per && eo < tile_out && ct * tile_out + eo < I) {
            P r = inbox[tid];
#pragma unroll 4
            for (int q = 1; q < split; ++q) r = M::combine(r, inbox[q * per + tid]);
            dims_store<Acc, Out, M>(r, st, ct * tile_out + eo + I * k);
        }
    } else {
        const int64_t i = ct * tile_out + e;
        if (h == 0 && e < tile_out && i < I) {
            if (split == 1) dims_store<Acc, Out, M>(a, st, i + I * k);
            else partials[((int64_t)s * K + k) * I + i] = a;
        }
    }
}

// Contiguous reduction: one warp per (output k, split s) segment.
template <class In, class Acc, class Out, class Map, class M>
__global__ void __launch_bounds__(kBlock) k_dims_rows(const In* __restrict__ x, int64_t J, int64_t K, int64_t ldk,
                                                      int split, typename M::P* __restrict__ partials,
                                                      DimsStore<Acc, Out, M> st) {
    using P = typename M::P;
    constexpr int kRun = 8;
    const int lane = threadIdx.x % kWarp;
    const int64_t gw = (int64_t)blockIdx.x * (kBlock / kWarp) + threadIdx.x / kWarp;
    if (gw >= K * split) return;
    const int64_t k = div_fast(gw, split);
    const int s = (int)(gw - k * split);
    const int64_t jper = div_fast(J + split - 1, split);
    const int64_t js = (int64_t)s * jper, je = min(J, js + jper);
    const In* row = x + ldk * k;
    P a = M::empty();
    if constexpr (M::commutative && sizeof(In) < 16 && 16 % sizeof(In) == 0) {
        // 16-byte vector loads, U per lane at a time: an element-wise
        // head up to the first 16-byte boundary, the vectors, an element-wise tail
        constexpr int V = 16 / (int)sizeof(In);
        constexpr int U = 4;
        const In* seg = row + js;
        const int64_t len = je - js;
        const int64_t head = min(len, (int64_t)(((16 - reinterpret_cast<uintptr_t>(seg) % 16) % 16) / sizeof(In)));
        const int64_t nvec = (len - head) / V;
        P acc[V];
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = M::empty();
        for (int64_t i = lane; i < head; i += kWarp) acc[0] = M::combine(acc[0], lift_elem<In, Acc, Map, M>(seg[i]));
        const In* body = seg + head;
        int64_t v = lane;
        for (; v + (U - 1) * kWarp < nvec; v += U * kWarp) {
            Raw<16> r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) r[u] = ld_stream16(body + (v + u * kWarp) * V);
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int q = 0; q < V; ++q)
                    acc[q] = M::combine(acc[q], lift_elem<In, Acc, Map, M>(raw_get<In>(r[u], q)));
        }
        for (; v < nvec; v += kWarp) {
            const Raw<16> r = ld_stream16(body + v * V);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = M::combine(acc[q], lift_elem<In, Acc, Map, M>(raw_get<In>(r, q)));
        }
        for (int64_t i = head + nvec * V + lane; i < len; i += kWarp)
            acc[V - 1] = M::combine(acc[V - 1], lift_elem<In, Acc, Map, M>(seg[i]));
        a = acc[0];
#pragma unroll
        for (int q = 1; q < V; ++q) a = M::combine(a, acc[q]);
        a = warp_reduce<M>(a);
    } else if constexpr (M::commutative) {
        int64_t j = js + lane;
        for (; j + 3 * kWarp < je; j += 4 * kWarp) {
            In v0 = row[j], v1 = row[j + kWarp], v2 = row[j + 2 * kWarp], v3 = row[j + 3 * kWarp];
            a = M::combine(a, lift_elem<In, Acc, Map, M>(v0));
            a = M::combine(a, lift_elem<In, Acc, Map, M>(v1));
            a = M::combine(a, lift_elem<In, Acc, Map, M>(v2));
            a = M::combine(a, lift_elem<In, Acc, Map, M>(v3));
        }
        for (; j < je; j += kWarp) a = M::combine(a, lift_elem<In, Acc, Map, M>(row[j]));
        a = warp_reduce<M>(a);
    } else {
        for (int64_t c = js; c < je; c += kWarp * kRun) {
            P r = M::empty();
            const int64_t b = c + (int64_t)lane * kRun;
#pragma unroll
            for (int q = 0; q < kRun; ++q)
                if (b + q < je) r = M::combine(r, lift_elem<In, Acc, Map, M>(row[b + q]));
            r = warp_reduce<M>(r);
            a = M::combine(a, r);
        }
    }
    griddep_launch_dependents();
    if (lane == 0) {
        if (split == 1) dims_store<Acc, Out, M>(a, st, k);
        else partials[(int64_t)s * K + k] = a;
    }
}

// Second pass of a split: output o folds partials[s*nout + o], s = 0..split-1.
template <class Acc, class Out, class M>
__global__ void __launch_bounds__(kBlock) k_dims_finish(const typename M::P* partials, int64_t nout,
                                                        int split, DimsStore<Acc, Out, M> st) {
    griddep_wait();
    const int64_t o = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    if (o >= nout) return;
    typename M::P a = partials[o];
    int s = 1;
    for (; s + 8 <= split; s += 8) {  // 8 loads in flight, folded in split order
        typename M::P v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = partials[(int64_t)(s + u) * nout + o];
#pragma unroll
        for (int u = 0; u < 8; ++u) a = M::combine(a, v[u]);
    }
    for (; s < split; ++s) a = M::combine(a, partials[(int64_t)s * nout + o]);
    dims_store<Acc, Out, M>(a, st, o);
}

// General fallback for any dims mask and any strides: reduced indices
// visited in increasing column-major order. Many outputs: one thread per
// output (k_dims_general); few outputs: blocks of (output, split) pairs
// (k_dims_general_blocks).
struct GeneralIndex {
    int ndim;
    int64_t shape[8];
    int64_t stride[8];
    int nk, nr;
    int kept[8], red[8];
    int64_t nout, nfold;
};

template <class In, class Acc, class Out, class Map, class M>
__global__ void __launch_bounds__(kBlock) k_dims_general(const In* __restrict__ x, GeneralIndex g,
                                                         DimsStore<Acc, Out, M> st) {
    const int64_t o = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    if (o >= g.nout) return;
    int64_t base = 0, t = o;
    for (int a = 0; a < g.nk; ++a) {
        const int d = g.kept[a];
        base += (t % g.shape[d]) * g.stride[d];
        t /= g.shape[d];
    }
    typename M::P acc = M::empty();
    for (int64_t r = 0; r < g.nfold; ++r) {
        int64_t off = base, u = r;
        for (int a = 0; a < g.nr; ++a) {
            const int d = g.red[a];
            off += (u % g.shape[d]) * g.stride[d];
            u /= g.shape[d];
        }
        acc = M::combine(acc, lift_elem<In, Acc, Map, M>(x[off]));
    }
    dims_store<Acc, Out, M>(acc, st, o);
}

// Block (o, s) folds part s of output o's reduction: its threads take
// consecutive ranges of the reduced index (walked with an odometer over the
// reduced dimensions, one division per thread at the start), and the block
// combines them in thread order, so every operator keeps its order. With
// split > 1 partials[s * nout + o] go to k_dims_finish.
template <class In, class Acc, class Out, class Map, class M>
__global__ void __launch_bounds__(kBlock) k_dims_general_blocks(const In* __restrict__ x, GeneralIndex g, int split,
                                                                typename M::P* __restrict__ partials,
                                                                DimsStore<Acc, Out, M> st) {
    using P = typename M::P;
    __shared__ P smem[kBlock / kWarp];
    const int64_t o = blockIdx.x;
    const int s = (int)blockIdx.y;
    int64_t base = 0, t = o;
    for (int a = 0; a < g.nk; ++a) {
        const int d = g.kept[a];
        base += (t % g.shape[d]) * g.stride[d];
        t /= g.shape[d];
    }
    const int64_t per = (g.nfold + split - 1) / split;
    const int64_t rb = (int64_t)s * per, re = min(g.nfold, rb + per);
    const int64_t tper = (max(re - rb, (int64_t)0) + kBlock - 1) / kBlock;
    const int64_t r0 = rb + (int64_t)threadIdx.x * tper, r1 = min(re, r0 + tper);
    P acc = M::empty();
    if (r0 < r1) {
        int64_t idx[8];
        int64_t off = base, u = r0;
        for (int a = 0; a < g.nr; ++a) {
            const int d = g.red[a];
            idx[a] = u % g.shape[d];
            u /= g.shape[d];
            off += idx[a] * g.stride[d];
        }
        for (int64_t r = r0; r < r1; ++r) {
            acc = M::combine(acc, lift_elem<In, Acc, Map, M>(x[off]));
            // next reduced index: odometer over the reduced dimensions
            for (int a = 0; a < g.nr; ++a) {
                const int d = g.red[a];
                off += g.stride[d];
                if (++idx[a] < g.shape[d]) break;
                off -= g.shape[d] * g.stride[d];
                idx[a] = 0;
            }
        }
    }
    griddep_launch_dependents();
    acc = block_reduce<M, kBlock>(acc, smem);
    if (threadIdx.x == 0) {
        if (split == 1) dims_store<Acc, Out, M>(acc, st, o);
        else partials[(int64_t)s * g.nout + o] = acc;
    }
}

template <class Acc, class Out, class M, class... Args>
cudaError_t launch_finish(dim3 grid, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kBlock);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_dims_finish<Acc, Out, M>, args...);
}

// Whether clusters of `split` blocks of this kernel can be scheduled on the
// current device at all (an MPS or green-context SM limit may forbid them),
// cached per device and cluster size.
template <class K>
bool cluster_fits(K kernel, const cudaLaunchConfig_t& cfg, int split) {
    static std::atomic<signed char> cache[64][kMaxClusterSplit + 1];  // 0 unknown, 1 fits, -1 does not
    DeviceInfo dev;
    if (!current_device(&dev) || dev.device >= 64 || split > kMaxClusterSplit) return false;
    std::atomic<signed char>& slot = cache[dev.device][split];
    const signed char known = slot.load(std::memory_order_relaxed);
    if (known != 0) return known > 0;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    slot.store(n > 0 ? 1 : -1, std::memory_order_relaxed);
    return n > 0;
}

template <class In, class Acc, class Out, class Map, class M>
ak_status launch(const DimsCall& c, const DimsPlan& plan) {
    using P = typename M::P;
    DimsPlan p = plan;
    DimsStore<Acc, Out, M> st;
    st.mode = c.mode;
    memcpy(&st.init, c.init.b, sizeof(Acc));
    st.dst = static_cast<Out*>(c.dst);
    P* partials = reinterpret_cast<P*>(static_cast<char*>(c.ws) + kWsHeader);
    const In* x = static_cast<const In*>(c.src);
    if (c.general) {
        GeneralIndex g = {};
        g.ndim = c.ndim;
        g.nout = g.nfold = 1;
        for (int d = 0; d < c.ndim; ++d) {
            g.shape[d] = c.shape[d];
            g.stride[d] = c.stride[d];
            if ((c.mask >> d) & 1u) { g.red[g.nr++] = d; g.nfold *= c.shape[d]; }
            else { g.kept[g.nk++] = d; g.nout *= c.shape[d]; }
        }
        if (p.shape == AK_SHAPE_THREAD) {
            const int64_t blocks = (g.nout + kBlock - 1) / kBlock;
            k_dims_general<In, Acc, Out, Map, M><<<(unsigned)blocks, kBlock, 0, c.stream>>>(x, g, st);
        } else {
            k_dims_general_blocks<In, Acc, Out, Map, M><<<dim3((unsigned)g.nout, (unsigned)p.split), kBlock, 0,
                                                         c.stream>>>(x, g, p.split, partials, st);
        }
        ak_status s = check_launch();
        if (s != AK_OK) return s;
        count_launches(1);
        if (p.split > 1) {
            cudaError_t e = launch_finish<Acc, Out, M>(dim3((unsigned)((g.nout + kBlock - 1) / kBlock)), c.stream,
                                                       (const P*)partials, g.nout, p.split, st);
            if (e != cudaSuccess) return cuda_fail(e);
            count_launches(1);
        }
        return AK_OK;
    }
    const int64_t nout = c.inner * c.outer;
    if (c.inner == 1) {
        const int64_t warps = c.outer * p.split;
        const int64_t blocks = (warps + kBlock / kWarp - 1) / (kBlock / kWarp);
        k_dims_rows<In, Acc, Out, Map, M><<<(unsigned)blocks, kBlock, 0, c.stream>>>(x, c.red, c.outer, c.ldk,
                                                                                    p.split, partials, st);
    } else {
        const int64_t tiles_i = (c.inner + p.tile_out - 1) / p.tile_out;
        const int tpr = p.tile_out / p.vec;
        auto go = [&](auto vb) -> cudaError_t {
            constexpr int VB = decltype(vb)::value;
            if (p.cluster) {
                // the cluster combine needs tiles that divide the block and at
                // most kMaxClusterSplit blocks per tile (the selector's plans)
                if (kBlock % p.tile_out != 0 || p.split > kMaxClusterSplit) return cudaErrorInvalidConfiguration;
                auto kernel = k_dims_strided<In, Acc, Out, Map, M, VB, true>;
                if (p.split > 8) {
                    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (e != cudaSuccess) return e;
                }
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3((unsigned)(tiles_i * c.outer * p.split));
                cfg.blockDim = dim3(kBlock);
                cfg.stream = c.stream;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = (unsigned)p.split;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cluster_fits(kernel, cfg, p.split)) {
                    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, x, c.inner, c.red, c.outer, c.ldj, c.ldk,
                                                             p.tile_out, tpr, p.row_groups, p.split, partials, st);
                    if (e != cudaErrorInvalidClusterSize && e != cudaErrorLaunchOutOfResources) return e;
                    cudaGetLastError();
                }
                // no cluster of this size can run here: plan the same call
                // with the workspace split and a second pass instead
                DimsCall c2 = c;
                c2.allow_cluster = c2.auto_cluster = false;
                DeviceInfo dev;
                if (!current_device(&dev)) return cudaErrorNoDevice;
                if (plan_dims(c2, dev, &p) != AK_OK || p.cluster) return cudaErrorInvalidConfiguration;
                if (c.ws_bytes < p.ws_bytes) return cudaErrorMemoryAllocation;
                const int64_t tiles2 = (c.inner + p.tile_out - 1) / p.tile_out;
                dim3 grid((unsigned)(tiles2 * c.outer), (unsigned)p.split);
                k_dims_strided<In, Acc, Out, Map, M, VB, false><<<grid, kBlock, 0, c.stream>>>(
                    x, c.inner, c.red, c.outer, c.ldj, c.ldk, p.tile_out, p.tile_out / p.vec, p.row_groups, p.split,
                    partials, st);
                return cudaGetLastError();
            }
            dim3 grid((unsigned)(tiles_i * c.outer), (unsigned)p.split);
            k_dims_strided<In, Acc, Out, Map, M, VB, false><<<grid, kBlock, 0, c.stream>>>(
                x, c.inner, c.red, c.outer, c.ldj, c.ldk, p.tile_out, tpr, p.row_groups, p.split, partials, st);
            return cudaGetLastError();
        };
        cudaError_t e = cudaSuccess;
        if (p.vec > 1) {
            if constexpr (16 % sizeof(In) == 0 && sizeof(In) < 16) e = go(std::integral_constant<int, 16>{});
        } else {
            e = go(std::integral_constant<int, (int)sizeof(In)>{});
        }
        if (e == cudaErrorMemoryAllocation) return AK_ERR_WORKSPACE;  // the fallback plan needs a larger workspace
        if (e != cudaSuccess) return cuda_fail(e);
    }
    ak_status s = check_launch();
    if (s != AK_OK) return s;
    count_launches(1);
    if (p.split > 1 && !p.cluster) {
        dim3 grid((unsigned)((nout + kBlock - 1) / kBlock));
        cudaError_t e = launch_finish<Acc, Out, M>(grid, c.stream, (const P*)partials, nout, p.split, st);
        if (e != cudaSuccess) return cuda_fail(e);
        count_launches(1);
    }
    return AK_OK;
}

// Runs the reduction for one input type: dispatches the accumulator /
// output types, operator, map and monoid. Each dims_*.cu instantiates it for
// its input types, so the kernels compile in parallel translation units.
template <class In>
ak_status run_for_input(const DimsCall& c, const DimsPlan& plan) {
    return dispatch_types(c.in, c.acc, c.out, [&](auto ti, auto ta, auto to) -> ak_status {
        using In2 = typename decltype(ti)::type;
        using Acc = typename decltype(ta)::type;
        using Out = typename decltype(to)::type;
        if constexpr (!std::is_same_v<In, In2>) {
            return AK_ERR_UNSUPPORTED;
        } else {
            return dispatch_op<Acc>(c.op, [&](auto top) -> ak_status {
                using Op = typename decltype(top)::type;
                if (c.no_neutral) {
                    // Optional partials: identity map only
                    if (c.f != AK_MAP_IDENTITY) return AK_ERR_UNSUPPORTED;
                    return launch<In, Acc, Out, MapIdentity, Lifted<Op, Acc>>(c, plan);
                }
                return dispatch_map<Acc>(c.f, [&](auto tm) -> ak_status {
                    using Map = typename decltype(tm)::type;
                    return launch<In, Acc, Out, Map, Plain<Op, Acc>>(c, plan);
                });
            });
        }
    });
}

}  // namespace dims
}  // namespace ak
