// reduce.cuh -- kernels and launcher of the whole-array mapreduce on GB300
// (templates: compiled into libak for the built-in operators, and into a
// caller's translation unit by the C++ template API in include/ak.hpp).
//
// Design (AcceleratedKernels.jl PR #139, "Finish whole-array reductions on
// the device", section "What changes"): at most two launches. A first pass
// of a bounded grid in which every block reduces one contiguous share of the
// input to one partial result, and a one-block second pass that reduces the
// partials and performs the store (apply init, fold into R's previous value,
// overwrite, or leave the bare partial for a host-side finish). An input
// small enough for one block takes one launch.
//
// GB300 specifics: the first pass streams 32-byte vector loads
// (ld.global.nc.v8, no L1 allocation, 256-byte L2 prefetch) with several
// independent loads in flight per thread; the grid is a multiple of the SM
// count; the second pass is launched with programmatic dependent launch, so
// its launch overlaps the first pass's tail and it waits on the device
// (griddepcontrol.wait) instead of behind a full kernel boundary.
#pragma once
#include <algorithm>

#include "ak_common.cuh"
#include "ak_internal.h"

namespace ak {
namespace red {

constexpr int kBlock = 512;       // first pass, commutative operators
constexpr int kBlockOrd = 256;    // first pass, order-preserving
constexpr int kFinishBlock = 256;
constexpr int kVecBytes = 32;     // one 256-bit load per vector
constexpr int kUnroll = 4;        // independent vector loads in flight per thread
constexpr int kRunOrd = 8;        // consecutive elements folded per lane (ordered path)
constexpr int kMaxBlocksPerSm = 4;
constexpr int64_t kSingleLaunchMax = 16384;  // elements reduced by one block in one launch

// Where and how the final value goes.
template <class Acc, class Out, class M>
struct StoreSpec {
    int mode;          // ak_store
    Acc init;          // for AK_STORE_INIT
    Out* dst;          // final element (device), or null
    typename M::P* bare;  // bare partial for the host finish, or null
    // with `bare` in mapped host memory: a word the host polls, set to
    // `seq` once the partial is there (null: the host synchronizes instead)
    unsigned long long* flag;
    unsigned long long seq;
};

template <class Acc, class Out, class M>
__device__ __forceinline__ void store_result(const typename M::P& r, const StoreSpec<Acc, Out, M>& st) {
    using Op = typename M::op;
    if (st.bare) {
        *st.bare = r;
        if (st.flag) {
            __threadfence_system();  // the partial is visible to the host before the flag
            *reinterpret_cast<volatile unsigned long long*>(st.flag) = st.seq;
        }
        return;
    }
    Acc v = M::value(r);
    if (st.mode == AK_STORE_INIT) v = Op::apply(st.init, v);
    else if (st.mode == AK_STORE_FOLD) v = Op::apply(convert<Acc>(*st.dst), v);
    *st.dst = convert<Out>(v);
}

template <class In, class Acc, class Map, class M>
__device__ __forceinline__ typename M::P lift_elem(In x) {
    return M::lift(Map::apply(convert<Acc>(x)));
}

// First pass for commutative operators. Block b reduces the vectors
// [b*per, (b+1)*per) of the 32-byte-aligned body; block 0 adds the unaligned
// head and the last block the ragged tail. Thread t keeps one accumulator
// per vector lane and folds vectors t, t+BLOCK, ... with kUnroll loads in
// flight.
template <class In, class Acc, class Out, class Map, class M>
__global__ void __launch_bounds__(kBlock) k_reduce_pass1(const In* __restrict__ x, int64_t n,
                                                         int64_t head, int64_t nvec,
                                                         typename M::P* __restrict__ partials,
                                                         StoreSpec<Acc, Out, M> st) {
    using P = typename M::P;
    constexpr int V = kVecBytes / sizeof(In);
    __shared__ P smem[kBlock / kWarp];

    P acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = M::empty();

    const In* body = x + head;
    const int64_t per = (nvec + gridDim.x - 1) / gridDim.x;
    const int64_t vb = (int64_t)blockIdx.x * per;
    const int64_t ve = min(nvec, vb + per);
    int64_t v = vb + threadIdx.x;
    for (; v + (kUnroll - 1) * kBlock < ve; v += kUnroll * kBlock) {
        Raw<kVecBytes> r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) r[u] = ld_stream<kVecBytes>(body + (v + u * kBlock) * V);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int k = 0; k < V; ++k)
                acc[k] = M::combine(acc[k], lift_elem<In, Acc, Map, M>(raw_get<In>(r[u], k)));
    }
    for (; v < ve; v += kBlock) {
        Raw<kVecBytes> r = ld_stream<kVecBytes>(body + v * V);
#pragma unroll
        for (int k = 0; k < V; ++k)
            acc[k] = M::combine(acc[k], lift_elem<In, Acc, Map, M>(raw_get<In>(r, k)));
    }
    if (blockIdx.x == 0 && threadIdx.x < head)
        acc[0] = M::combine(acc[0], lift_elem<In, Acc, Map, M>(x[threadIdx.x]));
    const int64_t tail = head + nvec * V;
    if (blockIdx.x == gridDim.x - 1 && tail + threadIdx.x < n)
        acc[V - 1] = M::combine(acc[V - 1], lift_elem<In, Acc, Map, M>(x[tail + threadIdx.x]));

    griddep_launch_dependents();
    P a = acc[0];
#pragma unroll
    for (int k = 1; k < V; ++k) a = M::combine(a, acc[k]);
    a = block_reduce<M, kBlock>(a, smem);
    if (threadIdx.x == 0) {
        if (gridDim.x == 1) store_result<Acc, Out, M>(a, st);
        else partials[blockIdx.x] = a;
    }
}

// First pass that keeps the element order (non-commutative operators). Block
// b owns the contiguous range [b*per, (b+1)*per); each warp owns a
// contiguous sub-range of it and walks it in chunks of 32*kRunOrd elements:
// lane l folds its run of kRunOrd consecutive elements, the warp combines
// the 32 runs in lane order and appends the chunk to its running value.
// Warps are then combined in warp order.
template <class In, class Acc, class Out, class Map, class M>
__global__ void __launch_bounds__(kBlockOrd) k_reduce_pass1_ordered(const In* __restrict__ x,
                                                                    int64_t n,
                                                                    typename M::P* __restrict__ partials,
                                                                    StoreSpec<Acc, Out, M> st) {
    using P = typename M::P;
    constexpr int W = kBlockOrd / kWarp;
    __shared__ P smem[W];
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;

    const int64_t per = (n + gridDim.x - 1) / gridDim.x;
    const int64_t bb = (int64_t)blockIdx.x * per, be = min(n, bb + per);
    const int64_t wper = (be - bb + W - 1) / W;
    const int64_t wb = min(be, bb + warp * wper), we = min(be, wb + wper);

    P run_acc = M::empty();  // meaningful in lane 0
    for (int64_t c = wb; c < we; c += kWarp * kRunOrd) {
        P r = M::empty();
        const int64_t s = c + (int64_t)lane * kRunOrd;
#pragma unroll
        for (int k = 0; k < kRunOrd; ++k)
            if (s + k < we) r = M::combine(r, lift_elem<In, Acc, Map, M>(x[s + k]));
        r = warp_reduce<M>(r);
        run_acc = M::combine(run_acc, r);
    }
    griddep_launch_dependents();
    if (lane == 0) smem[warp] = run_acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        P a = smem[0];
        for (int w = 1; w < W; ++w) a = M::combine(a, smem[w]);
        if (gridDim.x == 1) store_result<Acc, Out, M>(a, st);
        else partials[blockIdx.x] = a;
    }
}

// First pass over a fused two-source element f(a_i, b_i) (commutative
// operators). VB = 32: both sources share their offset within 32 bytes, so
// the 32-byte vectors of a and b line up (block 0 adds the unaligned head, the
// last block the tail, as in k_reduce_pass1); VB = sizeof(In): element-wise
// loads, coalesced across the block, for sources of different alignments.
template <class In, class Acc, class Out, class Map2, class M, int VB>
__global__ void __launch_bounds__(kBlock) k_reduce2_pass1(const In* __restrict__ a, const In* __restrict__ b,
                                                          int64_t n, int64_t head, int64_t nvec,
                                                          typename M::P* __restrict__ partials,
                                                          StoreSpec<Acc, Out, M> st) {
    using P = typename M::P;
    constexpr int V = VB / (int)sizeof(In);
    __shared__ P smem[kBlock / kWarp];
    auto elem = [](In u, In v) { return M::lift(Map2::apply(convert<Acc>(u), convert<Acc>(v))); };

    P acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = M::empty();
    const In* ba = a + head;
    const In* bb = b + head;
    const int64_t per = (nvec + gridDim.x - 1) / gridDim.x;
    const int64_t vb = (int64_t)blockIdx.x * per;
    const int64_t ve = min(nvec, vb + per);
    int64_t v = vb + threadIdx.x;
    for (; v + (kUnroll - 1) * kBlock < ve; v += kUnroll * kBlock) {
        if constexpr (VB == 32) {
            Raw<32> ra[kUnroll], rb[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                ra[u] = ld_stream32(ba + (v + u * kBlock) * V);
                rb[u] = ld_stream32(bb + (v + u * kBlock) * V);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int k = 0; k < V; ++k)
                    acc[k] = M::combine(acc[k], elem(raw_get<In>(ra[u], k), raw_get<In>(rb[u], k)));
        } else {
            In ra[kUnroll], rb[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                ra[u] = ba[v + u * kBlock];
                rb[u] = bb[v + u * kBlock];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) acc[0] = M::combine(acc[0], elem(ra[u], rb[u]));
        }
    }
    for (; v < ve; v += kBlock) {
#pragma unroll
        for (int k = 0; k < V; ++k) acc[k] = M::combine(acc[k], elem(ba[v * V + k], bb[v * V + k]));
    }
    if (blockIdx.x == 0 && threadIdx.x < head) acc[0] = M::combine(acc[0], elem(a[threadIdx.x], b[threadIdx.x]));
    const int64_t tail = head + nvec * V;
    if (blockIdx.x == gridDim.x - 1 && tail + threadIdx.x < n)
        acc[V - 1] = M::combine(acc[V - 1], elem(a[tail + threadIdx.x], b[tail + threadIdx.x]));

    griddep_launch_dependents();
    P r = acc[0];
#pragma unroll
    for (int k = 1; k < V; ++k) r = M::combine(r, acc[k]);
    r = block_reduce<M, kBlock>(r, smem);
    if (threadIdx.x == 0) {
        if (gridDim.x == 1) store_result<Acc, Out, M>(r, st);
        else partials[blockIdx.x] = r;
    }
}

// Second pass: one block folds the partials in block order and stores.
template <class Acc, class Out, class M>
__global__ void __launch_bounds__(kFinishBlock) k_reduce_finish(const typename M::P* partials, int g,
                                                                StoreSpec<Acc, Out, M> st) {
    using P = typename M::P;
    __shared__ P smem[kFinishBlock / kWarp];
    griddep_wait();
    const int per = (g + kFinishBlock - 1) / kFinishBlock;
    const int b = threadIdx.x * per, e = min(g, b + per);
    P a = M::empty();
    for (int i = b; i < e; ++i) a = M::combine(a, partials[i]);
    a = block_reduce<M, kFinishBlock>(a, smem);
    if (threadIdx.x == 0) store_result<Acc, Out, M>(a, st);
}

template <class K, class... Args>
cudaError_t launch_pdl(K kernel, int grid, int block, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <class In, class Acc, class Out, class Map, class M>
ak_status launch(const ReduceCall& c, const ReducePlan& plan) {
    using P = typename M::P;
    StoreSpec<Acc, Out, M> st;
    st.mode = c.mode;
    memcpy(&st.init, c.init.b, sizeof(Acc));
    st.dst = static_cast<Out*>(c.dst);
    st.bare = static_cast<P*>(c.bare);
    st.flag = static_cast<unsigned long long*>(c.host_flag);
    st.seq = c.host_seq;
    P* partials = reinterpret_cast<P*>(static_cast<char*>(c.ws) + plan.partials_off);
    const In* x = static_cast<const In*>(c.src);
    const int g = plan.grid;
    if constexpr (M::commutative) {
        constexpr int V = kVecBytes / sizeof(In);
        const uintptr_t addr = reinterpret_cast<uintptr_t>(x);
        int64_t head = (int64_t)(((kVecBytes - addr % kVecBytes) % kVecBytes) / sizeof(In));
        head = std::min<int64_t>(head, c.n);
        const int64_t nvec = (c.n - head) / V;
        k_reduce_pass1<In, Acc, Out, Map, M><<<g, kBlock, 0, c.stream>>>(x, c.n, head, nvec, partials, st);
    } else {
        k_reduce_pass1_ordered<In, Acc, Out, Map, M><<<g, kBlockOrd, 0, c.stream>>>(x, c.n, partials, st);
    }
    ak_status s = check_launch();
    if (s != AK_OK) return s;
    count_launches(1);
    if (g > 1) {
        cudaError_t e = launch_pdl(k_reduce_finish<Acc, Out, M>, 1, kFinishBlock, c.stream,
                                   (const P*)partials, g, st);
        if (e != cudaSuccess) return cuda_fail(e);
        count_launches(1);
    }
    return AK_OK;
}

// The fused two-source reduction: first pass over f(a_i, b_i), then the
// same one-block finish.
template <class In, class Acc, class Out, class Map2, class M>
ak_status launch2(const ReduceCall& c, const ReducePlan& plan) {
    static_assert(M::commutative, "fused sources take commutative operators");
    using P = typename M::P;
    StoreSpec<Acc, Out, M> st;
    st.mode = c.mode;
    memcpy(&st.init, c.init.b, sizeof(Acc));
    st.dst = static_cast<Out*>(c.dst);
    st.bare = static_cast<P*>(c.bare);
    st.flag = static_cast<unsigned long long*>(c.host_flag);
    st.seq = c.host_seq;
    P* partials = reinterpret_cast<P*>(static_cast<char*>(c.ws) + plan.partials_off);
    const In* a = static_cast<const In*>(c.src);
    const In* b = static_cast<const In*>(c.src2);
    const int g = plan.grid;
    const uintptr_t aa = reinterpret_cast<uintptr_t>(a), ab = reinterpret_cast<uintptr_t>(b);
    if (aa % kVecBytes == ab % kVecBytes) {
        constexpr int V = kVecBytes / sizeof(In);
        int64_t head = (int64_t)(((kVecBytes - aa % kVecBytes) % kVecBytes) / sizeof(In));
        head = std::min<int64_t>(head, c.n);
        const int64_t nvec = (c.n - head) / V;
        k_reduce2_pass1<In, Acc, Out, Map2, M, kVecBytes><<<g, kBlock, 0, c.stream>>>(a, b, c.n, head, nvec,
                                                                                      partials, st);
    } else {
        k_reduce2_pass1<In, Acc, Out, Map2, M, (int)sizeof(In)><<<g, kBlock, 0, c.stream>>>(a, b, c.n, 0, c.n,
                                                                                           partials, st);
    }
    ak_status s = check_launch();
    if (s != AK_OK) return s;
    count_launches(1);
    if (g > 1) {
        cudaError_t e = launch_pdl(k_reduce_finish<Acc, Out, M>, 1, kFinishBlock, c.stream, (const P*)partials, g, st);
        if (e != cudaSuccess) return cuda_fail(e);
        count_launches(1);
    }
    return AK_OK;
}

// Grid of the first pass and workspace layout from element / partial sizes
// (the C entry points plan through plan_reduce, the template API directly).
inline void plan_sizes(int64_t n, size_t esz, size_t psz, bool ordered, int target_blocks, int sm_count,
                       ReducePlan* plan) {
    const int max_grid = sm_count * kMaxBlocksPerSm;
    int64_t per_block = ordered ? (int64_t)kBlockOrd * kRunOrd : (int64_t)kBlock * (kVecBytes / (int64_t)esz);
    if (per_block < 1) per_block = kBlock;
    int64_t g = (n + per_block - 1) / per_block;
    g = std::max<int64_t>(1, std::min<int64_t>(g, max_grid));
    if (target_blocks > 0) g = std::min<int64_t>(g, target_blocks);
    if (n <= kSingleLaunchMax) g = 1;
    plan->grid = (int)g;
    plan->partials_off = kWsHeader;
    plan->bare_off = align_up(kWsHeader + (size_t)max_grid * psz, 64);
    plan->ws_bytes = align_up(plan->bare_off + psz, 256);
}

}  // namespace red
}  // namespace ak
