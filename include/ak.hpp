/*
 * ak.hpp -- C++ template API of the GB300 reduce / scan library: the
 * whole-array reduction and the scans under a USER associative operator.
 *
 * The pages state the problem for any associative operator: mapreduce(f, op,
 * A) with operators that may lack a neutral element or be non-commutative
 * ("Finish whole-array reductions on the device", PR #139, section
 * "Compatibility"; the tile-scan PR #202: Optional partials for operators
 * without a neutral element, 16-byte non-commutative partials in paragraph
 * "Alternatives"). The C ABI (ak.h) offers a closed set of operators; this
 * header instantiates the same kernels for the caller's own operator inside
 * the caller's translation unit: the whole-array reduction (reduce), the
 * reduction over a set of dimensions (reduce_dims) and the scan
 * (accumulate). Compile that unit with nvcc for sm_103a
 * (-gencode arch=compute_103a,code=sm_103a -std=c++17
 * --expt-relaxed-constexpr) and link it with libak.so, which holds the
 * host-side bookkeeping the launchers share (device properties, call
 * epochs, launch counter, CUDA error record).
 *
 * The operator
 * ------------
 *   struct MyOp {
 *     static constexpr bool commutative = ...;   // may the kernels reorder the fold?
 *     static constexpr bool has_identity = ...;  // is there a neutral element?
 *     __host__ __device__ static T apply(const T& a, const T& b);  // a is the left operand
 *     template <class U> __host__ __device__ static U identity();  // only if has_identity
 *   };
 * apply must be associative. Non-commutative operators keep the element
 * order exactly (ordered first pass, ordered combines, left-to-right scans).
 * Without an identity the partial results carry an Optional flag
 * (Opt<T>: the empty range is "absent"), as for ak_opts.no_neutral.
 * T: a trivially copyable type of 4, 8 or 16 bytes, e.g. float, int64_t, a
 * pair of uint32; arrays of T start on a multiple of sizeof(T) (the kernels
 * read whole 32-byte vectors of them).
 * Map (reduction only): struct { __host__ __device__ static T apply(T); },
 * applied to every element before op; ak::MapIdentity by default.
 *
 * Conventions as in ak.h: device pointers for arrays, a host pointer for
 * init (applied once, leftmost; nullable), caller-owned workspace of the
 * reported size, asynchronous on `stream`, errors as ak_status.
 */
#ifndef AK_HPP
#define AK_HPP

#include <algorithm>
#include <type_traits>

#include "ak.h"
#include "../mapreduce_prefix_scan_gb300/csrc/reduce.cuh"
#include "../mapreduce_prefix_scan_gb300/csrc/reduce_dims.cuh"
#include "../mapreduce_prefix_scan_gb300/csrc/scan.cuh"

namespace ak {

// The partial-result monoid of a user operator.
template <class Op, class T>
using monoid_of = std::conditional_t<Op::has_identity, Plain<Op, T>, Lifted<Op, T>>;

namespace user {

template <class T>
__global__ void k_store_one(T* dst, T v) {
    *dst = v;
}

template <class T>
inline ak_status store_one(T* dst, const T& v, cudaStream_t stream) {
    k_store_one<T><<<1, 1, 0, stream>>>(dst, v);
    const ak_status s = check_launch();
    if (s == AK_OK) count_launches(1);
    return s;
}

template <class T>
constexpr bool supported() {
    return std::is_trivially_copyable_v<T> && (sizeof(T) == 4 || sizeof(T) == 8 || sizeof(T) == 16);
}

template <class T>
inline bool size_aligned(const void* p) {
    return reinterpret_cast<uintptr_t>(p) % sizeof(T) == 0;
}

template <class T>
__global__ void k_fill(T* dst, int64_t n, T v) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = v;
}

template <class T>
inline ak_status fill(T* dst, int64_t n, const T& v, cudaStream_t stream) {
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4096);
    k_fill<T><<<(unsigned)blocks, 256, 0, stream>>>(dst, n, v);
    const ak_status s = check_launch();
    if (s == AK_OK) count_launches(1);
    return s;
}

// A built-in element type of T's size: the planners size vectors, partials
// and workspaces by it (a partial of T never outgrows that of the carrier).
template <class T>
constexpr ak_dtype carrier() {
    return sizeof(T) == 4 ? AK_I32 : (sizeof(T) == 8 ? AK_I64 : AK_MAT2_MODP);
}

}  // namespace user

// ---------------------------------------------------------------------------
// reduce: *dst = op(init?, f(src[0]), ..., f(src[n-1]))
// ---------------------------------------------------------------------------

template <class T, class Op, class Map = MapIdentity>
ak_status reduce_workspace_size(int64_t n, size_t* bytes) {
    static_assert(user::supported<T>(), "T: trivially copyable, 4, 8 or 16 bytes");
    using M = monoid_of<Op, T>;
    if (!bytes || n < 0) return AK_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    ReducePlan plan;
    red::plan_sizes(n > 0 ? n : 1, sizeof(T), sizeof(typename M::P), !M::commutative, 0, dev.sm_count, &plan);
    *bytes = plan.ws_bytes;
    return AK_OK;
}

template <class T, class Op, class Map = MapIdentity>
ak_status reduce(const T* src, int64_t n, T* dst, const T* init, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
    static_assert(user::supported<T>(), "T: trivially copyable, 4, 8 or 16 bytes");
    using M = monoid_of<Op, T>;
    if (n < 0 || !dst || (n > 0 && !src)) return AK_ERR_INVALID_ARG;
    if (!user::size_aligned<T>(src) || !user::size_aligned<T>(dst)) return AK_ERR_INVALID_ARG;
    if (n == 0) {
        if (init) return user::store_one(dst, *init, stream);
        if constexpr (Op::has_identity) return user::store_one(dst, Op::template identity<T>(), stream);
        else return AK_ERR_EMPTY_NO_INIT;
    }
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    ReducePlan plan;
    red::plan_sizes(n, sizeof(T), sizeof(typename M::P), !M::commutative, 0, dev.sm_count, &plan);
    if (!workspace || workspace_bytes < plan.ws_bytes || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return AK_ERR_WORKSPACE;
    ReduceCall c;
    memset(&c, 0, sizeof c);
    c.src = src;
    c.src2 = nullptr;
    c.n = n;
    c.mode = init ? AK_STORE_INIT : AK_STORE_OVERWRITE;
    if (init) memcpy(c.init.b, init, sizeof(T));
    c.dst = dst;
    c.bare = nullptr;
    c.ws = workspace;
    c.ws_bytes = workspace_bytes;
    c.stream = stream;
    return red::launch<T, T, T, Map, M>(c, plan);
}

// ---------------------------------------------------------------------------
// reduce_dims: dst[kept index] = op(init?, f(src[...]) over the reduced dims)
// ---------------------------------------------------------------------------
//
// As ak_reduce_dims (ak.h): a column-major array of ndim <= 8 dimensions
// (shape, element strides or NULL for dense), the dimensions in dims_mask
// (bit d = dimension d) reduced, the kept ones laid out densely in dst in
// column-major order; init, when given, is applied once per output,
// leftmost. Non-commutative operators keep the element order along the
// reduced dimensions.

template <class T, class Op, class Map = MapIdentity>
ak_status reduce_dims_workspace_size(int ndim, const int64_t* shape, const int64_t* strides, uint32_t dims_mask,
                                     size_t* bytes) {
    static_assert(user::supported<T>(), "T: trivially copyable, 4, 8 or 16 bytes");
    ak_opts o;
    ak_opts_default(&o);
    o.no_neutral = Op::has_identity ? 0 : 1;
    return ak_reduce_dims_workspace_size(ndim, shape, strides, dims_mask, user::carrier<T>(), user::carrier<T>(), &o,
                                         bytes);
}

template <class T, class Op, class Map = MapIdentity>
ak_status reduce_dims(const T* src, int ndim, const int64_t* shape, const int64_t* strides, uint32_t dims_mask,
                      T* dst, const T* init, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    static_assert(user::supported<T>(), "T: trivially copyable, 4, 8 or 16 bytes");
    using M = monoid_of<Op, T>;
    const ak_dtype dt = user::carrier<T>();
    if (sizeof(typename M::P) > partial_size(dt, !Op::has_identity)) return AK_ERR_UNSUPPORTED;
    ak_opts o;
    ak_opts_default(&o);
    o.no_neutral = Op::has_identity ? 0 : 1;
    DimsSetup d;
    ak_status s = setup_dims(src, ndim, shape, strides, dims_mask, dt, dt, o, &d);
    if (s != AK_OK) return s;
    const int64_t nin = d.cn.nout * d.cn.nfold;
    if ((nin > 0 && !src) || (d.cn.nout > 0 && !dst)) return AK_ERR_INVALID_ARG;
    if (!user::size_aligned<T>(src) || !user::size_aligned<T>(dst)) return AK_ERR_INVALID_ARG;
    if (d.cn.nout == 0) return AK_OK;
    if (d.cn.nfold == 0) {
        if (init) return user::fill(dst, d.cn.nout, *init, stream);
        if constexpr (Op::has_identity) return user::fill(dst, d.cn.nout, Op::template identity<T>(), stream);
        else return AK_ERR_EMPTY_NO_INIT;
    }
    if (!workspace || workspace_bytes < d.ws_bytes || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return AK_ERR_WORKSPACE;
    const ak_store mode = init ? AK_STORE_INIT : AK_STORE_OVERWRITE;
    if (d.path == 1) {
        ReduceCall c;
        memset(&c, 0, sizeof c);
        c.src = src;
        c.n = d.cn.nfold;
        c.mode = mode;
        if (init) memcpy(c.init.b, init, sizeof(T));
        c.dst = dst;
        c.ws = workspace;
        c.ws_bytes = workspace_bytes;
        c.stream = stream;
        return red::launch<T, T, T, Map, M>(c, d.rplan);
    }
    DimsCall& c = d.c;
    c.out = dt;
    c.mode = mode;
    memset(c.init.b, 0, sizeof c.init.b);
    if (init) memcpy(c.init.b, init, sizeof(T));
    c.dst = dst;
    c.ws = workspace;
    c.ws_bytes = workspace_bytes;
    c.stream = stream;
    return dims::launch<T, T, T, Map, M>(c, d.dplan);
}

// ---------------------------------------------------------------------------
// accumulate: the inclusive (or exclusive) scan of one line of n elements
// ---------------------------------------------------------------------------

template <class T, class Op>
constexpr bool tma_eligible() {
    return Op::has_identity &&
           (std::is_same_v<T, float> || std::is_same_v<T, int32_t> || std::is_same_v<T, int64_t>);
}

template <class T, class Op>
ak_status accumulate_workspace_size(int64_t n, size_t* bytes) {
    static_assert(user::supported<T>(), "T: trivially copyable, 4, 8 or 16 bytes");
    using M = monoid_of<Op, T>;
    if (!bytes || n < 0) return AK_ERR_INVALID_ARG;
    const bool o_single_pass = false;
    ScanPlan p;
    const ak_status s = scan::plan_sizes(1, n, 1, sizeof(T), sizeof(typename M::P), tma_eligible<T, Op>(), 0, &p, sizeof(T),
                                          o_single_pass);
    if (s != AK_OK) return s;
    *bytes = p.ws_bytes;
    return AK_OK;
}

// dst[i] = op(init?, src[0], ..., src[i]); with `exclusive`, dst[i] = op(init,
// src[0], ..., src[i-1]) (dst[0] = init; without init the identity stands
// for it, and an operator without one gives AK_ERR_EMPTY_NO_INIT). dst may
// equal src. opts: NULL or ak_opts (wait_limit_ns, check, fault injection).
template <class T, class Op>
ak_status accumulate(const T* src, T* dst, int64_t n, const T* init, bool exclusive, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream, const ak_opts* opts = nullptr) {
    static_assert(user::supported<T>(), "T: trivially copyable, 4, 8 or 16 bytes");
    using M = monoid_of<Op, T>;
    if (n < 0) return AK_ERR_INVALID_ARG;
    if (n == 0) return AK_OK;
    if (!src || !dst || !user::size_aligned<T>(src) || !user::size_aligned<T>(dst)) return AK_ERR_INVALID_ARG;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(src), b0 = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t bytes = (uintptr_t)n * sizeof(T);
    if (a0 != b0 && a0 < b0 + bytes && b0 < a0 + bytes) return AK_ERR_INVALID_ARG;
    ak_opts o;
    ak_opts_default(&o);
    if (opts) o = *opts;
    if (o.wait_limit_ns <= 0) o.wait_limit_ns = 1000000000LL;
    const bool o_single_pass = o.debug_skip_publish_tile >= 0;  // fault injection needs the single-pass waits
    ScanPlan p;
    ak_status s = scan::plan_sizes(1, n, 1, sizeof(T), sizeof(typename M::P), tma_eligible<T, Op>(), 0, &p, sizeof(T),
                                          o_single_pass);
    if (s != AK_OK) return s;
    if (!workspace || workspace_bytes < p.ws_bytes || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return AK_ERR_WORKSPACE;
    ScanCall c;
    memset(&c, 0, sizeof c);
    c.src = src;
    c.dst = dst;
    c.inner = 1;
    c.len = n;
    c.outer = 1;
    c.no_neutral = !Op::has_identity;
    c.has_init = init != nullptr;
    c.exclusive = exclusive;
    if (init) memcpy(c.init.b, init, sizeof(T));
    if (exclusive && !init) {
        if constexpr (Op::has_identity) {
            const T id = Op::template identity<T>();
            memcpy(c.init.b, &id, sizeof(T));
            c.has_init = true;
        } else {
            return AK_ERR_EMPTY_NO_INIT;
        }
    }
    c.ws = workspace;
    c.ws_bytes = workspace_bytes;
    c.wait_limit_ns = o.wait_limit_ns;
    c.skip_tile = o.debug_skip_publish_tile;
    c.epoch = next_epoch();
    c.stream = stream;
    s = scan::launch<T, T, T, M>(c, p);
    if (s != AK_OK || !o.check) return s;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return ak_scan_status(workspace);
}

}  // namespace ak

#endif  // AK_HPP
