// user_ops.cu -- a caller's translation unit for the template API tests:
// operators the C ABI does not offer, compiled against include/ak.hpp.
//
//   Affine          v -> a*v + b mod p (p = 2^31 - 1), composed left to right:
//                   op(f, g) applies f first, then g -- associative, not
//                   commutative, identity (1, 0); 8-byte elements.
//   AffineNoId      the same operator declared without an identity (Optional
//                   partials).
//   UserAdd         float addition declared by the caller (commutative,
//                   identity 0): takes the TMA tile scan.
// The extern "C" wrappers below (reduce, reduce over dimensions, scan) are
// what the test calls through ctypes.
#include <cstdint>

#include "ak.hpp"

namespace {

constexpr uint64_t kP = 2147483647ull;

struct Affine {
    uint32_t a, b;
};

struct AffineCompose {
    static constexpr bool commutative = false;
    static constexpr bool has_identity = true;
    __host__ __device__ static Affine apply(const Affine& f, const Affine& g) {
        Affine r;
        r.a = (uint32_t)(((uint64_t)g.a * f.a) % kP);
        r.b = (uint32_t)(((uint64_t)g.a * f.b + g.b) % kP);
        return r;
    }
    template <class U>
    __host__ __device__ static U identity() {
        return U{1u, 0u};
    }
};

struct AffineComposeNoId {
    static constexpr bool commutative = false;
    static constexpr bool has_identity = false;
    __host__ __device__ static Affine apply(const Affine& f, const Affine& g) { return AffineCompose::apply(f, g); }
};

struct UserAdd {
    static constexpr bool commutative = true;
    static constexpr bool has_identity = true;
    __host__ __device__ static float apply(float a, float b) { return a + b; }
    template <class U>
    __host__ __device__ static U identity() {
        return U(0);
    }
};

}  // namespace

extern "C" int user_affine_ws(int64_t n, int scan, int no_id, size_t* bytes) {
    if (scan) return no_id ? ak::accumulate_workspace_size<Affine, AffineComposeNoId>(n, bytes)
                           : ak::accumulate_workspace_size<Affine, AffineCompose>(n, bytes);
    return no_id ? ak::reduce_workspace_size<Affine, AffineComposeNoId>(n, bytes)
                 : ak::reduce_workspace_size<Affine, AffineCompose>(n, bytes);
}

extern "C" int user_affine_reduce(const void* src, int64_t n, void* dst, const void* init, int no_id, void* ws,
                                  size_t ws_bytes, void* stream) {
    auto x = static_cast<const Affine*>(src);
    auto y = static_cast<Affine*>(dst);
    auto i = static_cast<const Affine*>(init);
    auto s = static_cast<cudaStream_t>(stream);
    return no_id ? ak::reduce<Affine, AffineComposeNoId>(x, n, y, i, ws, ws_bytes, s)
                 : ak::reduce<Affine, AffineCompose>(x, n, y, i, ws, ws_bytes, s);
}

extern "C" int user_affine_scan(const void* src, void* dst, int64_t n, const void* init, int exclusive, int no_id,
                                void* ws, size_t ws_bytes, void* stream) {
    auto x = static_cast<const Affine*>(src);
    auto y = static_cast<Affine*>(dst);
    auto i = static_cast<const Affine*>(init);
    auto s = static_cast<cudaStream_t>(stream);
    ak_opts o;
    ak_opts_default(&o);
    o.check = 1;
    return no_id ? ak::accumulate<Affine, AffineComposeNoId>(x, y, n, i, exclusive != 0, ws, ws_bytes, s, &o)
                 : ak::accumulate<Affine, AffineCompose>(x, y, n, i, exclusive != 0, ws, ws_bytes, s, &o);
}

extern "C" int user_add_ws(int64_t n, int scan, size_t* bytes) {
    return scan ? ak::accumulate_workspace_size<float, UserAdd>(n, bytes) : ak::reduce_workspace_size<float, UserAdd>(n, bytes);
}

extern "C" int user_add_reduce(const float* src, int64_t n, float* dst, void* ws, size_t ws_bytes, void* stream) {
    return ak::reduce<float, UserAdd>(src, n, dst, nullptr, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int user_add_scan(const float* src, float* dst, int64_t n, int exclusive, void* ws, size_t ws_bytes,
                             void* stream) {
    return ak::accumulate<float, UserAdd>(src, dst, n, nullptr, exclusive != 0, ws, ws_bytes,
                                          static_cast<cudaStream_t>(stream));
}

extern "C" int user_affine_dims_ws(int ndim, const int64_t* shape, const int64_t* strides, uint32_t mask, int no_id,
                                   size_t* bytes) {
    return no_id ? ak::reduce_dims_workspace_size<Affine, AffineComposeNoId>(ndim, shape, strides, mask, bytes)
                 : ak::reduce_dims_workspace_size<Affine, AffineCompose>(ndim, shape, strides, mask, bytes);
}

extern "C" int user_affine_dims(const void* src, int ndim, const int64_t* shape, const int64_t* strides, uint32_t mask,
                                void* dst, const void* init, int no_id, void* ws, size_t ws_bytes, void* stream) {
    auto x = static_cast<const Affine*>(src);
    auto y = static_cast<Affine*>(dst);
    auto i = static_cast<const Affine*>(init);
    auto s = static_cast<cudaStream_t>(stream);
    return no_id ? ak::reduce_dims<Affine, AffineComposeNoId>(x, ndim, shape, strides, mask, y, i, ws, ws_bytes, s)
                 : ak::reduce_dims<Affine, AffineCompose>(x, ndim, shape, strides, mask, y, i, ws, ws_bytes, s);
}
