// ak_types.cuh -- element types, maps, operators and partial-result types of
// the GB300 reduce / scan kernels.
//
// The problem statement follows the AcceleratedKernels.jl pull requests:
// "Finish whole-array reductions on the device" (#139; sections "What
// changes" and "Compatibility": init is applied once, partial results keep
// the accumulator type until the final store, R never holds intermediates),
// and the tile-scan PR (#202; first paragraph: operators without a neutral
// element carry Optional partials; paragraph "Alternatives": 16-byte
// non-commutative partials).
#pragma once

#include <cstdint>
#include <cstring>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#define AK_HD __host__ __device__ __forceinline__

namespace ak {

// --------------------------------------------------------------------------
// element types
// --------------------------------------------------------------------------

constexpr uint32_t kModP = 2147483647u;  // 2^31 - 1, a Mersenne prime

// A 2x2 matrix over Z/pZ, column-major entries (a11, a21, a12, a22): the
// 16-byte non-commutative element of the matrix-product scans.
struct alignas(16) Mat2 {
    uint32_t a11, a21, a12, a22;
};

using bf16 = __nv_bfloat16;

// Optional partial: the accumulator of an operator with no neutral element.
// An absent value is the empty prefix; combining with it returns the other
// operand unchanged. For a Float32 accumulator this is 8 bytes.
template <class T>
struct Opt {
    T v;
    uint32_t present;
};

// --------------------------------------------------------------------------
// conversions: input -> accumulator -> output
// --------------------------------------------------------------------------

template <class To, class From>
struct Convert {
    static AK_HD To apply(From x) { return static_cast<To>(x); }
};
template <class T>
struct Convert<T, T> {
    static AK_HD T apply(T x) { return x; }
};
template <>
struct Convert<float, bf16> {
    static AK_HD float apply(bf16 x) { return __bfloat162float(x); }
};
template <>
struct Convert<bf16, float> {
    static AK_HD bf16 apply(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Convert<int32_t, int64_t> {  // wraps modulo 2^32
    static AK_HD int32_t apply(int64_t x) { return static_cast<int32_t>(static_cast<uint32_t>(x)); }
};

template <class To, class From>
AK_HD To convert(From x) { return Convert<To, From>::apply(x); }

// --------------------------------------------------------------------------
// wrapping integer arithmetic (two's complement, no undefined behaviour)
// --------------------------------------------------------------------------

AK_HD int32_t wadd(int32_t a, int32_t b) { return (int32_t)((uint32_t)a + (uint32_t)b); }
AK_HD int64_t wadd(int64_t a, int64_t b) { return (int64_t)((uint64_t)a + (uint64_t)b); }
AK_HD int32_t wmul(int32_t a, int32_t b) { return (int32_t)((uint32_t)a * (uint32_t)b); }
AK_HD int64_t wmul(int64_t a, int64_t b) { return (int64_t)((uint64_t)a * (uint64_t)b); }
AK_HD int32_t wneg(int32_t a) { return (int32_t)(0u - (uint32_t)a); }
AK_HD int64_t wneg(int64_t a) { return (int64_t)(0ull - (uint64_t)a); }

// --------------------------------------------------------------------------
// maps f applied to each element, in the accumulator type
// --------------------------------------------------------------------------

struct MapIdentity {
    template <class T>
    static AK_HD T apply(T x) { return x; }
};

struct MapAbs {
    static AK_HD float apply(float x) { return fabsf(x); }
    static AK_HD double apply(double x) { return fabs(x); }
    static AK_HD int32_t apply(int32_t x) { return x < 0 ? wneg(x) : x; }
    static AK_HD int64_t apply(int64_t x) { return x < 0 ? wneg(x) : x; }
};

struct MapAbs2 {
    static AK_HD float apply(float x) { return x * x; }
    static AK_HD double apply(double x) { return x * x; }
    static AK_HD int32_t apply(int32_t x) { return wmul(x, x); }
    static AK_HD int64_t apply(int64_t x) { return wmul(x, x); }
};

// maps f(a, b) of a fused two-source element (a Broadcasted source such as
// x .* y or abs2.(x .- y)), applied in the accumulator type; integers wrap
AK_HD int32_t wsub(int32_t a, int32_t b) { return (int32_t)((uint32_t)a - (uint32_t)b); }
AK_HD int64_t wsub(int64_t a, int64_t b) { return (int64_t)((uint64_t)a - (uint64_t)b); }

struct Map2Mul {
    static AK_HD float apply(float a, float b) { return a * b; }
    static AK_HD double apply(double a, double b) { return a * b; }
    static AK_HD int32_t apply(int32_t a, int32_t b) { return wmul(a, b); }
    static AK_HD int64_t apply(int64_t a, int64_t b) { return wmul(a, b); }
};

struct Map2SqDiff {
    static AK_HD float apply(float a, float b) { const float d = a - b; return d * d; }
    static AK_HD double apply(double a, double b) { const double d = a - b; return d * d; }
    static AK_HD int32_t apply(int32_t a, int32_t b) { const int32_t d = wsub(a, b); return wmul(d, d); }
    static AK_HD int64_t apply(int64_t a, int64_t b) { const int64_t d = wsub(a, b); return wmul(d, d); }
};

struct Map2AbsDiff {
    static AK_HD float apply(float a, float b) { return fabsf(a - b); }
    static AK_HD double apply(double a, double b) { return fabs(a - b); }
    static AK_HD int32_t apply(int32_t a, int32_t b) { const int32_t d = wsub(a, b); return d < 0 ? wneg(d) : d; }
    static AK_HD int64_t apply(int64_t a, int64_t b) { const int64_t d = wsub(a, b); return d < 0 ? wneg(d) : d; }
};

// --------------------------------------------------------------------------
// operators
// --------------------------------------------------------------------------

AK_HD float canonical_nan_f() {
    uint32_t u = 0x7fc00000u;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
AK_HD double canonical_nan_d() {
    uint64_t u = 0x7ff8000000000000ull;
    double f;
    memcpy(&f, &u, 8);
    return f;
}

// Julia's max / min on floats: NaN wins (returned as the canonical quiet NaN)
// and +0.0 > -0.0. This is the maximum of a total order, so any association
// tree gives the same bits.
template <class F>
AK_HD F julia_max(F a, F b, F nan) {
    if (a != a || b != b) return nan;
    if (a > b) return a;
    if (b > a) return b;
    return signbit(a) ? b : a;
}
template <class F>
AK_HD F julia_min(F a, F b, F nan) {
    if (a != a || b != b) return nan;
    if (a < b) return a;
    if (b < a) return b;
    return signbit(a) ? a : b;
}

// (a*b + c*d) mod p for a, b, c, d < p: the sum is < 2^63; two Mersenne folds
// (2^31 = 1 mod p) bring it below p + 4, one conditional subtraction below p.
AK_HD uint32_t mulmod2(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    uint64_t s = (uint64_t)a * b + (uint64_t)c * d;
    uint64_t t = (s & kModP) + (s >> 31);
    t = (t & kModP) + (t >> 31);
    return (uint32_t)(t >= kModP ? t - kModP : t);
}

AK_HD Mat2 matmul_modp(const Mat2& a, const Mat2& b) {
    Mat2 c;
    c.a11 = mulmod2(a.a11, b.a11, a.a12, b.a21);
    c.a21 = mulmod2(a.a21, b.a11, a.a22, b.a21);
    c.a12 = mulmod2(a.a11, b.a12, a.a12, b.a22);
    c.a22 = mulmod2(a.a21, b.a12, a.a22, b.a22);
    return c;
}

// Each operator: apply(a, b) with a on the left; identity<T>() where one
// exists; commutative tells the kernels whether the fold order may change.
struct OpAdd {
    static constexpr bool commutative = true;
    static constexpr bool has_identity = true;
    static AK_HD float apply(float a, float b) { return a + b; }
    static AK_HD double apply(double a, double b) { return a + b; }
    static AK_HD int32_t apply(int32_t a, int32_t b) { return wadd(a, b); }
    static AK_HD int64_t apply(int64_t a, int64_t b) { return wadd(a, b); }
    // -0.0 is the additive identity of IEEE floats (x + -0.0 == x for every x).
    template <class T>
    static AK_HD T identity() {
        if constexpr (std::is_floating_point_v<T>) return T(-0.0);
        else return T(0);
    }
};

struct OpMul {
    static constexpr bool commutative = true;
    static constexpr bool has_identity = true;
    static AK_HD float apply(float a, float b) { return a * b; }
    static AK_HD double apply(double a, double b) { return a * b; }
    static AK_HD int32_t apply(int32_t a, int32_t b) { return wmul(a, b); }
    static AK_HD int64_t apply(int64_t a, int64_t b) { return wmul(a, b); }
    template <class T>
    static AK_HD T identity() { return T(1); }
};

struct OpMax {
    static constexpr bool commutative = true;
    static constexpr bool has_identity = true;
    static AK_HD float apply(float a, float b) { return julia_max(a, b, canonical_nan_f()); }
    static AK_HD double apply(double a, double b) { return julia_max(a, b, canonical_nan_d()); }
    static AK_HD int32_t apply(int32_t a, int32_t b) { return a > b ? a : b; }
    static AK_HD int64_t apply(int64_t a, int64_t b) { return a > b ? a : b; }
    template <class T>
    static AK_HD T identity() {
        if constexpr (std::is_floating_point_v<T>) return -T(INFINITY);
        else if constexpr (sizeof(T) == 4) return (T)INT32_MIN;
        else return (T)INT64_MIN;
    }
};

struct OpMin {
    static constexpr bool commutative = true;
    static constexpr bool has_identity = true;
    static AK_HD float apply(float a, float b) { return julia_min(a, b, canonical_nan_f()); }
    static AK_HD double apply(double a, double b) { return julia_min(a, b, canonical_nan_d()); }
    static AK_HD int32_t apply(int32_t a, int32_t b) { return a < b ? a : b; }
    static AK_HD int64_t apply(int64_t a, int64_t b) { return a < b ? a : b; }
    template <class T>
    static AK_HD T identity() {
        if constexpr (std::is_floating_point_v<T>) return T(INFINITY);
        else if constexpr (sizeof(T) == 4) return (T)INT32_MAX;
        else return (T)INT64_MAX;
    }
};

struct OpMatMul {
    static constexpr bool commutative = false;
    static constexpr bool has_identity = true;
    static AK_HD Mat2 apply(const Mat2& a, const Mat2& b) { return matmul_modp(a, b); }
    template <class T>
    static AK_HD T identity() { return Mat2{1u, 0u, 0u, 1u}; }
};

// --------------------------------------------------------------------------
// monoids: how partial results combine
// --------------------------------------------------------------------------

// Plain: the partial is the accumulator itself and empty ranges hold the
// operator's identity.
template <class Op, class Acc>
struct Plain {
    using op = Op;
    using acc = Acc;
    using P = Acc;
    static constexpr bool commutative = Op::commutative;
    static AK_HD P empty() { return Op::template identity<Acc>(); }
    static AK_HD P lift(Acc a) { return a; }
    static AK_HD P combine(const P& a, const P& b) { return Op::apply(a, b); }
    static AK_HD bool present(const P&) { return true; }
    static AK_HD Acc value(const P& p) { return p; }
};

// Lifted: the operator is treated as having no neutral element; partials are
// Opt<Acc> and the empty range is the absent value.
template <class Op, class Acc>
struct Lifted {
    using op = Op;
    using acc = Acc;
    using P = Opt<Acc>;
    static constexpr bool commutative = Op::commutative;
    static AK_HD P empty() {
        P p;
        memset(&p, 0, sizeof p);
        return p;
    }
    static AK_HD P lift(Acc a) {
        P p;
        memset(&p, 0, sizeof p);
        p.v = a;
        p.present = 1u;
        return p;
    }
    static AK_HD P combine(const P& a, const P& b) {
        if (!a.present) return b;
        if (!b.present) return a;
        return lift(Op::apply(a.v, b.v));
    }
    static AK_HD bool present(const P& p) { return p.present != 0u; }
    static AK_HD Acc value(const P& p) { return p.v; }
};

}  // namespace ak
