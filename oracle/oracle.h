/*
 * oracle.h -- sequential CPU oracle for reductions and inclusive scans.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, __graft_entry__.smoke() and the
 * bench's CPU-baseline / reference arm may call this library. It shares no
 * code, header, table or constant with the CUDA library; the two meet only in
 * the seeded inputs of synth.py.
 *
 * What it computes (AcceleratedKernels.jl PRs: "Finish whole-array reductions
 * on the device" (#139), sections "What changes" and "Compatibility"; the
 * strided-reduction PR #176, first list; the tile-scan PR #202, first
 * paragraph):
 *   reduce      r = op(init, f(x_1), f(x_2), ..., f(x_n)), folded strictly
 *               left to right, init applied once at the left when given;
 *   reduce_dims the same fold per output of a column-major array, over the
 *               reduced indices in increasing column-major order;
 *   scan        y_1 = op(init, x_1) (or x_1), y_i = op(y_{i-1}, x_i), for the
 *               whole array or along one dimension; the exclusive scan
 *               y_1 = init, y_i = op(y_{i-1}, x_{i-1});
 *   findall     the indices of the nonzero elements, in order;
 *   reduce2     the reduce of f(x_i, y_i) over two sources (a fused source);
 *   affine      scans / reduces of affine maps mod p (the test operator of the
 *               C++ template API).
 * No neutral element is ever used: every fold starts from init or from the
 * first element, which is the meaning of an operator without one.
 *
 * Arithmetic: float inputs (f32, f64, bf16) in f64, sums compensated
 * (Neumaier 1974) so the oracle's own error stays below about one f64 ulp of
 * the result; integers in exact two's-complement arithmetic wrapped to the
 * accumulator width (32 or 64 bits); 2x2 matrices mod p = 2^31 - 1 with
 * 64-bit products reduced by '%'.
 *
 * Element layouts: f32/f64 IEEE; bf16 as uint16 bit patterns; i32/i64 two's
 * complement; a 2x2 matrix as four uint32 entries in column-major order
 * (a11, a21, a12, a22), each in [0, p).
 *
 * Return codes: 0 ok; 1 empty reduction with no init (no value exists);
 * -1 bad argument.
 */
#ifndef AK_ORACLE_H
#define AK_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_F64 = 1, ORC_BF16 = 2, ORC_I32 = 3, ORC_I64 = 4, ORC_MAT2 = 5, ORC_U8 = 6 };
enum { ORC_MAP_IDENTITY = 0, ORC_MAP_ABS = 1, ORC_MAP_ABS2 = 2 };
enum { ORC_OP_ADD = 0, ORC_OP_MUL = 1, ORC_OP_MAX = 2, ORC_OP_MIN = 3, ORC_OP_MATMUL = 4 };
/* maps of two sources (fused / Broadcasted sources): x*y, (x-y)^2, |x-y| */
enum { ORC_MAP2_MUL = 0, ORC_MAP2_SQDIFF = 1, ORC_MAP2_ABSDIFF = 2 };

#define ORC_MODP 2147483647u

/* --- scalar helpers ---------------------------------------------------- */
/* f64 -> bf16 bit pattern, round to nearest, ties to even, in one rounding. */
uint16_t orc_bf16_rne(double v);
/* Julia max/min on floats: NaN wins; max(-0.0, +0.0) = +0.0, min = -0.0. */
double orc_fmax(double a, double b);
double orc_fmin(double a, double b);
/* C = A * B mod p, column-major 2x2. */
void orc_mat2_mul(const uint32_t a[4], const uint32_t b[4], uint32_t c[4]);

/* --- whole-array reduce ------------------------------------------------ */
int orc_reduce_float(const void* x, int64_t n, int in_type, int map, int op,
                     int has_init, double init, double* out);
int orc_reduce_int(const void* x, int64_t n, int in_type, int acc_bits, int map, int op,
                   int has_init, int64_t init, int64_t* out);
int orc_reduce_mat2(const uint32_t* x, int64_t n, const uint32_t* init /* nullable */,
                    uint32_t out[4]);

/* --- reduce over the dimensions set in dims_mask (bit d = dimension d,
 *     0-based, column-major shape); out is dense column-major over the
 *     shape with reduced extents set to 1. Empty reductions without init
 *     leave the output untouched and return 1. ----------------------------- */
int orc_reduce_dims_float(const void* x, int ndim, const int64_t* shape, uint32_t dims_mask,
                          int in_type, int map, int op, int has_init, double init, double* out);
int orc_reduce_dims_int(const void* x, int ndim, const int64_t* shape, uint32_t dims_mask,
                        int in_type, int acc_bits, int map, int op, int has_init, int64_t init,
                        int64_t* out);
int orc_reduce_dims_mat2(const uint32_t* x, int ndim, const int64_t* shape, uint32_t dims_mask,
                         const uint32_t* init, uint32_t* out);
/* The same over a strided view: element (i_1, ..., i_d) of the source sits at
 * sum_k i_k * strides[k] (elements; strides = NULL is the dense layout). The
 * output stays dense column-major. */
int orc_reduce_dims_float_s(const void* x, int ndim, const int64_t* shape, const int64_t* strides,
                            uint32_t dims_mask, int in_type, int map, int op, int has_init, double init,
                            double* out);
int orc_reduce_dims_int_s(const void* x, int ndim, const int64_t* shape, const int64_t* strides,
                          uint32_t dims_mask, int in_type, int acc_bits, int map, int op, int has_init,
                          int64_t init, int64_t* out);
int orc_reduce_dims_mat2_s(const uint32_t* x, int ndim, const int64_t* shape, const int64_t* strides,
                           uint32_t dims_mask, const uint32_t* init, uint32_t* out);

/* --- inclusive scan, whole array (dim = -1) or along dimension dim -------- */
int orc_scan_float(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int op,
                   int has_init, double init, double* y);
int orc_scan_int(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int acc_bits,
                 int op, int has_init, int64_t init, int64_t* y);
int orc_scan_mat2(const uint32_t* x, int ndim, const int64_t* shape, int dim,
                  const uint32_t* init, uint32_t* y);

/* --- exclusive scan: y_1 = init, y_i = op(y_{i-1}, x_{i-1}) (init required:
 *     the first output is the empty prefix). The pages describe inclusive
 *     scans only; this is the plain exclusive counterpart, with init as the
 *     first output of every line. ------------------------------------------ */
int orc_scan_excl_float(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int op,
                        double init, double* y);
int orc_scan_excl_int(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int acc_bits,
                      int op, int64_t init, int64_t* y);
int orc_scan_excl_mat2(const uint32_t* x, int ndim, const int64_t* shape, int dim, const uint32_t* init,
                       uint32_t* y);

/* --- findall (tile-scan PR #202, ratio table and tests paragraph): the
 *     0-based indices of the elements that are not zero, in increasing
 *     order; returns their count (-1: bad argument). in_type: ORC_U8 (Bool
 *     flags), ORC_I32, ORC_I64, ORC_F32, ORC_F64. ----------------------- */
int64_t orc_findall(const void* x, int64_t n, int in_type, int64_t* idx);

/* --- fused two-source reduce ("Finish whole-array reductions on the
 *     device", section "What changes": a single-output reduction of a
 *     Broadcasted source): r = op(init?, f(x_1, y_1), ..., f(x_n, y_n)) with
 *     f one of ORC_MAP2_*, computed like orc_reduce_*. --------------------- */
int orc_reduce2_float(const void* x, const void* y, int64_t n, int in_type, int map2, int op,
                      int has_init, double init, double* out);
int orc_reduce2_int(const void* x, const void* y, int64_t n, int in_type, int acc_bits, int map2, int op,
                    int has_init, int64_t init, int64_t* out);

/* --- affine maps mod p (the user-defined operator of the C++ template API's
 *     tests): element (a, b) = the map v -> a*v + b mod p; op(f, g) applies f
 *     then g = (a_g*a_f, a_g*b_f + b_g) mod p. ------------------------------ */
void orc_affine_compose(const uint32_t f[2], const uint32_t g[2], uint32_t out[2]);
int orc_scan_affine(const uint32_t* x, int64_t n, const uint32_t* init /* nullable */, int exclusive,
                    uint32_t* y);
int orc_reduce_affine(const uint32_t* x, int64_t n, const uint32_t* init /* nullable */, uint32_t out[2]);

#ifdef __cplusplus
}
#endif
#endif
