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
 *               whole array or along one dimension.
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

enum { ORC_F32 = 0, ORC_F64 = 1, ORC_BF16 = 2, ORC_I32 = 3, ORC_I64 = 4, ORC_MAT2 = 5 };
enum { ORC_MAP_IDENTITY = 0, ORC_MAP_ABS = 1, ORC_MAP_ABS2 = 2 };
enum { ORC_OP_ADD = 0, ORC_OP_MUL = 1, ORC_OP_MAX = 2, ORC_OP_MIN = 3, ORC_OP_MATMUL = 4 };

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

/* --- inclusive scan, whole array (dim = -1) or along dimension dim -------- */
int orc_scan_float(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int op,
                   int has_init, double init, double* y);
int orc_scan_int(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int acc_bits,
                 int op, int has_init, int64_t init, int64_t* y);
int orc_scan_mat2(const uint32_t* x, int ndim, const int64_t* shape, int dim,
                  const uint32_t* init, uint32_t* y);

#ifdef __cplusplus
}
#endif
#endif
