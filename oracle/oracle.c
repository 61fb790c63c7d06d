/*
 * oracle.c -- plain sequential CPU oracle (test infrastructure only; see
 * oracle.h for what it computes, the passages it follows and who may call it).
 *
 * Everything here is a left-to-right loop over the elements. Nothing is
 * blocked, reordered or parallelised: a reader can check each function
 * against its definition by eye.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element access                                                            */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_float(const void* x, int in_type, int64_t i) {
    switch (in_type) {
    case ORC_F32: return (double)((const float*)x)[i];
    case ORC_F64: return ((const double*)x)[i];
    case ORC_BF16: return bf16_to_double(((const uint16_t*)x)[i]);
    default: return NAN;
    }
}

static int64_t load_int(const void* x, int in_type, int64_t i) {
    return in_type == ORC_I32 ? (int64_t)((const int32_t*)x)[i] : ((const int64_t*)x)[i];
}

static int is_float_type(int t) { return t == ORC_F32 || t == ORC_F64 || t == ORC_BF16; }
static int is_int_type(int t) { return t == ORC_I32 || t == ORC_I64; }

/* ------------------------------------------------------------------------ */
/* scalar helpers                                                            */
/* ------------------------------------------------------------------------ */

/* Round v to the nearest bf16 (8 significant bits, f32 exponent range),
 * ties to even, in a single rounding: scale so the rounding position is the
 * units place, round with nearbyint (the default mode is to-nearest-even and
 * the scaled value is exact), scale back. The result is exact in f32, whose
 * top 16 bits are the bf16 pattern. */
uint16_t orc_bf16_rne(double v) {
    if (isnan(v)) return 0x7fc0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    if (isinf(v)) return signbit(v) ? 0xff80 : 0x7f80;
    int e;
    frexp(v, &e);                /* |v| = m * 2^e, m in [0.5, 1) */
    int lsb = e - 8;             /* 8 significant bits: ulp = 2^(e-8) */
    if (lsb < -133) lsb = -133;  /* bf16 subnormal spacing 2^-133 */
    double r = nearbyint(ldexp(v, -lsb));
    double q = ldexp(r, lsb);
    if (fabs(q) >= 0x1p128) return signbit(v) ? 0xff80 : 0x7f80;
    float f = (float)q;          /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

double orc_fmax(double a, double b) {
    if (isnan(a) || isnan(b)) return NAN;
    if (a > b) return a;
    if (b > a) return b;
    return signbit(a) ? b : a; /* equal: only +0 / -0 differ; prefer +0 */
}

double orc_fmin(double a, double b) {
    if (isnan(a) || isnan(b)) return NAN;
    if (a < b) return a;
    if (b < a) return b;
    return signbit(a) ? a : b; /* equal: prefer -0 */
}

/* Product of two column-major 2x2 matrices modulo p. Entries are < p < 2^31,
 * so each product is < 2^62 and the sum of two is < 2^63. */
void orc_mat2_mul(const uint32_t a[4], const uint32_t b[4], uint32_t c[4]) {
    const uint64_t p = ORC_MODP;
    uint64_t a11 = a[0], a21 = a[1], a12 = a[2], a22 = a[3];
    uint64_t b11 = b[0], b21 = b[1], b12 = b[2], b22 = b[3];
    c[0] = (uint32_t)((a11 * b11 + a12 * b21) % p);
    c[1] = (uint32_t)((a21 * b11 + a22 * b21) % p);
    c[2] = (uint32_t)((a11 * b12 + a12 * b22) % p);
    c[3] = (uint32_t)((a21 * b12 + a22 * b22) % p);
}

/* ------------------------------------------------------------------------ */
/* float fold: f64 with a Neumaier-compensated running sum                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    double s; /* running value */
    double c; /* compensation of the running sum (op = add only) */
} ffold;

static double fmap(double v, int map) {
    switch (map) {
    case ORC_MAP_ABS: return fabs(v);
    case ORC_MAP_ABS2: return v * v;
    default: return v;
    }
}

static void ffold_start(ffold* a, double v) { a->s = v; a->c = 0.0; }

static void ffold_step(ffold* a, double v, int op) {
    switch (op) {
    case ORC_OP_ADD: {
        double t = a->s + v;
        if (isfinite(t)) {
            if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;
            else a->c += (v - t) + a->s;
        }
        a->s = t;
        break;
    }
    case ORC_OP_MUL: a->s = a->s * v; break;
    case ORC_OP_MAX: a->s = orc_fmax(a->s, v); break;
    case ORC_OP_MIN: a->s = orc_fmin(a->s, v); break;
    }
}

/* The compensated value; with no compensation the running value itself, so
 * a fold of negative zeros stays -0.0 (s + 0.0 would turn it into +0.0). */
static double ffold_value(const ffold* a) { return (isfinite(a->s) && a->c != 0.0) ? a->s + a->c : a->s; }

/* ------------------------------------------------------------------------ */
/* integer fold: exact, wrapped to 32 or 64 bits                           */
/* ------------------------------------------------------------------------ */

static int64_t wrap(uint64_t v, int bits) {
    if (bits == 64) {
        int64_t r;
        memcpy(&r, &v, sizeof r);
        return r;
    }
    uint32_t u = (uint32_t)v;
    return u >= 0x80000000u ? (int64_t)u - 0x100000000LL : (int64_t)u;
}

static int64_t imap(int64_t v, int map, int bits) {
    uint64_t u = (uint64_t)v;
    switch (map) {
    case ORC_MAP_ABS: return wrap(v < 0 ? (uint64_t)0 - u : u, bits);
    case ORC_MAP_ABS2: return wrap(u * u, bits);
    default: return wrap(u, bits);
    }
}

static int64_t istep(int64_t a, int64_t v, int op, int bits) {
    switch (op) {
    case ORC_OP_ADD: return wrap((uint64_t)a + (uint64_t)v, bits);
    case ORC_OP_MUL: return wrap((uint64_t)a * (uint64_t)v, bits);
    case ORC_OP_MAX: return a > v ? a : v;
    case ORC_OP_MIN: return a < v ? a : v;
    default: return a;
    }
}

static int valid_float_args(int in_type, int map, int op) {
    return is_float_type(in_type) && map >= ORC_MAP_IDENTITY && map <= ORC_MAP_ABS2 &&
           op >= ORC_OP_ADD && op <= ORC_OP_MIN;
}

static int valid_int_args(int in_type, int acc_bits, int map, int op) {
    if (!is_int_type(in_type)) return 0;
    if (acc_bits != 32 && acc_bits != 64) return 0;
    if (in_type == ORC_I64 && acc_bits == 32) return 0;
    return map >= ORC_MAP_IDENTITY && map <= ORC_MAP_ABS2 && op >= ORC_OP_ADD && op <= ORC_OP_MIN;
}

/* ------------------------------------------------------------------------ */
/* whole-array reduce                                                        */
/* ------------------------------------------------------------------------ */

int orc_reduce_float(const void* x, int64_t n, int in_type, int map, int op,
                     int has_init, double init, double* out) {
    if (!valid_float_args(in_type, map, op) || n < 0) return -1;
    ffold a;
    int64_t i = 0;
    if (has_init) ffold_start(&a, init);
    else if (n > 0) ffold_start(&a, fmap(load_float(x, in_type, i++), map));
    else return 1;
    for (; i < n; ++i) ffold_step(&a, fmap(load_float(x, in_type, i), map), op);
    *out = ffold_value(&a);
    return 0;
}

int orc_reduce_int(const void* x, int64_t n, int in_type, int acc_bits, int map, int op,
                   int has_init, int64_t init, int64_t* out) {
    if (!valid_int_args(in_type, acc_bits, map, op) || n < 0) return -1;
    int64_t a;
    int64_t i = 0;
    if (has_init) a = wrap((uint64_t)init, acc_bits);
    else if (n > 0) a = imap(load_int(x, in_type, i++), map, acc_bits);
    else return 1;
    for (; i < n; ++i) a = istep(a, imap(load_int(x, in_type, i), map, acc_bits), op, acc_bits);
    *out = a;
    return 0;
}

int orc_reduce_mat2(const uint32_t* x, int64_t n, const uint32_t* init, uint32_t out[4]) {
    if (n < 0) return -1;
    uint32_t a[4], t[4];
    int64_t i = 0;
    if (init) memcpy(a, init, sizeof a);
    else if (n > 0) memcpy(a, x + 4 * i++, sizeof a);
    else return 1;
    for (; i < n; ++i) {
        orc_mat2_mul(a, x + 4 * i, t);
        memcpy(a, t, sizeof a);
    }
    memcpy(out, a, sizeof a);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* reduce over a set of dimensions                                           */
/* ------------------------------------------------------------------------ */

/* Index bookkeeping for a column-major array: the kept dimensions define the
 * output index, the reduced dimensions the position along the fold. */
typedef struct {
    int ndim;
    int64_t shape[16];
    int64_t stride[16]; /* column-major element strides */
    int nkept, nred;
    int kept[16], red[16];
    int64_t nout, nfold;
} dims_plan;

/* strides: element strides of the source per dimension (a strided view), or
 * NULL for the dense column-major layout. */
static int make_plan(dims_plan* p, int ndim, const int64_t* shape, const int64_t* strides, uint32_t mask) {
    if (ndim < 1 || ndim > 16) return -1;
    p->ndim = ndim;
    p->nkept = p->nred = 0;
    p->nout = p->nfold = 1;
    int64_t st = 1;
    for (int d = 0; d < ndim; ++d) {
        if (shape[d] < 0) return -1;
        p->shape[d] = shape[d];
        p->stride[d] = strides ? strides[d] : st;
        st *= shape[d];
        if (mask & (1u << d)) { p->red[p->nred++] = d; p->nfold *= shape[d]; }
        else { p->kept[p->nkept++] = d; p->nout *= shape[d]; }
    }
    if (mask >> ndim) return -1;
    return 0;
}

/* Offset of the o-th combination (column-major) of the listed dimensions. */
static int64_t offset_of(const dims_plan* p, const int* dims, int nd, int64_t o) {
    int64_t off = 0;
    for (int k = 0; k < nd; ++k) {
        int d = dims[k];
        off += (o % p->shape[d]) * p->stride[d];
        o /= p->shape[d];
    }
    return off;
}

int orc_reduce_dims_float(const void* x, int ndim, const int64_t* shape, uint32_t mask,
                          int in_type, int map, int op, int has_init, double init, double* out) {
    return orc_reduce_dims_float_s(x, ndim, shape, NULL, mask, in_type, map, op, has_init, init, out);
}

int orc_reduce_dims_float_s(const void* x, int ndim, const int64_t* shape, const int64_t* strides,
                            uint32_t mask, int in_type, int map, int op, int has_init, double init,
                            double* out) {
    dims_plan p;
    if (make_plan(&p, ndim, shape, strides, mask) || !valid_float_args(in_type, map, op)) return -1;
    if (p.nfold == 0 && !has_init) return 1;
    for (int64_t o = 0; o < p.nout; ++o) {
        int64_t base = offset_of(&p, p.kept, p.nkept, o);
        ffold a;
        int64_t r = 0;
        if (has_init) ffold_start(&a, init);
        else ffold_start(&a, fmap(load_float(x, in_type, base + offset_of(&p, p.red, p.nred, r++)), map));
        for (; r < p.nfold; ++r)
            ffold_step(&a, fmap(load_float(x, in_type, base + offset_of(&p, p.red, p.nred, r)), map), op);
        out[o] = ffold_value(&a);
    }
    return 0;
}

int orc_reduce_dims_int(const void* x, int ndim, const int64_t* shape, uint32_t mask,
                        int in_type, int acc_bits, int map, int op, int has_init, int64_t init,
                        int64_t* out) {
    return orc_reduce_dims_int_s(x, ndim, shape, NULL, mask, in_type, acc_bits, map, op, has_init, init, out);
}

int orc_reduce_dims_int_s(const void* x, int ndim, const int64_t* shape, const int64_t* strides,
                          uint32_t mask, int in_type, int acc_bits, int map, int op, int has_init,
                          int64_t init, int64_t* out) {
    dims_plan p;
    if (make_plan(&p, ndim, shape, strides, mask) || !valid_int_args(in_type, acc_bits, map, op)) return -1;
    if (p.nfold == 0 && !has_init) return 1;
    for (int64_t o = 0; o < p.nout; ++o) {
        int64_t base = offset_of(&p, p.kept, p.nkept, o);
        int64_t a;
        int64_t r = 0;
        if (has_init) a = wrap((uint64_t)init, acc_bits);
        else a = imap(load_int(x, in_type, base + offset_of(&p, p.red, p.nred, r++)), map, acc_bits);
        for (; r < p.nfold; ++r)
            a = istep(a, imap(load_int(x, in_type, base + offset_of(&p, p.red, p.nred, r)), map, acc_bits),
                      op, acc_bits);
        out[o] = a;
    }
    return 0;
}

int orc_reduce_dims_mat2(const uint32_t* x, int ndim, const int64_t* shape, uint32_t mask,
                         const uint32_t* init, uint32_t* out) {
    return orc_reduce_dims_mat2_s(x, ndim, shape, NULL, mask, init, out);
}

int orc_reduce_dims_mat2_s(const uint32_t* x, int ndim, const int64_t* shape, const int64_t* strides,
                           uint32_t mask, const uint32_t* init, uint32_t* out) {
    dims_plan p;
    if (make_plan(&p, ndim, shape, strides, mask)) return -1;
    if (p.nfold == 0 && !init) return 1;
    for (int64_t o = 0; o < p.nout; ++o) {
        int64_t base = offset_of(&p, p.kept, p.nkept, o);
        uint32_t a[4], t[4];
        int64_t r = 0;
        if (init) memcpy(a, init, sizeof a);
        else memcpy(a, x + 4 * (base + offset_of(&p, p.red, p.nred, r++)), sizeof a);
        for (; r < p.nfold; ++r) {
            orc_mat2_mul(a, x + 4 * (base + offset_of(&p, p.red, p.nred, r)), t);
            memcpy(a, t, sizeof a);
        }
        memcpy(out + 4 * o, a, sizeof a);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* inclusive scans                                                           */
/* ------------------------------------------------------------------------ */

/* Lines of a scan: dim = -1 is the whole array as one line; otherwise every
 * index tuple whose dim-th index is 0 starts a line of shape[dim] elements
 * spaced stride[dim] apart. */
typedef struct {
    int64_t n, len, step;
    int64_t stride_dim, extent_dim;
} scan_lines;

static int make_lines(scan_lines* s, int ndim, const int64_t* shape, int dim) {
    if (ndim < 1 || ndim > 16 || dim < -1 || dim >= ndim) return -1;
    int64_t n = 1, st = 1, st_dim = 1;
    for (int d = 0; d < ndim; ++d) {
        if (shape[d] < 0) return -1;
        if (d == dim) st_dim = st;
        st *= shape[d];
        n *= shape[d];
    }
    s->n = n;
    if (dim < 0) { s->len = n; s->step = 1; s->stride_dim = 1; s->extent_dim = n; }
    else { s->len = shape[dim]; s->step = st_dim; s->stride_dim = st_dim; s->extent_dim = shape[dim]; }
    return 0;
}

static int is_line_start(const scan_lines* s, int64_t e) {
    return s->extent_dim == 0 || (e / s->stride_dim) % s->extent_dim == 0;
}

int orc_scan_float(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int op,
                   int has_init, double init, double* y) {
    scan_lines s;
    if (make_lines(&s, ndim, shape, dim) || !valid_float_args(in_type, ORC_MAP_IDENTITY, op)) return -1;
    if (s.len == 0) return 0;
    for (int64_t e = 0; e < s.n; ++e) {
        if (!is_line_start(&s, e)) continue;
        ffold a;
        if (has_init) {
            ffold_start(&a, init);
            ffold_step(&a, load_float(x, in_type, e), op);
        } else {
            ffold_start(&a, load_float(x, in_type, e));
        }
        y[e] = ffold_value(&a);
        for (int64_t j = 1; j < s.len; ++j) {
            int64_t k = e + j * s.step;
            ffold_step(&a, load_float(x, in_type, k), op);
            y[k] = ffold_value(&a);
        }
    }
    return 0;
}

int orc_scan_int(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int acc_bits,
                 int op, int has_init, int64_t init, int64_t* y) {
    scan_lines s;
    if (make_lines(&s, ndim, shape, dim) || !valid_int_args(in_type, acc_bits, ORC_MAP_IDENTITY, op))
        return -1;
    if (s.len == 0) return 0;
    for (int64_t e = 0; e < s.n; ++e) {
        if (!is_line_start(&s, e)) continue;
        int64_t v = wrap((uint64_t)load_int(x, in_type, e), acc_bits);
        int64_t a = has_init ? istep(wrap((uint64_t)init, acc_bits), v, op, acc_bits) : v;
        y[e] = a;
        for (int64_t j = 1; j < s.len; ++j) {
            int64_t k = e + j * s.step;
            a = istep(a, wrap((uint64_t)load_int(x, in_type, k), acc_bits), op, acc_bits);
            y[k] = a;
        }
    }
    return 0;
}

int orc_scan_mat2(const uint32_t* x, int ndim, const int64_t* shape, int dim,
                  const uint32_t* init, uint32_t* y) {
    scan_lines s;
    if (make_lines(&s, ndim, shape, dim)) return -1;
    if (s.len == 0) return 0;
    for (int64_t e = 0; e < s.n; ++e) {
        if (!is_line_start(&s, e)) continue;
        uint32_t a[4], t[4];
        if (init) orc_mat2_mul(init, x + 4 * e, a);
        else memcpy(a, x + 4 * e, sizeof a);
        memcpy(y + 4 * e, a, sizeof a);
        for (int64_t j = 1; j < s.len; ++j) {
            int64_t k = e + j * s.step;
            orc_mat2_mul(a, x + 4 * k, t);
            memcpy(a, t, sizeof a);
            memcpy(y + 4 * k, a, sizeof a);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* exclusive scans                                                           */
/* ------------------------------------------------------------------------ */

/* Exclusive scan along each line: y_1 = init, y_i = op(y_{i-1}, x_{i-1}),
 * i.e. element i holds the fold of init and every element before it. init
 * is required: the first output is the empty prefix, which has a value only
 * through init. */
int orc_scan_excl_float(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int op,
                        double init, double* y) {
    scan_lines s;
    if (make_lines(&s, ndim, shape, dim) || !valid_float_args(in_type, ORC_MAP_IDENTITY, op)) return -1;
    if (s.len == 0) return 0;
    for (int64_t e = 0; e < s.n; ++e) {
        if (!is_line_start(&s, e)) continue;
        ffold a;
        ffold_start(&a, init);
        for (int64_t j = 0; j < s.len; ++j) {
            int64_t k = e + j * s.step;
            y[k] = ffold_value(&a);
            ffold_step(&a, load_float(x, in_type, k), op);
        }
    }
    return 0;
}

int orc_scan_excl_int(const void* x, int ndim, const int64_t* shape, int dim, int in_type, int acc_bits,
                      int op, int64_t init, int64_t* y) {
    scan_lines s;
    if (make_lines(&s, ndim, shape, dim) || !valid_int_args(in_type, acc_bits, ORC_MAP_IDENTITY, op))
        return -1;
    if (s.len == 0) return 0;
    for (int64_t e = 0; e < s.n; ++e) {
        if (!is_line_start(&s, e)) continue;
        int64_t a = wrap((uint64_t)init, acc_bits);
        for (int64_t j = 0; j < s.len; ++j) {
            int64_t k = e + j * s.step;
            y[k] = a;
            a = istep(a, wrap((uint64_t)load_int(x, in_type, k), acc_bits), op, acc_bits);
        }
    }
    return 0;
}

int orc_scan_excl_mat2(const uint32_t* x, int ndim, const int64_t* shape, int dim, const uint32_t* init,
                       uint32_t* y) {
    scan_lines s;
    if (make_lines(&s, ndim, shape, dim) || !init) return -1;
    if (s.len == 0) return 0;
    for (int64_t e = 0; e < s.n; ++e) {
        if (!is_line_start(&s, e)) continue;
        uint32_t a[4], t[4];
        memcpy(a, init, sizeof a);
        for (int64_t j = 0; j < s.len; ++j) {
            int64_t k = e + j * s.step;
            memcpy(y + 4 * k, a, sizeof a);
            orc_mat2_mul(a, x + 4 * k, t);
            memcpy(a, t, sizeof a);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* findall                                                                   */
/* ------------------------------------------------------------------------ */

/* Indices (0-based, increasing) of the elements that are not zero; returns
 * their count. Bytes (Bool flags) and integers compare with 0; floats with
 * 0.0, so -0.0 counts as zero and NaN as not zero. */
int64_t orc_findall(const void* x, int64_t n, int in_type, int64_t* idx) {
    if (n < 0) return -1;
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i) {
        int set;
        switch (in_type) {
        case ORC_U8: set = ((const uint8_t*)x)[i] != 0; break;
        case ORC_I32: set = ((const int32_t*)x)[i] != 0; break;
        case ORC_I64: set = ((const int64_t*)x)[i] != 0; break;
        case ORC_F32: set = ((const float*)x)[i] != 0.0f; break;
        case ORC_F64: set = ((const double*)x)[i] != 0.0; break;
        default: return -1;
        }
        if (set) idx[c++] = i;
    }
    return c;
}

/* ------------------------------------------------------------------------ */
/* fused two-source reductions: r = op(init, f(x_1, y_1), ..., f(x_n, y_n)) */
/* ------------------------------------------------------------------------ */

static double fmap2(double a, double b, int map2) {
    switch (map2) {
    case ORC_MAP2_MUL: return a * b;
    case ORC_MAP2_SQDIFF: return (a - b) * (a - b);
    case ORC_MAP2_ABSDIFF: return fabs(a - b);
    default: return NAN;
    }
}

static int64_t imap2(int64_t a, int64_t b, int map2, int bits) {
    uint64_t d = (uint64_t)a - (uint64_t)b;
    switch (map2) {
    case ORC_MAP2_MUL: return wrap((uint64_t)a * (uint64_t)b, bits);
    case ORC_MAP2_SQDIFF: return wrap(wrap(d, bits) * (uint64_t)wrap(d, bits), bits);
    case ORC_MAP2_ABSDIFF: {
        int64_t w = wrap(d, bits);
        return wrap(w < 0 ? (uint64_t)0 - (uint64_t)w : (uint64_t)w, bits);
    }
    default: return 0;
    }
}

int orc_reduce2_float(const void* x, const void* y, int64_t n, int in_type, int map2, int op,
                      int has_init, double init, double* out) {
    if (!valid_float_args(in_type, ORC_MAP_IDENTITY, op) || map2 < ORC_MAP2_MUL || map2 > ORC_MAP2_ABSDIFF ||
        n < 0)
        return -1;
    ffold a;
    int64_t i = 0;
    if (has_init) ffold_start(&a, init);
    else if (n > 0) {
        ffold_start(&a, fmap2(load_float(x, in_type, 0), load_float(y, in_type, 0), map2));
        i = 1;
    } else return 1;
    for (; i < n; ++i) ffold_step(&a, fmap2(load_float(x, in_type, i), load_float(y, in_type, i), map2), op);
    *out = ffold_value(&a);
    return 0;
}

int orc_reduce2_int(const void* x, const void* y, int64_t n, int in_type, int acc_bits, int map2, int op,
                    int has_init, int64_t init, int64_t* out) {
    if (!valid_int_args(in_type, acc_bits, ORC_MAP_IDENTITY, op) || map2 < ORC_MAP2_MUL ||
        map2 > ORC_MAP2_ABSDIFF || n < 0)
        return -1;
    int64_t a;
    int64_t i = 0;
    if (has_init) a = wrap((uint64_t)init, acc_bits);
    else if (n > 0) {
        a = imap2(wrap((uint64_t)load_int(x, in_type, 0), acc_bits), wrap((uint64_t)load_int(y, in_type, 0), acc_bits),
                  map2, acc_bits);
        i = 1;
    } else return 1;
    for (; i < n; ++i)
        a = istep(a, imap2(wrap((uint64_t)load_int(x, in_type, i), acc_bits),
                           wrap((uint64_t)load_int(y, in_type, i), acc_bits), map2, acc_bits), op, acc_bits);
    *out = a;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* affine maps mod p: the user-defined operator of the template API's tests  */
/* ------------------------------------------------------------------------ */

/* An element (a, b) is the map v -> a*v + b mod p, entries in [0, p). The
 * operator composes left to right: op(f, g) applies f first, then g:
 * g(f(v)) = a_g*(a_f*v + b_f) + b_g, i.e. (a_g*a_f, a_g*b_f + b_g). It is
 * associative, not commutative, and (1, 0) is its identity. */
void orc_affine_compose(const uint32_t f[2], const uint32_t g[2], uint32_t out[2]) {
    const uint64_t p = ORC_MODP;
    uint64_t a = ((uint64_t)g[0] * f[0]) % p;
    uint64_t b = ((uint64_t)g[0] * f[1] + g[1]) % p;
    out[0] = (uint32_t)a;
    out[1] = (uint32_t)b;
}

/* Inclusive (exclusive = 0) or exclusive scan of n affine maps with an
 * optional init on the left (required for the exclusive scan). */
int orc_scan_affine(const uint32_t* x, int64_t n, const uint32_t* init, int exclusive, uint32_t* y) {
    if (n < 0 || (exclusive && !init)) return -1;
    uint32_t a[2], t[2];
    int64_t i = 0;
    if (init) memcpy(a, init, sizeof a);
    else if (n > 0) {
        memcpy(a, x, sizeof a);
        memcpy(y, a, sizeof a);
        i = 1;
    }
    for (; i < n; ++i) {
        if (exclusive) memcpy(y + 2 * i, a, sizeof a);
        orc_affine_compose(a, x + 2 * i, t);
        memcpy(a, t, sizeof a);
        if (!exclusive) memcpy(y + 2 * i, a, sizeof a);
    }
    return 0;
}

int orc_reduce_affine(const uint32_t* x, int64_t n, const uint32_t* init, uint32_t out[2]) {
    if (n < 0) return -1;
    uint32_t a[2], t[2];
    int64_t i = 0;
    if (init) memcpy(a, init, sizeof a);
    else if (n > 0) memcpy(a, x + 2 * i++, sizeof a);
    else return 1;
    for (; i < n; ++i) {
        orc_affine_compose(a, x + 2 * i, t);
        memcpy(a, t, sizeof a);
    }
    memcpy(out, a, sizeof a);
    return 0;
}
