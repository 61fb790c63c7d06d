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

static int make_plan(dims_plan* p, int ndim, const int64_t* shape, uint32_t mask) {
    if (ndim < 1 || ndim > 16) return -1;
    p->ndim = ndim;
    p->nkept = p->nred = 0;
    p->nout = p->nfold = 1;
    int64_t st = 1;
    for (int d = 0; d < ndim; ++d) {
        if (shape[d] < 0) return -1;
        p->shape[d] = shape[d];
        p->stride[d] = st;
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
    dims_plan p;
    if (make_plan(&p, ndim, shape, mask) || !valid_float_args(in_type, map, op)) return -1;
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
    dims_plan p;
    if (make_plan(&p, ndim, shape, mask) || !valid_int_args(in_type, acc_bits, map, op)) return -1;
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
    dims_plan p;
    if (make_plan(&p, ndim, shape, mask)) return -1;
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
