/*
 * ak.h -- C ABI of the GB300 (sm_103a) device-wide reduce / prefix-scan library.
 *
 * Three operations, as stated in the AcceleratedKernels.jl pull requests
 * this library re-designs for GB300:
 *
 *   ak_reduce       whole-array mapreduce(f, op, A) into a host scalar or a
 *                   one-element device array ("Finish whole-array reductions
 *                   on the device", PR #139, sections "What changes" and
 *                   "Compatibility");
 *   ak_reduce_dims  mapreducedim!(f, op, R, A) over a set of dimensions of a
 *                   dense column-major array, e.g. sum(x; dims=2) of a matrix
 *                   or of the middle dimension of a 3-d array (strided
 *                   reduction PR #176, first two lists);
 *   ak_accumulate   accumulate!(op, dst, src) / cumsum: the inclusive scan of
 *                   the whole array or along one dimension, including
 *                   operators with no neutral element and non-commutative
 *                   ones (tile-scan PR #202, first paragraph and paragraph
 *                   "Alternatives").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers. Arrays (src, dst, workspace) are DEVICE pointers to memory of the
 *   current CUDA device; init and dst_host are HOST pointers. The caller owns
 *   every buffer; the library allocates no device memory.
 * Layout. Arrays are dense and column-major: element (i1, i2, ..., id) of a
 *   shape (n1, ..., nd) sits at i1 + n1*(i2 + n2*(i3 + ...)) (0-based). This
 *   is the memory of a contiguous row-major tensor of the reversed shape.
 *   Dimensions are numbered from 0 (Julia's dims=2 is dimension 1 here).
 * Element types (ak_dtype). AK_BF16 is the bfloat16 bit pattern; AK_MAT2_MODP
 *   is a 2x2 matrix over Z/pZ, p = 2^31 - 1, stored as four uint32 entries in
 *   column-major order (a11, a21, a12, a22), each in [0, p); its only operator
 *   is AK_OP_MATMUL_MODP, the product mod p, with the left operand first.
 * Types of a call. `in` is the element type of src; `acc` the accumulator in
 *   which f is applied and op folds; `out` the type stored. Supported
 *   (in -> acc -> out): F32->F32->F32, F32->F64->{F64,F32}, F64->F64->F64,
 *   BF16->F32->{BF16,F32}, I32->I32->I32, I32->I64->I64, I64->I64->I64,
 *   MAT2->MAT2->MAT2. f32 -> bf16 and f64 -> f32 stores round to nearest
 *   even; integer accumulators wrap modulo 2^32 / 2^64.
 * Order. Results equal the left-to-right fold up to the rounding of a
 *   different association tree; non-commutative operators keep the element
 *   order exactly. max / min follow Julia: NaN wins (returned as the
 *   canonical quiet NaN) and +0.0 > -0.0.
 * init. A host pointer to ONE value of the accumulator type, applied exactly
 *   once, leftmost: op(init, ...).
 * Asynchrony. Calls enqueue work on `stream` (a cudaStream_t, NULL = legacy
 *   default stream) and return without waiting, except where stated. Calls
 *   that share a workspace must be ordered on one stream.
 * Workspace. A device buffer of at least the size the matching
 *   *_workspace_size function reports for the same arguments (16-byte
 *   aligned). Its contents on entry are arbitrary: no clearing is needed
 *   between calls.
 * Errors. Every call returns an ak_status. Arguments are validated before
 *   anything is launched, so invalid calls have no effect on the device.
 *   AK_ERR_CUDA keeps the CUDA error, readable with ak_last_cuda_error().
 * Logging. With AK_LOG set in the environment (and not "0"), every call
 *   prints one line to stderr naming the path it takes: the first-pass grid
 *   of a reduction, the dims kernel with its shape, tile and split, the
 *   scan kernel with its tile count, findall's tile count. The variable is
 *   read on every call.
 */
#ifndef AK_H
#define AK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ak_status {
    AK_OK = 0,
    AK_ERR_INVALID_ARG = 1,   /* bad pointer, size, enum, dims or store mode */
    AK_ERR_UNSUPPORTED = 2,   /* valid but unsupported type / op / map combination */
    AK_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned */
    AK_ERR_EMPTY_NO_INIT = 4, /* empty reduction, no init and no neutral element */
    AK_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    AK_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out (scan look-back) */
} ak_status;

typedef enum ak_dtype {
    AK_F32 = 0,
    AK_F64 = 1,
    AK_BF16 = 2,
    AK_I32 = 3,
    AK_I64 = 4,
    AK_MAT2_MODP = 5,
    AK_U8 = 6  /* bytes (Julia Bool flags): findall input only */
} ak_dtype;

/* f, applied to each element in the accumulator type before op. */
typedef enum ak_map { AK_MAP_IDENTITY = 0, AK_MAP_ABS = 1, AK_MAP_ABS2 = 2 } ak_map;

/* f of a fused two-source element (ak_reduce2), in the accumulator type:
 * a*b, (a-b)^2, |a-b| (integers wrap). */
typedef enum ak_map2 { AK_MAP2_MUL = 0, AK_MAP2_SQDIFF = 1, AK_MAP2_ABSDIFF = 2 } ak_map2;

typedef enum ak_op {
    AK_OP_ADD = 0,
    AK_OP_MUL = 1,
    AK_OP_MAX = 2,
    AK_OP_MIN = 3,
    AK_OP_MATMUL_MODP = 4
} ak_op;

/* How a reduction's result r is stored into R (PR #139, "What changes": the
 * last pass applies init, folds into R's previous value, or writes):
 *   AK_STORE_OVERWRITE  R = r
 *   AK_STORE_INIT       R = op(init, r)    (init required)
 *   AK_STORE_FOLD       R = op(R_old, r)   (R_old converted to acc first) */
typedef enum ak_store { AK_STORE_OVERWRITE = 0, AK_STORE_INIT = 1, AK_STORE_FOLD = 2 } ak_store;

/* Kernel shape of a strided dims reduction (PR #176, item 1): one thread per
 * output, one pass over tiles of outputs, or tiles of outputs with the
 * reduction split across blocks and a second pass. AUTO chooses by the
 * number of outputs versus the reduction length. */
typedef enum ak_dims_shape {
    AK_SHAPE_AUTO = 0,
    AK_SHAPE_THREAD = 1,
    AK_SHAPE_TILED = 2,
    AK_SHAPE_COLUMNS = 3
} ak_dims_shape;

/* Options; pass NULL for defaults or fill with ak_opts_default(). */
typedef struct ak_opts {
    int32_t no_neutral;       /* 1: treat op as having no neutral element; partial results
                                 carry an Optional flag (e.g. 8 bytes for a Float32 acc) */
    int32_t target_blocks;    /* whole-array first pass / persistent scan grid; 0 = auto */
    int32_t items_per_thread; /* scan run length / reduce loads in flight; 0 = auto */
    int32_t dims_shape;       /* ak_dims_shape */
    int32_t check;            /* 1: synchronize `stream` before returning and report
                                 device-side failures (AK_ERR_TIMEOUT) */
    int32_t flags;            /* tuning switches, AK_FLAG_* (0 = none) */
    int32_t exclusive;        /* ak_accumulate: 1 = exclusive scan (see ak_accumulate) */
    int32_t reserved;         /* must be 0 */
    int64_t wait_limit_ns;    /* bound of each device-side wait of the scan; 0 = 1 s. Without
                                 `check` a wait that runs out is not reported by the call
                                 itself: read it with ak_scan_status */
    int64_t debug_skip_publish_tile; /* fault injection for tests: the scan tile with this
                                 index never publishes its state, so its successors'
                                 bounded waits run out; -1 = off */
} ak_opts;

/* AK_FLAG_DIMS_CLUSTER: a strided dims reduction whose split fits 2..16
 * blocks runs each output tile's blocks as one thread-block cluster and
 * combines their partials in distributed shared memory (one kernel, no
 * workspace partials) instead of a workspace and a second pass, at any input
 * size. Without the flag the automatic shape does so only for inputs of at
 * most 16 MB, where saving the second launch pays on GB300; larger inputs
 * split through the workspace. */
#define AK_FLAG_DIMS_CLUSTER 1

void ak_opts_default(ak_opts* opts);

const char* ak_status_string(ak_status status);
/* Size in bytes of one element of the type; 0 for an invalid type. */
size_t ak_dtype_size(ak_dtype dtype);
/* The cudaError_t of the last AK_ERR_CUDA returned on this thread. */
int ak_last_cuda_error(void);
/* Number of kernels this library has launched in this process. */
uint64_t ak_kernel_launch_count(void);

/* ---------------------------------------------------------------------------
 * ak_reduce: r = op(f(src[0]), f(src[1]), ..., f(src[n-1])), then stored by
 * `mode` into a one-element device array and/or returned to the host.
 * PR #139, "What changes": a first pass of a bounded number of blocks, each
 * reducing its share of the input to one partial, and a one-block second
 * pass that reduces the partials and performs the store; a small input takes
 * one launch; for a host result the last pass stores the bare partial, which
 * is copied back and finished on the host.
 *
 *   src        device, n elements of `in` (n == 0 allowed)
 *   dst_dev    device, one element of `out`, or NULL
 *   dst_host   host, one element of `out`, or NULL; when given the call
 *              returns only once the result is there (with AK_STORE_FOLD,
 *              *dst_host holds R_old on entry, unless dst_dev is also
 *              given, in which case R is the device element). The last
 *              pass writes the bare partial straight into a small mapped,
 *              pinned host slot of the calling thread (64 bytes, allocated
 *              by its first host-result call and kept until the process
 *              exits), then the call's sequence number beside it after a
 *              system-scope fence. The host polls that word for about
 *              200 us, then synchronizes `stream` (which also reports any
 *              error on it), and finishes the partial. The call may thus
 *              return before the kernel has retired on the stream; later
 *              work on the stream is ordered after it as usual. An
 *              asynchronous error that strikes after the result landed
 *              surfaces on the next synchronizing call.
 *   At least one of dst_dev / dst_host must be non-NULL.
 * Empty input: AK_STORE_INIT stores init; AK_STORE_FOLD leaves R unchanged;
 *   AK_STORE_OVERWRITE stores the neutral element of op (0 for +, 1 for *,
 *   the identity matrix), or fails with AK_ERR_EMPTY_NO_INIT for max / min
 *   and under no_neutral.
 * ------------------------------------------------------------------------- */
ak_status ak_reduce_workspace_size(int64_t n, ak_dtype in, ak_dtype acc, const ak_opts* opts,
                                   size_t* bytes);
ak_status ak_reduce(const void* src, int64_t n, ak_dtype in, ak_map f, ak_op op, ak_dtype acc,
                    ak_dtype out, const void* init, ak_store mode, void* dst_dev, void* dst_host,
                    void* workspace, size_t workspace_bytes, const ak_opts* opts, void* stream);

/* ---------------------------------------------------------------------------
 * ak_reduce2: r = op(f(a[0], b[0]), ..., f(a[n-1], b[n-1])) over two sources
 * of n elements of `in` read side by side -- a fused (Broadcasted) source such
 * as sum(x .* y) or sum(abs2.(x .- y)), reduced without materialising the
 * elementwise array. PR #139, "What changes": a single-output reduction whose
 * source is a Broadcasted takes the whole-array path. Arguments, workspace
 * (ak_reduce_workspace_size with the same n, in, acc), store modes and empty
 * rules are ak_reduce's; f is an ak_map2; matrices are not supported. Sources
 * whose addresses differ by a multiple of 32 bytes are read with 32-byte
 * vectors, others element by element.
 * ------------------------------------------------------------------------- */
ak_status ak_reduce2(const void* src_a, const void* src_b, int64_t n, ak_dtype in, ak_map2 f, ak_op op,
                     ak_dtype acc, ak_dtype out, const void* init, ak_store mode, void* dst_dev,
                     void* dst_host, void* workspace, size_t workspace_bytes, const ak_opts* opts,
                     void* stream);

/* ---------------------------------------------------------------------------
 * ak_reduce_dims: R[kept index] = op over the reduced dimensions of
 * f(src[...]), folded in increasing column-major order of the reduced
 * indices. PR #176: strided reductions into contiguous outputs take a 2-d
 * block of outputs x reduction rows, split across blocks (plus a second
 * pass) only when the outputs alone do not fill the device; the middle
 * dimension of a 3-d array is handled as runs of contiguous outputs at the
 * offsets of the other kept dimensions. PR #139: a reduction to a single
 * output over one contiguous range takes the whole-array path; its tests
 * cover offset views, which strides describe here.
 *
 *   ndim, shape   1 <= ndim <= 8, column-major extents (>= 0)
 *   strides       element strides of src per dimension (>= 0): a strided
 *                 view (a sub-array, a transpose, a stepped slice); NULL =
 *                 dense column-major. Views whose kept innermost dimension
 *                 has unit stride take the strided / row kernels (16-byte
 *                 loads when src and the strides are 16-byte multiples);
 *                 others a general kernel (slower: it walks the reduced
 *                 indices per thread).
 *   dims_mask     bit d set = dimension d is reduced (bits >= ndim invalid)
 *   dst           device, DENSE column-major array of `out` with the shape
 *                 of src where reduced extents are 1
 * Empty reductions (a reduced extent is 0) follow ak_reduce's empty rules.
 * ------------------------------------------------------------------------- */
ak_status ak_reduce_dims_workspace_size(int ndim, const int64_t* shape, const int64_t* strides,
                                        uint32_t dims_mask, ak_dtype in, ak_dtype acc,
                                        const ak_opts* opts, size_t* bytes);
ak_status ak_reduce_dims(const void* src, int ndim, const int64_t* shape, const int64_t* strides,
                         uint32_t dims_mask, ak_dtype in, ak_map f, ak_op op, ak_dtype acc,
                         ak_dtype out, const void* init, ak_store mode, void* dst, void* workspace,
                         size_t workspace_bytes, const ak_opts* opts, void* stream);

/* ---------------------------------------------------------------------------
 * ak_accumulate: inclusive scan. Along a line x_1, x_2, ...:
 *   y_1 = op(init, x_1) (or x_1 without init), y_i = op(y_{i-1}, x_i).
 * dim = -1 scans the whole array as one line (column-major order); dim = d
 * scans every line along dimension d independently. PR #202, first
 * paragraph: a tile is loaded, each thread scans its own run of consecutive
 * elements, and the tile prefix is applied (runs of lines that fit one tile
 * sit at an odd stride in shared memory, as there; long lines are copied by
 * the TMA engine into a swizzled ring, or walked in 32-byte segments). Tiles
 * pass their prefixes on in a single pass from published tile aggregates
 * (after decoupled look-back, Merrill & Garland 2016); every wait is bounded.
 * Long-line calls clear their own tile state on `stream` first, so a call
 * captured in a CUDA graph is correct on every replay.
 *
 *   src, dst      device, same shape; dst may equal src (in place) but must
 *                 not otherwise overlap it
 * Exclusive scan (opts->exclusive = 1): element i holds the fold of init and
 *   the elements before it, y_1 = init, y_i = op(y_{i-1}, x_{i-1}). The pages
 *   describe inclusive scans only; this is its plain exclusive counterpart.
 *   Without init the neutral element stands for it (0 for +, 1 for *, the
 *   identity matrix); max / min and no_neutral then fail with
 *   AK_ERR_EMPTY_NO_INIT, since the first output has no value.
 * A wait that runs out (only possible through debug_skip_publish_tile or a
 * hardware fault) stops the kernel early; with opts->check set the call then
 * returns AK_ERR_TIMEOUT and dst is unspecified. Without check the call
 * returns AK_OK and the failure is recorded in the workspace: after the
 * stream has reached the end of the call, ak_scan_status(workspace) tells.
 * ------------------------------------------------------------------------- */
ak_status ak_accumulate_workspace_size(int ndim, const int64_t* shape, int dim, ak_dtype in,
                                       ak_dtype acc, ak_op op, const ak_opts* opts,
                                       size_t* bytes);
ak_status ak_accumulate(const void* src, void* dst, int ndim, const int64_t* shape, int dim,
                        ak_dtype in, ak_op op, ak_dtype acc, ak_dtype out, const void* init,
                        void* workspace, size_t workspace_bytes, const ak_opts* opts,
                        void* stream);
/* Outcome of the last ak_accumulate that used this workspace: AK_OK, or
 * AK_ERR_TIMEOUT when one of its bounded waits ran out. A blocking read of
 * the workspace's first word: call it once the caller's stream has passed the
 * scan (e.g. after cudaStreamSynchronize), not while it runs. */
ak_status ak_scan_status(const void* workspace);

/* ---------------------------------------------------------------------------
 * ak_findall: the indices of the nonzero elements of src, in increasing
 * order, and their count (Julia's findall over a Bool array, or over
 * x .!= 0). The tile-scan PR #202 counts findall among its scans (ratio
 * table; its tests paragraph): the output slot of a selected element is the
 * exclusive count of the selected elements before it. One pass: tiles count
 * their selected elements, publish the counts and derive their output
 * offsets by decoupled look-back (bounded waits), then store the indices.
 *
 *   src        device, n elements of `in`: AK_U8 (nonzero byte = true),
 *              AK_I32, AK_I64 (!= 0), AK_F32, AK_F64 (!= 0.0: -0.0 is
 *              false, NaN true)
 *   idx        device, room for n int64 (the count is at most n); receives
 *              the 0-based indices; entries past the count are untouched
 *   count_dev  device, one int64, or NULL
 *   count_host host, one int64, or NULL; when given the call synchronizes
 *              `stream` and returns the count there
 *   At least one of count_dev / count_host must be non-NULL.
 * The workspace is cleared by the call on its stream (graph-replay safe).
 * ------------------------------------------------------------------------- */
ak_status ak_findall_workspace_size(int64_t n, ak_dtype in, const ak_opts* opts, size_t* bytes);
ak_status ak_findall(const void* src, int64_t n, ak_dtype in, int64_t* idx, int64_t* count_dev,
                     int64_t* count_host, void* workspace, size_t workspace_bytes, const ak_opts* opts,
                     void* stream);

/* ---------------------------------------------------------------------------
 * ak_reduce_noalloc: ak_reduce for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers
 * that must not call cudaMalloc or any allocating routine when they reduce:
 * a real-time loop that cannot afford the implicit device synchronisation
 * of cudaMalloc / cudaFree, a process whose device memory is already fully
 * reserved by another allocator, or code held to a fixed memory budget.
 *
 * Arguments, results, store and empty-input rules are those of ak_reduce;
 * the caller still passes src and dst_dev / dst_host. The scratch (first-pass
 * partials and the bare result slot) lives in a fixed array of
 * AK_NOALLOC_SCRATCH_BYTES inside the library's device image, so every GPU
 * that loads the library holds that much memory until the process exits. A
 * call whose plan needs more scratch than that (it grows with the SM count
 * and the partial size, about 20 KB on a 152-SM GPU) returns
 * AK_ERR_WORKSPACE without launching anything.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture. The address is kept per device and CUDA
 * context: after a cudaDeviceReset the device's new context holds the array
 * at a new address, and the next call (again: outside any capture) looks it
 * up anew. Every call on a device shares the one array:
 * calls that may overlap on the GPU (different streams, no ordering) race
 * on it and give wrong results; order them on one stream. Nothing in the
 * array needs clearing between calls.
 * ------------------------------------------------------------------------- */
#define AK_NOALLOC_SCRATCH_BYTES 65536
ak_status ak_reduce_noalloc(const void* src, int64_t n, ak_dtype in, ak_map f, ak_op op, ak_dtype acc,
                            ak_dtype out, const void* init, ak_store mode, void* dst_dev, void* dst_host,
                            const ak_opts* opts, void* stream);

/* ---------------------------------------------------------------------------
 * Shape selector of ak_reduce_dims, exposed for inspection and tests (pure
 * host logic, no device needed). For a canonical strided problem of
 * `inner` contiguous outputs, reduction length `red_len` at stride `inner`
 * and `outer` output runs, elements of `elem_bytes` and vector width
 * `vec_elems`, on a device of `sm_count` SMs, writes the chosen shape, the
 * outputs per block along the contiguous dimension, the reduction rows per
 * block and the split factor.
 * ------------------------------------------------------------------------- */
ak_status ak_dims_select(int64_t inner, int64_t red_len, int64_t outer, int elem_bytes,
                         int vec_elems, int sm_count, int forced_shape, int32_t* shape_out,
                         int32_t* tile_outputs, int32_t* row_groups, int32_t* split);

#ifdef __cplusplus
}
#endif
#endif /* AK_H */
