// ak_internal.h -- host-side plumbing shared by the entry points: device
// properties, call epochs, launch accounting, type dispatch and the call
// descriptors handed from the validating front end (api.cu) to the kernel
// launchers (reduce.cu, reduce_dims.cu, scan.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <type_traits>
#include <cuda_runtime.h>

#include "../../include/ak.h"
#include "ak_types.cuh"

namespace ak {

// ---------------------------------------------------------------------------
// device properties (cached per device)
// ---------------------------------------------------------------------------
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;   // bytes per block with opt-in
    int max_threads_per_sm = 0;
    int l2_bytes = 0;
};
// Properties of the current device; returns false (and records the CUDA
// error) when there is none.
bool current_device(DeviceInfo* info);

// ---------------------------------------------------------------------------
// bookkeeping
// ---------------------------------------------------------------------------
// A process-unique 62-bit tag for one call: tile-state words written by
// older calls (or arbitrary memory) never match it, so workspaces need no
// clearing.
uint64_t next_epoch();
void count_launches(uint64_t k);
ak_status cuda_fail(cudaError_t e);  // records e, returns AK_ERR_CUDA
inline ak_status check_launch() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? AK_OK : cuda_fail(e);
}

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    uint64_t error_word;  // the call's epoch, written by a kernel that gave up waiting
    uint64_t pad[31];
};
constexpr size_t kWsHeader = 256;
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// type dispatch
// ---------------------------------------------------------------------------
template <class T>
struct Tag {
    using type = T;
};

// Calls f(Tag<In>, Tag<Acc>, Tag<Out>) for the supported type triples.
template <class F>
ak_status dispatch_types(ak_dtype in, ak_dtype acc, ak_dtype out, F&& f) {
#define AK_TRIPLE(I, A, O, TI, TA, TO) \
    if (in == I && acc == A && out == O) return f(Tag<TI>{}, Tag<TA>{}, Tag<TO>{});
    AK_TRIPLE(AK_F32, AK_F32, AK_F32, float, float, float)
    AK_TRIPLE(AK_F32, AK_F64, AK_F64, float, double, double)
    AK_TRIPLE(AK_F32, AK_F64, AK_F32, float, double, float)
    AK_TRIPLE(AK_F64, AK_F64, AK_F64, double, double, double)
    AK_TRIPLE(AK_BF16, AK_F32, AK_BF16, bf16, float, bf16)
    AK_TRIPLE(AK_BF16, AK_F32, AK_F32, bf16, float, float)
    AK_TRIPLE(AK_I32, AK_I32, AK_I32, int32_t, int32_t, int32_t)
    AK_TRIPLE(AK_I32, AK_I64, AK_I64, int32_t, int64_t, int64_t)
    AK_TRIPLE(AK_I64, AK_I64, AK_I64, int64_t, int64_t, int64_t)
    AK_TRIPLE(AK_MAT2_MODP, AK_MAT2_MODP, AK_MAT2_MODP, Mat2, Mat2, Mat2)
#undef AK_TRIPLE
    return AK_ERR_UNSUPPORTED;
}

template <class Acc>
constexpr bool is_mat2_v = std::is_same_v<Acc, Mat2>;

// Calls f(Tag<Op>) for an operator valid on Acc.
template <class Acc, class F>
ak_status dispatch_op(ak_op op, F&& f) {
    if constexpr (is_mat2_v<Acc>) {
        if (op == AK_OP_MATMUL_MODP) return f(Tag<OpMatMul>{});
        return AK_ERR_UNSUPPORTED;
    } else {
        switch (op) {
        case AK_OP_ADD: return f(Tag<OpAdd>{});
        case AK_OP_MUL: return f(Tag<OpMul>{});
        case AK_OP_MAX: return f(Tag<OpMax>{});
        case AK_OP_MIN: return f(Tag<OpMin>{});
        default: return AK_ERR_UNSUPPORTED;
        }
    }
}

template <class Acc, class F>
ak_status dispatch_map(ak_map m, F&& f) {
    if constexpr (is_mat2_v<Acc>) {
        if (m == AK_MAP_IDENTITY) return f(Tag<MapIdentity>{});
        return AK_ERR_UNSUPPORTED;
    } else {
        switch (m) {
        case AK_MAP_IDENTITY: return f(Tag<MapIdentity>{});
        case AK_MAP_ABS: return f(Tag<MapAbs>{});
        case AK_MAP_ABS2: return f(Tag<MapAbs2>{});
        default: return AK_ERR_UNSUPPORTED;
        }
    }
}

template <class Op, class Acc, class F>
ak_status dispatch_monoid(bool no_neutral, F&& f) {
    if (no_neutral) return f(Tag<Lifted<Op, Acc>>{});
    return f(Tag<Plain<Op, Acc>>{});
}

// Size of a partial result (accumulator, or Optional accumulator).
size_t partial_size(ak_dtype acc, bool no_neutral);

// ---------------------------------------------------------------------------
// call descriptors (validated by api.cu)
// ---------------------------------------------------------------------------
struct alignas(16) Value16 {
    unsigned char b[16];
};

struct ReduceCall {
    const void* src;
    const void* src2;  // second source of a fused element f(src[i], src2[i]), or NULL
    int map2;          // ak_map2 of the fused element
    int64_t n;  // > 0
    ak_dtype in, acc, out;
    ak_map f;
    ak_op op;
    bool no_neutral;
    ak_store mode;
    Value16 init;  // accumulator value (valid when mode == AK_STORE_INIT)
    void* dst;     // device output element, or NULL when `bare` is used
    void* bare;    // device slot for the bare partial result (host finish), or NULL
    void* host_flag = nullptr;  // with `bare` in mapped host memory: the word set to host_seq after it
    uint64_t host_seq = 0;
    void* ws;
    size_t ws_bytes;
    int target_blocks;
    cudaStream_t stream;
};

// Grid of the whole-array first pass and the workspace it needs.
struct ReducePlan {
    int grid;         // 1 = single launch
    size_t ws_bytes;  // header + partials + bare slot
    size_t partials_off, bare_off;
};
ak_status plan_reduce(int64_t n, ak_dtype in, ak_dtype acc, bool no_neutral, int target_blocks,
                      const DeviceInfo& dev, ReducePlan* plan);
ak_status run_reduce(const ReduceCall& c, const ReducePlan& plan);
// The whole-array entry behind ak_reduce / ak_reduce2 / ak_reduce_noalloc
// (api.cu): validation, empty rules, launch, host finish. host_slot: a host
// result may use the calling thread's pinned host slot.
ak_status reduce_entry(const void* src, const void* src2, int map2, int64_t n, ak_dtype in, ak_map f, ak_op op,
                       ak_dtype acc, ak_dtype out, const void* init, ak_store mode, void* dst_dev, void* dst_host,
                       void* ws, size_t ws_bytes, const ak_opts* opts, void* stream, bool host_slot);

// Canonical strided problem: out[i + inner*k] = fold_j x[i + ldj*j + ldk*k]
// (a dense array has ldj = inner, ldk = inner*red).
struct DimsCall {
    const void* src;
    int64_t inner, red, outer;
    int64_t ldj, ldk;  // source strides (elements) of the reduced and of the outer dimension
    ak_dtype in, acc, out;
    ak_map f;
    ak_op op;
    bool no_neutral;
    ak_store mode;
    Value16 init;
    void* dst;
    void* ws;
    size_t ws_bytes;
    int forced_shape;
    bool allow_cluster;  // AK_FLAG_DIMS_CLUSTER: combine split blocks in a cluster whenever one fits
    bool auto_cluster;   // auto shape: combine in a cluster for small inputs (see select_shape)
    cudaStream_t stream;
    // general fallback (any dims mask, any strides): full shape, strides and mask
    int ndim;
    int64_t shape[8];
    int64_t stride[8];
    uint32_t mask;
    bool general;
};

struct DimsPlan {
    int shape;        // ak_dims_shape actually used
    int vec;          // elements per vector load along the contiguous dimension
    int tile_out;     // outputs per block along the contiguous dimension
    int row_groups;   // reduction rows processed in parallel per block
    int split;        // blocks along the reduction (> 1: combined in a cluster or by a second pass)
    bool cluster;     // the split blocks of an output tile form one thread-block cluster
    size_t ws_bytes;
};
ak_status plan_dims(const DimsCall& c, const DeviceInfo& dev, DimsPlan* plan);
ak_status run_reduce_dims(const DimsCall& c, const DimsPlan& plan);

// Merged view of a dims reduction: size-1 dimensions dropped, neighbouring
// dimensions of the same kind (kept / reduced) merged when the source
// strides continue each other (always, for a dense array).
struct Canon {
    int64_t nout, nfold;
    int nseg;
    int64_t ext[8];
    int64_t st[8];  // source stride (elements) of each merged dimension
    bool red[8];
};

// The plan of a dims reduction: its merged view, the kernel call (source,
// types, geometry; the caller fills in output, operator, store mode, init,
// destination, workspace and stream), and either the whole-array plan
// (path 1: every element folds into one output) or the dims kernels' plan.
struct DimsSetup {
    Canon cn;
    DimsCall c;
    int path;  // 0 strided / rows / general, 1 whole-array
    ReducePlan rplan;
    DimsPlan dplan;
    size_t ws_bytes;
};
ak_status setup_dims(const void* src, int ndim, const int64_t* shape, const int64_t* strides, uint32_t mask,
                     ak_dtype in, ak_dtype acc, const ak_opts& o, DimsSetup* d);
// Fills R where the reduction is empty (store rules of ak_reduce).
ak_status run_fill(void* dst, int64_t count, ak_dtype out, const Value16& value, cudaStream_t s);

struct ScanCall {
    const void* src;
    void* dst;
    int64_t inner, len, outer;  // line of `len` elements at stride `inner`; inner*outer lines
    ak_dtype in, acc, out;
    ak_op op;
    bool no_neutral;
    bool has_init;
    bool exclusive;  // element i = fold of init and the elements before it (has_init is then set)
    Value16 init;
    void* ws;
    size_t ws_bytes;
    int target_blocks;
    int items;
    int64_t wait_limit_ns;
    int64_t skip_tile;
    uint64_t epoch;
    cudaStream_t stream;
};
struct ScanPlan {
    int kind;        // 0 = super-tile scan of long contiguous lines, 1 = strided (inner > 1),
                     // 2 = contiguous lines that fit one tile
    int block, items;
    int grid;
    int64_t tiles_per_line, tiles;
    size_t state_off, ws_bytes;
    // kind 0 only: the TMA tile scan applies (one element type throughout,
    // 128-byte rows); it is tried first and the super-tile scan is the
    // fallback (unaligned pointers), so ws_bytes covers both
    bool tma;
    int64_t tma_tiles_per_line, tma_tiles;
    size_t tma_ws_bytes;
    // kind 0, one line that fits L2 (not TMA): reduce-then-scan in three
    // launches; workspace offsets of the segment totals, tile aggregates and
    // tile prefixes
    bool three;
    size_t seg_off, agg_off, pre_off;
    // kind 1: the scanned dimension in `chunks` chunks of chunk_rows rows
    // (1: one thread per column walks it all); the chunk totals at seg_off
    int64_t chunks, chunk_rows;
};
ak_status plan_scan(int64_t inner, int64_t len, int64_t outer, ak_dtype in, ak_dtype acc, ak_dtype out,
                    ak_op op, bool no_neutral, int target_blocks, int items,
                    const DeviceInfo& dev, ScanPlan* plan, bool single_pass = false);
ak_status run_scan(const ScanCall& c, const ScanPlan& plan);

// findall: tiles and workspace; the kernel of findall.cu.
ak_status plan_findall(int64_t n, ak_dtype in, int64_t* ntiles, size_t* ws_bytes, size_t* count_off);
ak_status run_findall(const void* src, int64_t n, ak_dtype in, int64_t* idx, int64_t* count, void* ws,
                      int64_t ntiles, size_t ws_bytes, uint64_t epoch, int64_t wait_limit_ns, int64_t skip_tile,
                      int target_blocks, cudaStream_t stream);

}  // namespace ak
