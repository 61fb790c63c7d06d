// api.cu -- the C entry points of include/ak.h: argument validation (before
// anything touches the device), dimension canonicalisation, workspace
// sizing, empty-input rules and the host-side finish of a host result.
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <random>

#include "ak_common.cuh"
#include "ak_internal.h"

namespace ak {

// ---------------------------------------------------------------------------
// bookkeeping
// ---------------------------------------------------------------------------

static thread_local int g_last_cuda_error = 0;
static std::atomic<uint64_t> g_launches{0};

ak_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    cudaGetLastError();  // clear a sticky-free error so later calls are unaffected
    return AK_ERR_CUDA;
}

void count_launches(uint64_t k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

uint64_t next_epoch() {
    // Start from a random 62-bit value so that two processes sharing recycled
    // device memory do not produce the same tags either.
    static std::atomic<uint64_t> counter{[] {
        std::random_device rd;
        uint64_t s = ((uint64_t)rd() << 32) ^ rd() ^
                     (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
        return s & ((1ull << 61) - 1);
    }()};
    return (counter.fetch_add(1) + 1) & ((1ull << 62) - 1);
}

bool current_device(DeviceInfo* info) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        if (e != cudaSuccess) cuda_fail(e);
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].device != dev) {
        DeviceInfo d;
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) {
            cuda_fail(e);
            return false;
        }
        cache[dev] = d;
    }
    *info = cache[dev];
    return true;
}

size_t partial_size(ak_dtype acc, bool no_neutral) {
    const size_t a = ak_dtype_size(acc);
    if (a == 0) return 0;
    if (!no_neutral) return a;
    // Opt<T> = {T v; uint32 present} with T's alignment
    const size_t align = a >= 16 ? 16 : a;
    return align_up(a + 4, std::max<size_t>(align, 4));
}

// ---------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------

static bool valid_dtype(int t) { return t >= AK_F32 && t <= AK_U8; }

static ak_status check_types(ak_dtype in, ak_map f, ak_op op, ak_dtype acc, ak_dtype out) {
    if (!valid_dtype(in) || !valid_dtype(acc) || !valid_dtype(out)) return AK_ERR_INVALID_ARG;
    if (f < AK_MAP_IDENTITY || f > AK_MAP_ABS2) return AK_ERR_INVALID_ARG;
    if (op < AK_OP_ADD || op > AK_OP_MATMUL_MODP) return AK_ERR_INVALID_ARG;
    const bool mat = in == AK_MAT2_MODP;
    if (mat != (op == AK_OP_MATMUL_MODP)) return AK_ERR_UNSUPPORTED;
    if (mat && f != AK_MAP_IDENTITY) return AK_ERR_UNSUPPORTED;
    return dispatch_types(in, acc, out, [](auto, auto, auto) { return AK_OK; });
}

static bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

static ak_opts resolve_opts(const ak_opts* o) {
    ak_opts r;
    ak_opts_default(&r);
    if (o) r = *o;
    if (r.wait_limit_ns <= 0) r.wait_limit_ns = 1000000000LL;
    return r;
}

// Neutral element of op in the accumulator type (Julia's reduce_empty:
// zero for +, one for *, the identity matrix); false for max / min.
static bool neutral_value(ak_op op, ak_dtype acc, Value16* v) {
    memset(v->b, 0, sizeof v->b);
    auto put = [&](auto x) { memcpy(v->b, &x, sizeof x); };
    switch (op) {
    case AK_OP_ADD:
        return true;  // all-zero bytes: +0.0, 0
    case AK_OP_MUL:
        switch (acc) {
        case AK_F32: put(1.0f); return true;
        case AK_F64: put(1.0); return true;
        case AK_I32: put((int32_t)1); return true;
        case AK_I64: put((int64_t)1); return true;
        default: return false;
        }
    case AK_OP_MATMUL_MODP: put(Mat2{1u, 0u, 0u, 1u}); return true;
    default: return false;
    }
}

// Converts one accumulator value to the output type (host side).
static Value16 acc_to_out(const Value16& a, ak_dtype acc, ak_dtype out) {
    Value16 r;
    memset(r.b, 0, sizeof r.b);
    auto conv = [&](auto from, auto to) {
        using A = decltype(from);
        using O = decltype(to);
        A v;
        memcpy(&v, a.b, sizeof v);
        O o = convert<O>(v);
        memcpy(r.b, &o, sizeof o);
    };
    if (acc == AK_F32 && out == AK_BF16) conv(float{}, bf16{});
    else if (acc == AK_F64 && out == AK_F32) conv(double{}, float{});
    else memcpy(r.b, a.b, sizeof r.b);  // same type
    return r;
}

// Host finish of a bare partial: apply the store mode, convert to out.
static ak_status host_finish(const void* bare, ak_dtype in, ak_dtype acc, ak_dtype out, ak_op op,
                             bool no_neutral, ak_store mode, const Value16& init, void* dst_host) {
    return dispatch_types(in, acc, out, [&](auto, auto ta, auto to) -> ak_status {
        using Acc = typename decltype(ta)::type;
        using Out = typename decltype(to)::type;
        return dispatch_op<Acc>(op, [&](auto top) -> ak_status {
            using Op = typename decltype(top)::type;
            return dispatch_monoid<Op, Acc>(no_neutral, [&](auto tmo) -> ak_status {
                using M = typename decltype(tmo)::type;
                typename M::P p;
                memcpy(&p, bare, sizeof p);
                if (!M::present(p)) return AK_ERR_EMPTY_NO_INIT;
                Acc v = M::value(p);
                if (mode == AK_STORE_INIT) {
                    Acc i;
                    memcpy(&i, init.b, sizeof i);
                    v = Op::apply(i, v);
                } else if (mode == AK_STORE_FOLD) {
                    Out old;
                    memcpy(&old, dst_host, sizeof old);
                    v = Op::apply(convert<Acc>(old), v);
                }
                Out o = convert<Out>(v);
                memcpy(dst_host, &o, sizeof o);
                return AK_OK;
            });
        });
    });
}

// AK_LOG set (and not "0") in the environment: one line per call on stderr
// naming the path the call takes -- kernel, grid or tile count, dims shape.
// The variable is read on every call, so it can be switched at run time.
static bool log_on() {
    const char* v = getenv("AK_LOG");
    return v && *v && strcmp(v, "0") != 0;
}

static void log_call(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    char line[256];
    vsnprintf(line, sizeof line, fmt, ap);
    va_end(ap);
    fprintf(stderr, "[ak] %s\n", line);
}

static const char* dtype_name(ak_dtype t) {
    static const char* names[] = {"f32", "f64", "i32", "i64", "bf16", "mat2", "u8"};
    return (int)t >= 0 && (int)t < 7 ? names[t] : "?";
}

static const char* op_name(ak_op op) {
    static const char* names[] = {"add", "mul", "max", "min", "matmul_modp"};
    return (int)op >= 0 && (int)op < 5 ? names[op] : "?";
}

static ak_status sync_and_check(cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? AK_OK : cuda_fail(e);
}

// Byte offset of the flag word in a host-result slot (after the bare partial).
constexpr size_t kSlotFlagOff = 32;

// Waits until the host-result slot's flag word holds seq: polled for up to
// about 200 us (the result lands before the grid has retired and before the
// stream would report completion), then a stream synchronization, which also
// reports any error of the stream.
static ak_status wait_slot(const unsigned char* slot, uint64_t seq, cudaStream_t s) {
    const uint64_t* flag = reinterpret_cast<const uint64_t*>(slot + kSlotFlagOff);
    const auto t0 = std::chrono::steady_clock::now();
    for (int i = 1;; ++i) {
        if (__atomic_load_n(flag, __ATOMIC_ACQUIRE) == seq) return AK_OK;
        if ((i & 1023) == 0 && std::chrono::steady_clock::now() - t0 > std::chrono::microseconds(200)) break;
    }
    const ak_status st = sync_and_check(s);
    if (st != AK_OK) return st;
    return __atomic_load_n(flag, __ATOMIC_ACQUIRE) == seq ? AK_OK : cuda_fail(cudaErrorUnknown);
}

}  // namespace ak

using namespace ak;

// ===========================================================================
// misc
// ===========================================================================

extern "C" void ak_opts_default(ak_opts* o) {
    if (!o) return;
    memset(o, 0, sizeof *o);
    o->debug_skip_publish_tile = -1;
}

extern "C" const char* ak_status_string(ak_status s) {
    switch (s) {
    case AK_OK: return "ok";
    case AK_ERR_INVALID_ARG: return "invalid argument";
    case AK_ERR_UNSUPPORTED: return "unsupported type / operator / map combination";
    case AK_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case AK_ERR_EMPTY_NO_INIT: return "empty reduction without init or neutral element";
    case AK_ERR_CUDA: return "CUDA runtime error";
    case AK_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    default: return "unknown status";
    }
}

extern "C" size_t ak_dtype_size(ak_dtype t) {
    switch (t) {
    case AK_F32: return 4;
    case AK_F64: return 8;
    case AK_BF16: return 2;
    case AK_I32: return 4;
    case AK_I64: return 8;
    case AK_MAT2_MODP: return 16;
    case AK_U8: return 1;
    default: return 0;
    }
}

extern "C" int ak_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" uint64_t ak_kernel_launch_count(void) { return g_launches.load(); }

// ===========================================================================
// ak_reduce
// ===========================================================================

extern "C" ak_status ak_reduce_workspace_size(int64_t n, ak_dtype in, ak_dtype acc, const ak_opts* opts,
                                              size_t* bytes) {
    if (!bytes || n < 0 || !valid_dtype(in) || !valid_dtype(acc)) return AK_ERR_INVALID_ARG;
    const ak_opts o = resolve_opts(opts);
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    ReducePlan plan;
    ak_status s = plan_reduce(std::max<int64_t>(n, 1), in, acc, o.no_neutral != 0, o.target_blocks, dev, &plan);
    if (s != AK_OK) return s;
    *bytes = plan.ws_bytes;
    return AK_OK;
}

// A per-thread slot of mapped, pinned host memory for host results: the
// finishing kernel writes the bare partial straight into its first 32 bytes
// (no copy to enqueue, no staging of a pageable buffer), then the call's
// sequence number into the word at byte 32, which the host polls. Allocated
// on a thread's first host-result call and kept until the process exits (64
// bytes). Null when the allocation fails: the caller then copies through
// the workspace.
static unsigned char* host_result_slot(void** dev_ptr) {
    struct Slot {
        unsigned char* host = nullptr;
        void* dev = nullptr;
        bool tried = false;
    };
    static thread_local Slot slot;
    if (!slot.tried) {
        slot.tried = true;
        void* h = nullptr;
        if (cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess) {
            // a zero flag word: no call's sequence number (they start at 1)
            memset(h, 0, 64);
            void* d = nullptr;
            if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) {
                slot.host = static_cast<unsigned char*>(h);
                slot.dev = d;
            } else {
                cudaFreeHost(h);
            }
        }
        cudaGetLastError();
    }
    *dev_ptr = slot.dev;
    return slot.host;
}

// ak_reduce, ak_reduce2 and ak_reduce_noalloc: one source, or a fused
// element f(src[i], src2[i]). host_slot: a host result may go through the
// calling thread's pinned slot (not for callers that must not allocate).
ak_status ak::reduce_entry(const void* src, const void* src2, int map2, int64_t n, ak_dtype in, ak_map f,
                           ak_op op, ak_dtype acc, ak_dtype out, const void* init, ak_store mode, void* dst_dev,
                           void* dst_host, void* ws, size_t ws_bytes, const ak_opts* opts, void* stream,
                           bool host_slot) {
    ak_status s = check_types(in, f, op, acc, out);
    if (s != AK_OK) return s;
    if (n < 0 || (n > 0 && !src) || (!dst_dev && !dst_host)) return AK_ERR_INVALID_ARG;
    if (src2) {
        if (map2 < AK_MAP2_MUL || map2 > AK_MAP2_ABSDIFF || f != AK_MAP_IDENTITY) return AK_ERR_INVALID_ARG;
        if (in == AK_MAT2_MODP) return AK_ERR_UNSUPPORTED;
        if (!aligned(src2, ak_dtype_size(in))) return AK_ERR_INVALID_ARG;
    }
    if (mode < AK_STORE_OVERWRITE || mode > AK_STORE_FOLD || (mode == AK_STORE_INIT && !init))
        return AK_ERR_INVALID_ARG;
    if (src && !aligned(src, ak_dtype_size(in) >= 16 ? 16 : ak_dtype_size(in))) return AK_ERR_INVALID_ARG;
    if (dst_dev && !aligned(dst_dev, ak_dtype_size(out) >= 16 ? 16 : ak_dtype_size(out))) return AK_ERR_INVALID_ARG;
    const ak_opts o = resolve_opts(opts);
    const bool no_neutral = o.no_neutral != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Value16 ini;
    memset(ini.b, 0, sizeof ini.b);
    if (init) memcpy(ini.b, init, ak_dtype_size(acc));

    if (n == 0) {
        // Empty input: init / unchanged R / neutral element.
        Value16 val;
        if (mode == AK_STORE_INIT) val = ini;
        else if (mode == AK_STORE_FOLD) {
            if (dst_host && dst_dev) {
                cudaError_t e = cudaMemcpyAsync(dst_host, dst_dev, ak_dtype_size(out), cudaMemcpyDeviceToHost, st);
                if (e != cudaSuccess) return cuda_fail(e);
                return sync_and_check(st);
            }
            return AK_OK;
        } else if (no_neutral || !neutral_value(op, acc, &val)) {
            return AK_ERR_EMPTY_NO_INIT;
        }
        Value16 ov = acc_to_out(val, acc, out);
        if (dst_dev) {
            s = run_fill(dst_dev, 1, out, ov, st);
            if (s != AK_OK) return s;
        }
        if (dst_host) {
            memcpy(dst_host, ov.b, ak_dtype_size(out));
            if (dst_dev) return sync_and_check(st);
        }
        return AK_OK;
    }

    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    ReducePlan plan;
    s = plan_reduce(n, in, acc, no_neutral, o.target_blocks, dev, &plan);
    if (s != AK_OK) return s;
    if (!ws || ws_bytes < plan.ws_bytes || !aligned(ws, 16)) return AK_ERR_WORKSPACE;

    ReduceCall c;
    c.src = src;
    c.src2 = src2;
    c.map2 = map2;
    c.n = n;
    c.in = in;
    c.acc = acc;
    c.out = out;
    c.f = f;
    c.op = op;
    c.no_neutral = no_neutral;
    c.mode = mode;
    c.init = ini;
    c.dst = dst_dev;
    c.bare = dst_dev ? nullptr : static_cast<char*>(ws) + plan.bare_off;
    unsigned char* slot = nullptr;
    if (!dst_dev && host_slot) {
        void* slot_dev = nullptr;
        slot = host_result_slot(&slot_dev);
        if (slot) {
            static thread_local uint64_t seq = 0;
            c.bare = slot_dev;
            c.host_flag = static_cast<char*>(slot_dev) + kSlotFlagOff;
            c.host_seq = ++seq;
        }
    }
    c.ws = ws;
    c.ws_bytes = ws_bytes;
    c.target_blocks = o.target_blocks;
    c.stream = st;
    if (log_on())
        log_call("%s n=%lld in=%s acc=%s op=%s first pass %d block(s)%s, result to %s", src2 ? "reduce2" : "reduce",
                 (long long)n, dtype_name(in), dtype_name(acc), op_name(op), plan.grid,
                 plan.grid > 1 ? " + one-block finish" : "",
                 dst_dev ? "device" : (slot ? "host (mapped slot, polled)" : "host (copy)"));
    s = run_reduce(c, plan);
    if (s != AK_OK) return s;

    if (dst_host) {
        if (dst_dev) {
            cudaError_t e = cudaMemcpyAsync(dst_host, dst_dev, ak_dtype_size(out), cudaMemcpyDeviceToHost, st);
            if (e != cudaSuccess) return cuda_fail(e);
            return sync_and_check(st);
        }
        if (slot) {
            s = wait_slot(slot, c.host_seq, st);
            if (s != AK_OK) return s;
            alignas(16) unsigned char bare[32];
            memcpy(bare, slot, sizeof bare);
            return host_finish(bare, in, acc, out, op, no_neutral, mode, ini, dst_host);
        }
        const size_t psz = partial_size(acc, no_neutral);
        alignas(16) unsigned char bare[32];
        cudaError_t e = cudaMemcpyAsync(bare, c.bare, psz, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_fail(e);
        s = sync_and_check(st);
        if (s != AK_OK) return s;
        return host_finish(bare, in, acc, out, op, no_neutral, mode, ini, dst_host);
    }
    if (o.check) return sync_and_check(st);
    return AK_OK;
}

extern "C" ak_status ak_reduce(const void* src, int64_t n, ak_dtype in, ak_map f, ak_op op, ak_dtype acc,
                               ak_dtype out, const void* init, ak_store mode, void* dst_dev, void* dst_host,
                               void* ws, size_t ws_bytes, const ak_opts* opts, void* stream) {
    return reduce_entry(src, nullptr, 0, n, in, f, op, acc, out, init, mode, dst_dev, dst_host, ws, ws_bytes, opts,
                        stream, true);
}

extern "C" ak_status ak_reduce2(const void* src_a, const void* src_b, int64_t n, ak_dtype in, ak_map2 f,
                                ak_op op, ak_dtype acc, ak_dtype out, const void* init, ak_store mode,
                                void* dst_dev, void* dst_host, void* ws, size_t ws_bytes, const ak_opts* opts,
                                void* stream) {
    if (n > 0 && !src_b) return AK_ERR_INVALID_ARG;
    // a fused element needs a second source even when n == 0 decides nothing
    const void* b = src_b ? src_b : reinterpret_cast<const void*>(uintptr_t(256));
    return reduce_entry(src_a, b, (int)f, n, in, AK_MAP_IDENTITY, op, acc, out, init, mode, dst_dev, dst_host, ws,
                        ws_bytes, opts, stream, true);
}

// ===========================================================================
// ak_reduce_dims
// ===========================================================================

namespace {

ak_status canonicalize(int ndim, const int64_t* shape, const int64_t* strides, uint32_t mask, Canon* c) {
    if (ndim < 1 || ndim > 8 || !shape) return AK_ERR_INVALID_ARG;
    if (mask >> ndim) return AK_ERR_INVALID_ARG;
    c->nout = c->nfold = 1;
    c->nseg = 0;
    int64_t dense = 1;
    for (int d = 0; d < ndim; ++d) {
        if (shape[d] < 0 || (strides && strides[d] < 0)) return AK_ERR_INVALID_ARG;
        const int64_t sd = strides ? strides[d] : dense;
        dense *= shape[d];
        const bool r = (mask >> d) & 1u;
        if (r) c->nfold *= shape[d];
        else c->nout *= shape[d];
        if (shape[d] == 1) continue;
        const int q = c->nseg - 1;
        if (q >= 0 && c->red[q] == r && sd == c->st[q] * c->ext[q]) c->ext[q] *= shape[d];
        else {
            c->ext[c->nseg] = shape[d];
            c->st[c->nseg] = sd;
            c->red[c->nseg] = r;
            ++c->nseg;
        }
    }
    return AK_OK;
}

// Fill the DimsCall's canonical fields; returns 0 strided / rows / general,
// 1 whole-array (one output over one contiguous range).
int classify(const Canon& cn, DimsCall* c) {
    c->general = false;
    c->inner = c->red = c->outer = 1;
    c->ldj = c->ldk = 0;
    if (cn.nseg == 0) return 0;  // a single element
    if (cn.nseg == 1) {
        if (cn.red[0] && cn.st[0] == 1) return 1;
        if (!cn.red[0] && cn.st[0] == 1) {
            c->inner = cn.ext[0];
            return 0;
        }
    } else if (cn.nseg == 2 && cn.red[0] != cn.red[1]) {
        if (cn.red[0] && cn.st[0] == 1) {  // rows: contiguous reductions at stride ldk
            c->red = cn.ext[0];
            c->outer = cn.ext[1];
            c->ldk = cn.st[1];
            return 0;
        }
        if (!cn.red[0] && cn.st[0] == 1) {  // strided: contiguous outputs, rows at stride ldj
            c->inner = cn.ext[0];
            c->red = cn.ext[1];
            c->ldj = cn.st[1];
            return 0;
        }
    } else if (cn.nseg == 3 && !cn.red[0] && cn.red[1] && !cn.red[2] && cn.st[0] == 1) {
        c->inner = cn.ext[0];
        c->red = cn.ext[1];
        c->outer = cn.ext[2];
        c->ldj = cn.st[1];
        c->ldk = cn.st[2];
        return 0;
    }
    c->general = true;
    return 0;
}

}  // namespace

ak_status ak::setup_dims(const void* src, int ndim, const int64_t* shape, const int64_t* strides, uint32_t mask,
                     ak_dtype in, ak_dtype acc, const ak_opts& o, DimsSetup* d) {
    ak_status s = canonicalize(ndim, shape, strides, mask, &d->cn);
    if (s != AK_OK) return s;
    memset(&d->c, 0, sizeof d->c);
    d->c.src = src;
    d->c.in = in;
    d->c.acc = acc;
    d->c.no_neutral = o.no_neutral != 0;
    d->c.forced_shape = o.dims_shape;
    d->c.allow_cluster = (o.flags & AK_FLAG_DIMS_CLUSTER) != 0;
    d->c.auto_cluster = true;
    d->c.ndim = ndim;
    d->c.mask = mask;
    int64_t dense = 1;
    for (int i = 0; i < ndim; ++i) {
        d->c.shape[i] = shape[i];
        d->c.stride[i] = strides ? strides[i] : dense;
        dense *= shape[i];
    }
    d->path = classify(d->cn, &d->c);
    d->ws_bytes = kWsHeader;
    if (d->cn.nout == 0 || d->cn.nfold == 0) return AK_OK;
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    if (d->path == 1) {
        s = plan_reduce(d->cn.nfold, in, acc, d->c.no_neutral, o.target_blocks, dev, &d->rplan);
        d->ws_bytes = d->rplan.ws_bytes;
    } else {
        s = plan_dims(d->c, dev, &d->dplan);
        d->ws_bytes = d->dplan.ws_bytes;
    }
    return s;
}

extern "C" ak_status ak_reduce_dims_workspace_size(int ndim, const int64_t* shape, const int64_t* strides,
                                                   uint32_t dims_mask, ak_dtype in, ak_dtype acc, const ak_opts* opts,
                                                   size_t* bytes) {
    if (!bytes || !valid_dtype(in) || !valid_dtype(acc)) return AK_ERR_INVALID_ARG;
    if (opts && (opts->dims_shape < AK_SHAPE_AUTO || opts->dims_shape > AK_SHAPE_COLUMNS)) return AK_ERR_INVALID_ARG;
    const ak_opts o = resolve_opts(opts);
    // The plan depends on the source alignment (vector width) and on whether
    // a cluster fits; report the largest workspace any of them needs: an
    // aligned and an element-aligned source, with and without the cluster
    // combine.
    size_t most = 0;
    for (int variant = 0; variant < 4; ++variant) {
        ak_opts ov = o;
        if (variant & 2) ov.flags &= ~AK_FLAG_DIMS_CLUSTER;
        DimsSetup d;
        const uintptr_t addr = 256 + ((variant & 1) ? ak_dtype_size(in) : 0);
        ak_status s = setup_dims(reinterpret_cast<const void*>(addr), ndim, shape, strides, dims_mask, in, acc, ov,
                                 &d);
        if (s != AK_OK) return s;
        if (variant & 2) {
            // the same call planned without the cluster combine
            d.c.auto_cluster = false;
            d.c.allow_cluster = false;
            if (d.path != 1 && d.cn.nout != 0 && d.cn.nfold != 0) {
                DeviceInfo dev;
                if (!current_device(&dev)) return AK_ERR_CUDA;
                s = plan_dims(d.c, dev, &d.dplan);
                if (s != AK_OK) return s;
                d.ws_bytes = d.dplan.ws_bytes;
            }
        }
        most = std::max(most, d.ws_bytes);
    }
    *bytes = most;
    return AK_OK;
}

extern "C" ak_status ak_reduce_dims(const void* src, int ndim, const int64_t* shape, const int64_t* strides,
                                    uint32_t dims_mask, ak_dtype in, ak_map f, ak_op op, ak_dtype acc, ak_dtype out,
                                    const void* init, ak_store mode, void* dst, void* ws, size_t ws_bytes,
                                    const ak_opts* opts, void* stream) {
    ak_status s = check_types(in, f, op, acc, out);
    if (s != AK_OK) return s;
    if (mode < AK_STORE_OVERWRITE || mode > AK_STORE_FOLD || (mode == AK_STORE_INIT && !init))
        return AK_ERR_INVALID_ARG;
    if (opts && (opts->dims_shape < AK_SHAPE_AUTO || opts->dims_shape > AK_SHAPE_COLUMNS)) return AK_ERR_INVALID_ARG;
    const ak_opts o = resolve_opts(opts);
    DimsSetup d;
    s = setup_dims(src, ndim, shape, strides, dims_mask, in, acc, o, &d);
    if (s != AK_OK) return s;
    const int64_t nin = d.cn.nout * d.cn.nfold;
    if ((nin > 0 && !src) || (d.cn.nout > 0 && !dst)) return AK_ERR_INVALID_ARG;
    if (src && !aligned(src, ak_dtype_size(in) >= 16 ? 16 : ak_dtype_size(in))) return AK_ERR_INVALID_ARG;
    if (dst && !aligned(dst, ak_dtype_size(out) >= 16 ? 16 : ak_dtype_size(out))) return AK_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Value16 ini;
    memset(ini.b, 0, sizeof ini.b);
    if (init) memcpy(ini.b, init, ak_dtype_size(acc));
    if (d.cn.nout == 0) return AK_OK;
    if (d.cn.nfold == 0) {
        Value16 val;
        if (mode == AK_STORE_FOLD) return AK_OK;
        if (mode == AK_STORE_INIT) val = ini;
        else if (o.no_neutral || !neutral_value(op, acc, &val)) return AK_ERR_EMPTY_NO_INIT;
        s = run_fill(dst, d.cn.nout, out, acc_to_out(val, acc, out), st);
        if (s == AK_OK && o.check) s = sync_and_check(st);
        return s;
    }
    if (!ws || ws_bytes < d.ws_bytes || !aligned(ws, 16)) return AK_ERR_WORKSPACE;
    if (log_on()) {
        static const char* shapes[] = {"auto", "thread", "tiled", "columns"};
        if (d.path == 1)
            log_call("reduce_dims nout=%lld nfold=%lld in=%s op=%s whole-array reduce, %d block(s)",
                     (long long)d.cn.nout, (long long)d.cn.nfold, dtype_name(in), op_name(op), d.rplan.grid);
        else if (d.c.general)
            log_call("reduce_dims nout=%lld nfold=%lld in=%s op=%s general kernel", (long long)d.cn.nout,
                     (long long)d.cn.nfold, dtype_name(in), op_name(op));
        else
            log_call("reduce_dims nout=%lld nfold=%lld in=%s op=%s %s kernel shape=%s vec=%d tile_out=%d "
                     "row_groups=%d split=%d%s",
                     (long long)d.cn.nout, (long long)d.cn.nfold, dtype_name(in), op_name(op),
                     d.c.inner == 1 ? "rows" : "strided",
                     d.dplan.shape >= 0 && d.dplan.shape < 4 ? shapes[d.dplan.shape] : "?", d.dplan.vec,
                     d.dplan.tile_out, d.dplan.row_groups, d.dplan.split,
                     d.dplan.split > 1 ? (d.dplan.cluster ? " (cluster combine)" : " (second pass)") : "");
    }
    if (d.path == 1) {
        ReduceCall c;
        c.src = src;
        c.src2 = nullptr;
        c.map2 = 0;
        c.n = d.cn.nfold;
        c.in = in;
        c.acc = acc;
        c.out = out;
        c.f = f;
        c.op = op;
        c.no_neutral = o.no_neutral != 0;
        c.mode = mode;
        c.init = ini;
        c.dst = dst;
        c.bare = nullptr;
        c.ws = ws;
        c.ws_bytes = ws_bytes;
        c.target_blocks = o.target_blocks;
        c.stream = st;
        s = run_reduce(c, d.rplan);
    } else {
        DimsCall& c = d.c;
        c.out = out;
        c.f = f;
        c.op = op;
        c.mode = mode;
        c.init = ini;
        c.dst = dst;
        c.ws = ws;
        c.ws_bytes = ws_bytes;
        c.stream = st;
        s = run_reduce_dims(c, d.dplan);
    }
    if (s == AK_OK && o.check) s = sync_and_check(st);
    return s;
}

// ===========================================================================
// ak_accumulate
// ===========================================================================

namespace {

ak_status scan_geometry(int ndim, const int64_t* shape, int dim, int64_t* inner, int64_t* len, int64_t* outer) {
    if (ndim < 1 || ndim > 8 || !shape || dim < -1 || dim >= ndim) return AK_ERR_INVALID_ARG;
    int64_t n = 1;
    for (int d = 0; d < ndim; ++d) {
        if (shape[d] < 0) return AK_ERR_INVALID_ARG;
        n *= shape[d];
    }
    if (dim < 0) {
        *inner = 1;
        *len = n;
        *outer = 1;
        return AK_OK;
    }
    int64_t a = 1, b = 1;
    for (int d = 0; d < dim; ++d) a *= shape[d];
    for (int d = dim + 1; d < ndim; ++d) b *= shape[d];
    *inner = a;
    *len = shape[dim];
    *outer = b;
    return AK_OK;
}

}  // namespace

extern "C" ak_status ak_accumulate_workspace_size(int ndim, const int64_t* shape, int dim, ak_dtype in,
                                                  ak_dtype acc, ak_op op, const ak_opts* opts, size_t* bytes) {
    if (!bytes || !valid_dtype(in) || !valid_dtype(acc)) return AK_ERR_INVALID_ARG;
    int64_t inner, len, outer;
    ak_status s = scan_geometry(ndim, shape, dim, &inner, &len, &outer);
    if (s != AK_OK) return s;
    const ak_opts o = resolve_opts(opts);
    DeviceInfo dev = {};
    ScanPlan p;
    // the output type is not part of this query: planning with out = acc
    // covers the largest workspace any output type can need
    s = plan_scan(inner, len, outer, in, acc, acc, op, o.no_neutral != 0, o.target_blocks, o.items_per_thread, dev, &p);
    if (s != AK_OK) return s;
    *bytes = p.ws_bytes;
    return AK_OK;
}

extern "C" ak_status ak_accumulate(const void* src, void* dst, int ndim, const int64_t* shape, int dim,
                                   ak_dtype in, ak_op op, ak_dtype acc, ak_dtype out, const void* init,
                                   void* ws, size_t ws_bytes, const ak_opts* opts, void* stream) {
    ak_status s = check_types(in, AK_MAP_IDENTITY, op, acc, out);
    if (s != AK_OK) return s;
    int64_t inner, len, outer;
    s = scan_geometry(ndim, shape, dim, &inner, &len, &outer);
    if (s != AK_OK) return s;
    const int64_t n = inner * len * outer;
    if (opts && (opts->exclusive < 0 || opts->exclusive > 1 || opts->reserved != 0)) return AK_ERR_INVALID_ARG;
    if (n == 0) return AK_OK;
    if (!src || !dst) return AK_ERR_INVALID_ARG;
    const size_t isz = ak_dtype_size(in), osz = ak_dtype_size(out);
    if (!aligned(src, isz >= 16 ? 16 : isz) || !aligned(dst, osz >= 16 ? 16 : osz)) return AK_ERR_INVALID_ARG;
    // in place only when both views coincide exactly
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(src), a1 = a0 + (uintptr_t)(n * isz);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(dst), b1 = b0 + (uintptr_t)(n * osz);
    if (a0 < b1 && b0 < a1 && !(a0 == b0 && isz == osz)) return AK_ERR_INVALID_ARG;
    const ak_opts o = resolve_opts(opts);
    DeviceInfo dev;
    if (!current_device(&dev)) return AK_ERR_CUDA;
    ScanPlan p;
    // fault injection targets the single-pass kernels' bounded waits
    s = plan_scan(inner, len, outer, in, acc, out, op, o.no_neutral != 0, o.target_blocks, o.items_per_thread, dev, &p,
                  o.debug_skip_publish_tile >= 0);
    if (s != AK_OK) return s;
    if (!ws || ws_bytes < p.ws_bytes || !aligned(ws, 16)) return AK_ERR_WORKSPACE;
    ScanCall c;
    c.src = src;
    c.dst = dst;
    c.inner = inner;
    c.len = len;
    c.outer = outer;
    c.in = in;
    c.acc = acc;
    c.out = out;
    c.op = op;
    c.no_neutral = o.no_neutral != 0;
    c.has_init = init != nullptr;
    c.exclusive = o.exclusive != 0;
    memset(c.init.b, 0, sizeof c.init.b);
    if (init) memcpy(c.init.b, init, ak_dtype_size(acc));
    if (c.exclusive && !init) {
        // the first output is the empty prefix: the neutral element stands
        // for init where one exists (+0.0 for a float sum, as Julia's zero)
        if (c.no_neutral || !neutral_value(op, acc, &c.init)) return AK_ERR_EMPTY_NO_INIT;
        c.has_init = true;
    }
    c.ws = ws;
    c.ws_bytes = ws_bytes;
    c.target_blocks = o.target_blocks;
    c.items = o.items_per_thread;
    c.wait_limit_ns = o.wait_limit_ns;
    c.skip_tile = o.debug_skip_publish_tile;
    c.epoch = next_epoch();
    c.stream = static_cast<cudaStream_t>(stream);
    if (log_on()) {
        const char* k = p.kind == 1 ? "strided (a thread per column)"
                        : p.kind == 2 ? "lines (one block per line)"
                        : p.tma ? "TMA tile ring (super-tiles if the pointers are not 16-byte aligned)"
                        : p.three ? "three-launch reduce-then-scan"
                                  : "single-pass super-tiles";
        log_call("accumulate inner=%lld len=%lld outer=%lld in=%s acc=%s op=%s%s%s: %s, %lld tile(s)",
                 (long long)inner, (long long)len, (long long)outer, dtype_name(in), dtype_name(acc), op_name(op),
                 c.exclusive ? " exclusive" : "", c.no_neutral ? " optional partials" : "", k,
                 (long long)(p.tma ? p.tma_tiles : p.tiles));
    }
    s = run_scan(c, p);
    if (s != AK_OK || !o.check) return s;
    s = sync_and_check(c.stream);
    if (s != AK_OK) return s;
    uint64_t word = 0;
    cudaError_t e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return word == c.epoch ? AK_ERR_TIMEOUT : AK_OK;
}

extern "C" ak_status ak_scan_status(const void* ws) {
    if (!ws || !aligned(ws, 16)) return AK_ERR_INVALID_ARG;
    // the call clears the whole header before its kernel, and a kernel that
    // gives up writes its (non-zero) epoch into the first word
    uint64_t word = 0;
    cudaError_t e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return word != 0 ? AK_ERR_TIMEOUT : AK_OK;
}

// ===========================================================================
// ak_findall
// ===========================================================================

extern "C" ak_status ak_findall_workspace_size(int64_t n, ak_dtype in, const ak_opts* opts, size_t* bytes) {
    (void)opts;
    if (!bytes || n < 0 || !valid_dtype(in)) return AK_ERR_INVALID_ARG;
    int64_t ntiles;
    size_t ws, count_off;
    ak_status s = plan_findall(n, in, &ntiles, &ws, &count_off);
    if (s != AK_OK) return s;
    *bytes = ws;
    return AK_OK;
}

extern "C" ak_status ak_findall(const void* src, int64_t n, ak_dtype in, int64_t* idx, int64_t* count_dev,
                                int64_t* count_host, void* ws, size_t ws_bytes, const ak_opts* opts,
                                void* stream) {
    if (!valid_dtype(in) || n < 0 || (!count_dev && !count_host)) return AK_ERR_INVALID_ARG;
    int64_t ntiles;
    size_t need, count_off;
    ak_status s = plan_findall(n, in, &ntiles, &need, &count_off);
    if (s != AK_OK) return s;
    const size_t esz = ak_dtype_size(in);
    if (n > 0 && (!src || !idx || !aligned(src, esz) || !aligned(idx, 8))) return AK_ERR_INVALID_ARG;
    if (count_dev && !aligned(count_dev, 8)) return AK_ERR_INVALID_ARG;
    const ak_opts o = resolve_opts(opts);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (count_host) *count_host = 0;
        if (count_dev) {
            Value16 zero;
            memset(zero.b, 0, sizeof zero.b);
            s = run_fill(count_dev, 1, AK_I64, zero, st);
            if (s == AK_OK && o.check) s = sync_and_check(st);
            return s;
        }
        return AK_OK;
    }
    if (!ws || ws_bytes < need || !aligned(ws, 16)) return AK_ERR_WORKSPACE;
    int64_t* count = count_dev ? count_dev : reinterpret_cast<int64_t*>(static_cast<char*>(ws) + count_off);
    const uint64_t epoch = next_epoch();
    if (log_on())
        log_call("findall n=%lld in=%s: single pass, %lld tile(s), count to %s", (long long)n, dtype_name(in),
                 (long long)ntiles, count_host ? "host" : "device");
    s = run_findall(src, n, in, idx, count, ws, ntiles, need, epoch, o.wait_limit_ns, o.debug_skip_publish_tile,
                    o.target_blocks, st);
    if (s != AK_OK) return s;
    if (count_host) {
        cudaError_t e = cudaMemcpyAsync(count_host, count, sizeof(int64_t), cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (!count_host && !o.check) return AK_OK;
    s = sync_and_check(st);
    if (s != AK_OK || !o.check) return s;
    uint64_t word = 0;
    cudaError_t e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    return word == epoch ? AK_ERR_TIMEOUT : AK_OK;
}
