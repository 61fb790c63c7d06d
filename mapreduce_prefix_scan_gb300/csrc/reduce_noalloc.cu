// reduce_noalloc.cu -- ak_reduce_noalloc: the whole-array reduction for
// callers that cannot allocate device memory at call time.
//
// Some callers cannot call cudaMalloc (or any allocating routine) when they
// need a reduction: a real-time loop that cannot afford the implicit device
// synchronisation cudaMalloc / cudaFree may perform, a process whose device
// memory is already fully reserved by another allocator (so a fresh
// cudaMalloc would fail), or code held to a fixed, up-front memory budget.
// They still own their input and output, but not a workspace. This entry
// point gives them ak_reduce with its scratch (the first pass's partial
// results and the bare result slot) in a fixed array that lives in the
// library's device image: every GPU that loads the library holds
// AK_NOALLOC_SCRATCH_BYTES of it until the process exits.
#include <mutex>

#include <cuda.h>

#include "ak_internal.h"

// The scratch itself. In host code this name is only a host-side stand-in,
// not a device address: the address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[AK_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The unique ID of the context current on this thread (driver calls reached
// through the runtime's entry-point query, so nothing links libcuda); false
// when no context is current yet or the driver lacks the query.
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        else
            cudaGetLastError();
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        else
            cudaGetLastError();
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch for the current device, looked up with
// that device current the first time and again whenever the device's context
// has changed since (a cudaDeviceReset gives the device a new context, in
// which the library's module, and so the array, sits at a new address).
ak_status scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ak::cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return AK_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long id = 0;
    if (addr[dev] && current_context_id(&id) && id == ctx_of[dev]) {
        *out = addr[dev];
        return AK_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return ak::cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    // the lookup made the device's primary context current if it was not
    if (!current_context_id(&id)) id = 0;  // unknown: looked up again on every call
    addr[dev] = id != 0 ? p : nullptr;
    ctx_of[dev] = id;
    *out = p;
    return AK_OK;
}

}  // namespace

extern "C" ak_status ak_reduce_noalloc(const void* src, int64_t n, ak_dtype in, ak_map f, ak_op op, ak_dtype acc,
                                       ak_dtype out, const void* init, ak_store mode, void* dst_dev, void* dst_host,
                                       const ak_opts* opts, void* stream) {
    void* scratch = nullptr;
    ak_status s = scratch_address(&scratch);
    if (s != AK_OK) return s;
    // Same validation, kernels and store rules as ak_reduce; a plan needing
    // more scratch than the fixed array holds is refused there with
    // AK_ERR_WORKSPACE before anything is launched.
    // A host result is copied out of the fixed array (no pinned host slot:
    // that would be an allocation).
    return ak::reduce_entry(src, nullptr, 0, n, in, f, op, acc, out, init, mode, dst_dev, dst_host, scratch,
                            (size_t)AK_NOALLOC_SCRATCH_BYTES, opts, stream, false);
}
