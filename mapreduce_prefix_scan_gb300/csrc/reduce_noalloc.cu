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

#include "ak_internal.h"

// The scratch itself. In host code this name is only a host-side stand-in,
// not a device address: the address is looked up with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[AK_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch per device, looked up once per device
// with that device current (the lookup is what the first call does).
ak_status scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ak::cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return AK_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return ak::cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        addr[dev] = p;
    }
    *out = addr[dev];
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
    return ak_reduce(src, n, in, f, op, acc, out, init, mode, dst_dev, dst_host, scratch,
                     (size_t)AK_NOALLOC_SCRATCH_BYTES, opts, stream);
}
