// sdc_noalloc.cu -- sdc_grad_average_scan_noalloc: the fused gradient
// average-and-scan with its scratch in a fixed device array of this library,
// for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option -- inside a
// host callback or a custom allocator's own hooks, in a process whose memory
// pool is owned and capped by another framework, or in a tool injected into
// someone else's training job -- still wants the check-1 scan of its gradient
// buffers.  The regular entry point needs a caller-provided workspace; this
// one uses g_noalloc_scratch below instead and allocates nothing.
//
// The scratch is a file-scope __device__ array of SDC_NOALLOC_SCRATCH_BYTES:
// every GPU that loads this library holds it until the process exits.  Host
// code cannot use the array's name as a device address (in host code it is a
// host-side shadow), so the first call on each device looks up the device
// address with cudaGetSymbolAddress, with that device current, and caches it
// together with the ID of the context it belongs to.  If that context is
// destroyed and another one made current on the device (cudaDeviceReset, or a
// primary context released and retained again), the module is loaded anew and
// the array may sit elsewhere: a call that finds a different current context
// looks the address up again instead of using the stale one.
#include <cuda.h>

#include <mutex>

#include "sdc_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SDC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct CachedAddr {
    unsigned long long ctx_id;  // 0: nothing cached
    void *addr;
};
std::mutex g_mu;
CachedAddr g_cache[kMaxDevices] = {};

typedef CUresult (*PFN_ctx_current)(CUcontext *ctx);
typedef CUresult (*PFN_ctx_id)(CUcontext ctx, unsigned long long *id);

// The unique ID of the calling thread's current context, 0 when no context is
// current or the driver cannot say (then nothing is cached: every call looks
// the address up).  Driver calls reached through the runtime's entry points.
unsigned long long current_ctx_id() {
    static std::once_flag once;
    static PFN_ctx_current get_current = nullptr;
    static PFN_ctx_id get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (PFN_ctx_current)p;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (PFN_ctx_id)p;
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on `device` (the current device) in
// the current context.
sdc_status scratch_address(int device, void **out) {
    if (device < 0 || device >= kMaxDevices)
        return sdc::fail(SDC_ERR_BAD_ARG, "device ordinal out of range for the static scratch");
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = current_ctx_id();
    if (id != 0 && g_cache[device].ctx_id == id) {
        *out = g_cache[device].addr;
        return SDC_OK;
    }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return sdc::cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_cache[device] = CachedAddr{current_ctx_id(), p};  // the lookup made the device's context current
    *out = p;
    return SDC_OK;
}

}  // namespace

extern "C" sdc_status sdc_grad_average_scan_noalloc(const void *const *bufs, uint32_t n_bufs, void *d_avg,
                                                    uint64_t numel, uint32_t dtype, sdc_grad_stats *d_pre,
                                                    sdc_grad_stats *d_post, sdc_stream_t stream) {
    if (n_bufs == 0 || n_bufs > 8) return sdc::fail(SDC_ERR_TOO_MANY_REPLICAS, "n_bufs must be 1..8");
    if (dtype != SDC_DTYPE_F32 && dtype != SDC_DTYPE_BF16 && dtype != SDC_DTYPE_F16)
        return sdc::fail(SDC_ERR_BAD_DTYPE, "dtype must be F32, BF16 or F16");
    const size_t need = sdc_grad_average_scan_workspace_size(numel, n_bufs, dtype);
    if (need > (size_t)SDC_NOALLOC_SCRATCH_BYTES)
        return sdc::fail(SDC_ERR_BAD_ARG, "numel " + std::to_string(numel) + " with " + std::to_string(n_bufs) +
                                              " buffers needs " + std::to_string(need) +
                                              " bytes of scratch; the static scratch holds " +
                                              std::to_string((size_t)SDC_NOALLOC_SCRATCH_BYTES) +
                                              " (use sdc_grad_average_scan with a workspace)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return sdc::cuda_fail(e, "cudaGetDevice");
    void *scratch = nullptr;
    sdc_status st = scratch_address(dev, &scratch);
    if (st != SDC_OK) return st;
    // Nothing in the scratch needs to start at zero: every partial and group
    // sum is written by this call before it is read.
    return sdc::grad_average_scan(bufs, n_bufs, d_avg, numel, dtype, d_pre, d_post, scratch,
                                  (size_t)SDC_NOALLOC_SCRATCH_BYTES, true, stream);
}
