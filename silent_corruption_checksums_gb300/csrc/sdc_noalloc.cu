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
// address with cudaGetSymbolAddress, with that device current, and caches it.
#include <mutex>

#include "sdc_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SDC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on `device` (the current device).
sdc_status scratch_address(int device, void **out) {
    if (device < 0 || device >= kMaxDevices)
        return sdc::fail(SDC_ERR_BAD_ARG, "device ordinal out of range for the static scratch");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return sdc::cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
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
