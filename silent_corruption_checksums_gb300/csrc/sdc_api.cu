// sdc_api.cu -- the C ABI of libsdc: argument validation, the plan (descriptor
// and chunk tables), workspace sizing and the launch sequence of every call.
// The declarations and their contracts are in include/sdc.h.
#include <cuda.h>  // driver types for the pointer-attribute query (no libcuda link)

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "sdc_internal.cuh"

namespace sdc {

// ---------------------------------------------------------------- errors
static thread_local std::string g_last_error;

void set_error(const std::string &msg) { g_last_error = msg; }

sdc_status fail(sdc_status st, const std::string &msg) {
    set_error(msg);
    return st;
}

sdc_status cuda_fail(cudaError_t e, const char *what) {
    return fail(SDC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

int sm_count(int device) {
    static std::mutex mu;
    static int cached[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return 1;
    if (cached[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 1;
        cached[device] = n;
    }
    return cached[device];
}

// ---------------------------------------------------------------- pointer checks
namespace {

typedef CUresult (*PFN_getattr)(void *data, CUpointer_attribute attribute, CUdeviceptr ptr);

PFN_getattr pointer_attr_fn() {
    static std::once_flag once;
    static PFN_getattr fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_getattr)p;
    });
    return fn;
}

}  // namespace

sdc_status check_device_range(const void *ptr, uint64_t bytes, int device, const char *what) {
    if (bytes == 0) return SDC_OK;
    if (!ptr) return fail(SDC_ERR_NULL, std::string(what) + ": NULL pointer with non-zero size");
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SDC_ERR_BAD_POINTER, std::string(what) + ": not a CUDA pointer");
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fail(SDC_ERR_BAD_POINTER, std::string(what) + ": not device memory");
    if (at.device != device)
        return fail(SDC_ERR_BAD_POINTER, std::string(what) + ": memory of device " + std::to_string(at.device) +
                                             ", current device is " + std::to_string(device));
    PFN_getattr fn = pointer_attr_fn();
    if (fn) {
        CUdeviceptr start = 0;
        size_t size = 0;
        if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, (CUdeviceptr)ptr) == CUDA_SUCCESS &&
            fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, (CUdeviceptr)ptr) == CUDA_SUCCESS && size > 0) {
            const uint64_t p = (uint64_t)ptr;
            if (p + bytes < p || p + bytes > (uint64_t)start + size)
                return fail(SDC_ERR_BAD_POINTER, std::string(what) + ": range of " + std::to_string(bytes) +
                                                     " bytes leaves its allocation");
        }
    }
    return SDC_OK;
}

sdc_status check_spans(std::initializer_list<DevSpan> spans, int device) {
    for (const DevSpan &sp : spans) {
        const sdc_status st = check_device_range(sp.ptr, sp.bytes, device, sp.what);
        if (st != SDC_OK) return st;
    }
    return SDC_OK;
}

sdc_status check_plan_device(const sdc_plan *plan) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != plan->device)
        return fail(SDC_ERR_WRONG_DEVICE, "plan built on device " + std::to_string(plan->device) +
                                              ", current device is " + std::to_string(dev));
    return SDC_OK;
}

namespace {

uint32_t log2_of(uint32_t es) { return es == 1 ? 0 : es == 2 ? 1 : es == 4 ? 2 : 3; }

bool valid_esize(uint32_t es) { return es == 1 || es == 2 || es == 4 || es == 8; }

bool dtype_matches(uint32_t dtype, uint32_t es) {
    switch (dtype) {
        case SDC_DTYPE_RAW: return true;
        case SDC_DTYPE_F32: return es == 4;
        case SDC_DTYPE_BF16:
        case SDC_DTYPE_F16: return es == 2;
        default: return false;
    }
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

void free_plan_tables(sdc_plan *p) {
    if (p->d_chunks) cudaFree(p->d_chunks);
    if (p->d_descs) cudaFree(p->d_descs);
    if (p->d_replica_first_chunk) cudaFree(p->d_replica_first_chunk);
    if (p->d_replica_numel) cudaFree(p->d_replica_numel);
    p->d_chunks = nullptr;
    p->d_descs = nullptr;
    p->d_replica_first_chunk = nullptr;
    p->d_replica_numel = nullptr;
}

template <typename T>
cudaError_t upload(T **dst, const std::vector<T> &src) {
    if (src.empty()) return cudaSuccess;
    cudaError_t e = cudaMalloc((void **)dst, src.size() * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
}

// device < 0: the workspace is this library's own static scratch (no range query).
sdc_status check_ws(const void *ws, size_t ws_bytes, size_t need, int device) {
    if (need == 0) return SDC_OK;
    if (!ws) return fail(SDC_ERR_NULL, "workspace is NULL");
    if (ws_bytes < need)
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace of " + std::to_string(ws_bytes) + " bytes, need " +
                                              std::to_string(need));
    if (((uint64_t)ws & 255u) != 0) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    return device < 0 ? SDC_OK : check_device_range(ws, need, device, "d_ws");
}

// Workspace: per-chunk partials, then the statistics combine's group sums.
size_t plan_partials_bytes(const sdc_plan *p) { return round_up((size_t)p->n_chunks * sizeof(StatPartial), 256); }
size_t plan_ws_bytes(const sdc_plan *p) {
    return plan_partials_bytes(p) + round_up((size_t)p->R * kStatGroups * sizeof(StatGroup), 256);
}

size_t avg_chunks(uint64_t numel, uint32_t dtype) {
    const uint64_t es = dtype == SDC_DTYPE_F32 ? 4 : 2;
    return (size_t)((numel * es + kAvgChunkBytes - 1) / kAvgChunkBytes);
}

}  // namespace
}  // namespace sdc

using namespace sdc;

// ---------------------------------------------------------------- ABI
extern "C" {

const char *sdc_status_string(sdc_status s) {
    switch (s) {
        case SDC_OK: return "SDC_OK";
        case SDC_ERR_NULL: return "SDC_ERR_NULL";
        case SDC_ERR_BAD_ELEM_SIZE: return "SDC_ERR_BAD_ELEM_SIZE";
        case SDC_ERR_SHAPE_MISMATCH: return "SDC_ERR_SHAPE_MISMATCH";
        case SDC_ERR_TOO_MANY_REPLICAS: return "SDC_ERR_TOO_MANY_REPLICAS";
        case SDC_ERR_WS_TOO_SMALL: return "SDC_ERR_WS_TOO_SMALL";
        case SDC_ERR_CUDA: return "SDC_ERR_CUDA";
        case SDC_ERR_BAD_DTYPE: return "SDC_ERR_BAD_DTYPE";
        case SDC_ERR_BAD_POINTER: return "SDC_ERR_BAD_POINTER";
        case SDC_ERR_BAD_ARG: return "SDC_ERR_BAD_ARG";
        case SDC_ERR_WRONG_DEVICE: return "SDC_ERR_WRONG_DEVICE";
        default: return "SDC_ERR_UNKNOWN";
    }
}

const char *sdc_last_error(void) { return g_last_error.c_str(); }

sdc_status sdc_plan_create(const sdc_tensor_desc *host_descs, uint32_t T, uint32_t R, const sdc_plan_opts *opts,
                           sdc_plan **out) {
    if (!out) return fail(SDC_ERR_NULL, "out is NULL");
    *out = nullptr;
    if (R == 0 || R > SDC_MAX_REPLICAS)
        return fail(SDC_ERR_TOO_MANY_REPLICAS, "R = " + std::to_string(R) + ", must be 1..64");
    const uint64_t n_desc = (uint64_t)R * T;
    if (n_desc >= kMaxDescs) return fail(SDC_ERR_BAD_ARG, "R * T too large");
    if (n_desc && !host_descs) return fail(SDC_ERR_NULL, "host_descs is NULL");

    uint32_t chunk_bytes = 0;  // 0: chosen below from the plan's size
    uint32_t ctas_per_sm = 0;
    bool check_ptrs = true;
    if (opts) {
        chunk_bytes = opts->chunk_bytes;
        ctas_per_sm = opts->ctas_per_sm;
        check_ptrs = opts->skip_pointer_checks == 0;
    }
    const bool auto_chunk = chunk_bytes == 0;
    if (auto_chunk) chunk_bytes = 16384;
    if (chunk_bytes < 4096 || chunk_bytes > 32768 || (chunk_bytes & (chunk_bytes - 1)))
        return fail(SDC_ERR_BAD_ARG, "chunk_bytes must be a power of two in [4096, 32768]");

    // descriptor validation (host only; runs before any CUDA call)
    bool all_float = true;
    for (uint64_t d = 0; d < n_desc; ++d) {
        const sdc_tensor_desc &x = host_descs[d];
        const uint64_t k = d % T;
        const sdc_tensor_desc &ref = host_descs[k];
        if (!valid_esize(x.elem_size))
            return fail(SDC_ERR_BAD_ELEM_SIZE, "descriptor " + std::to_string(d) + ": elem_size " +
                                                   std::to_string(x.elem_size));
        if (x.dtype > SDC_DTYPE_F16) return fail(SDC_ERR_BAD_DTYPE, "descriptor " + std::to_string(d) + ": dtype");
        if (!dtype_matches(x.dtype, x.elem_size))
            return fail(SDC_ERR_BAD_ELEM_SIZE, "descriptor " + std::to_string(d) + ": elem_size does not match dtype");
        if (x.numel != ref.numel || x.elem_size != ref.elem_size || x.dtype != ref.dtype)
            return fail(SDC_ERR_SHAPE_MISMATCH, "replica " + std::to_string(d / T) + " of tensor " +
                                                    std::to_string(k) + " differs from replica 0");
        if (x.dtype == SDC_DTYPE_RAW) all_float = false;
        if (x.numel) {
            if (!x.ptr) return fail(SDC_ERR_NULL, "descriptor " + std::to_string(d) + ": NULL ptr");
            if ((uint64_t)x.ptr % x.elem_size)
                return fail(SDC_ERR_BAD_POINTER, "descriptor " + std::to_string(d) + ": ptr not aligned to elem_size");
            if (x.numel > (~0ull) / x.elem_size || (uint64_t)x.ptr + x.numel * x.elem_size < (uint64_t)x.ptr)
                return fail(SDC_ERR_BAD_ARG, "descriptor " + std::to_string(d) + ": size overflows");
        }
    }

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");

    // The default chunk: 16 KiB, halved (down to 4 KiB) while the plan would give fewer than 16 warp
    // tasks per warp of the persistent grid (32 warps per SM), so that a small plan still spreads
    // evenly over the SMs (its last wave of tasks is then a small part of the pass).
    if (auto_chunk) {
        uint64_t total = 0;
        for (uint64_t d = 0; d < n_desc; ++d) total += host_descs[d].numel * host_descs[d].elem_size;
        const uint64_t want = 16ull * 32ull * (uint64_t)sm_count(dev);
        while (chunk_bytes > 4096 && total / chunk_bytes < want) chunk_bytes >>= 1;
    }

    // every descriptor's byte range must lie in one allocation of this device;
    // ranges already proven by an earlier query are reused (sorted scan)
    if (check_ptrs && n_desc) {
        std::vector<uint64_t> order;
        order.reserve(n_desc);
        for (uint64_t d = 0; d < n_desc; ++d)
            if (host_descs[d].numel) order.push_back(d);
        std::sort(order.begin(), order.end(),
                  [&](uint64_t a, uint64_t b) { return (uint64_t)host_descs[a].ptr < (uint64_t)host_descs[b].ptr; });
        PFN_getattr fn = pointer_attr_fn();
        uint64_t known_lo = 1, known_hi = 0;  // empty
        for (uint64_t d : order) {
            const uint64_t p = (uint64_t)host_descs[d].ptr;
            const uint64_t bytes = host_descs[d].numel * host_descs[d].elem_size;
            if (p >= known_lo && p + bytes <= known_hi) continue;
            std::string what = "descriptor " + std::to_string(d);
            sdc_status st = check_device_range(host_descs[d].ptr, bytes, dev, what.c_str());
            if (st != SDC_OK) return st;
            known_lo = 1;
            known_hi = 0;
            if (fn) {
                CUdeviceptr start = 0;
                size_t size = 0;
                if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, (CUdeviceptr)p) == CUDA_SUCCESS &&
                    fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, (CUdeviceptr)p) == CUDA_SUCCESS && size > 0) {
                    known_lo = start;
                    known_hi = start + size;
                }
            }
        }
    }

    sdc_plan *p = new (std::nothrow) sdc_plan();
    if (!p) return fail(SDC_ERR_BAD_ARG, "out of host memory");
    p->device = dev;
    p->T = T;
    p->R = R;
    p->chunk_bytes = chunk_bytes;
    p->n_desc = n_desc;
    p->all_float = all_float;
    p->descs.assign(host_descs, host_descs + n_desc);

    // chunk table: interior boundaries on absolute multiples of chunk_bytes
    std::vector<Chunk> chunks;
    std::vector<DescDev> dd(n_desc);
    p->replica_numel.assign(R, 0);
    p->replica_first_chunk.assign(R + 1, 0);
    uint64_t total_chunks = 0;
    for (uint64_t d = 0; d < n_desc; ++d) {
        const sdc_tensor_desc &x = host_descs[d];
        if (x.numel == 0) continue;
        const uint64_t a = (uint64_t)x.ptr, end = a + x.numel * x.elem_size;
        total_chunks += (end - 1) / chunk_bytes - a / chunk_bytes + 1;
    }
    try {
        chunks.reserve(total_chunks);
    } catch (...) {
        delete p;
        return fail(SDC_ERR_BAD_ARG, "out of host memory for the chunk table");
    }
    for (uint64_t d = 0; d < n_desc; ++d) {
        const sdc_tensor_desc &x = host_descs[d];
        const uint32_t r = (uint32_t)(d / T);
        if (d % T == 0) p->replica_first_chunk[r] = chunks.size();
        const uint32_t l2 = log2_of(x.elem_size);
        dd[d].ptr = (uint64_t)x.ptr;
        dd[d].first_chunk = chunks.size();
        dd[d].log2es = l2;
        p->replica_numel[r] += x.numel;
        if (x.numel) {
            const uint64_t a = (uint64_t)x.ptr, end = a + x.numel * x.elem_size;
            uint64_t c0 = a;
            while (c0 < end) {
                uint64_t c1 = (c0 / chunk_bytes + 1) * chunk_bytes;
                if (c1 > end) c1 = end;
                chunks.push_back(Chunk{c0, (uint32_t)(c1 - c0), make_tag((uint32_t)d, l2, x.dtype)});
                c0 = c1;
            }
        }
        dd[d].n_chunks = (uint32_t)(chunks.size() - dd[d].first_chunk);
    }
    p->replica_first_chunk[R] = chunks.size();
    p->n_chunks = chunks.size();

    e = upload(&p->d_chunks, chunks);
    if (e == cudaSuccess) e = upload(&p->d_descs, dd);
    if (e == cudaSuccess) e = upload(&p->d_replica_first_chunk, p->replica_first_chunk);
    if (e == cudaSuccess) e = upload(&p->d_replica_numel, p->replica_numel);
    if (e != cudaSuccess) {
        free_plan_tables(p);
        delete p;
        return cuda_fail(e, "plan tables");
    }

    // persistent grid: every SM filled to the scan kernel's occupancy
    int per_sm = fp_scan_blocks_per_sm();
    if (ctas_per_sm && (int)ctas_per_sm < per_sm) per_sm = (int)ctas_per_sm;
    uint64_t grid = (uint64_t)sm_count(dev) * per_sm;
    const uint64_t need = (p->n_chunks * 32 + kScanBlock - 1) / kScanBlock;
    if (need < grid) grid = need ? need : 1;
    p->grid = (uint32_t)grid;
    p->block = kScanBlock;
    *out = p;
    return SDC_OK;
}

sdc_status sdc_plan_destroy(sdc_plan *plan) {
    if (!plan) return SDC_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != plan->device) cudaSetDevice(plan->device);
    free_plan_tables(plan);
    if (cur != plan->device && cur >= 0) cudaSetDevice(cur);
    delete plan;
    return SDC_OK;
}

size_t sdc_workspace_size(const sdc_plan *plan) { return plan ? plan_ws_bytes(plan) : 0; }

sdc_status sdc_plan_info(const sdc_plan *plan, uint64_t *n_chunks, uint32_t *grid, uint32_t *block) {
    if (!plan) return fail(SDC_ERR_NULL, "plan is NULL");
    if (n_chunks) *n_chunks = plan->n_chunks;
    if (grid) *grid = plan->grid;
    if (block) *block = plan->block;
    return SDC_OK;
}

sdc_status sdc_fingerprint(const sdc_plan *plan, uint64_t *d_out, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    if (!plan) return fail(SDC_ERR_NULL, "plan is NULL");
    sdc_status st = check_plan_device(plan);
    if (st != SDC_OK) return st;
    if (plan->n_desc && !d_out) return fail(SDC_ERR_NULL, "d_out is NULL");
    st = check_device_range(d_out, plan->n_desc * 16, plan->device, "d_out");
    if (st == SDC_OK) st = check_ws(d_ws, ws_bytes, plan_ws_bytes(plan), plan->device);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    FpPartial *part = (FpPartial *)d_ws;
    cudaError_t e = launch_fp_scan(plan, part, s);
    if (e == cudaSuccess) e = launch_fp_combine(plan, part, d_out, s);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_fingerprint launch");
}

sdc_status sdc_xorsum(const sdc_plan *plan, uint64_t *d_out, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    if (!plan) return fail(SDC_ERR_NULL, "plan is NULL");
    sdc_status st = check_plan_device(plan);
    if (st != SDC_OK) return st;
    if (plan->n_desc && !d_out) return fail(SDC_ERR_NULL, "d_out is NULL");
    st = check_device_range(d_out, plan->n_desc * 8, plan->device, "d_out");
    if (st == SDC_OK) st = check_ws(d_ws, ws_bytes, plan_ws_bytes(plan), plan->device);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    uint64_t *part = (uint64_t *)d_ws;
    cudaError_t e = launch_xor_scan(plan, part, s);
    if (e == cudaSuccess) e = launch_xor_combine(plan, part, d_out, s);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_xorsum launch");
}

sdc_status sdc_xorsum_compare(const uint64_t *d_a, const uint64_t *d_b, uint32_t n, uint8_t *d_mismatch,
                              uint64_t *d_diff, sdc_stream_t stream) {
    if (n == 0) return SDC_OK;
    if (!d_a || !d_b || !d_mismatch) return fail(SDC_ERR_NULL, "NULL input or output");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const sdc_status st = check_spans({{d_a, (uint64_t)n * 8, "d_a"},
                                       {d_b, (uint64_t)n * 8, "d_b"},
                                       {d_mismatch, n, "d_mismatch"},
                                       {d_diff, d_diff ? (uint64_t)n * 8 : 0, "d_diff"}},
                                      dev);
    if (st != SDC_OK) return st;
    e = launch_xor_compare(d_a, d_b, n, d_mismatch, d_diff, (cudaStream_t)stream);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_xorsum_compare launch");
}

sdc_status sdc_vote(const uint64_t *d_fp, uint32_t R, uint32_t T, int32_t *d_suspect, uint64_t *d_mask,
                    sdc_vote_summary *d_summary, sdc_stream_t stream) {
    if (R == 0 || R > SDC_MAX_REPLICAS)
        return fail(SDC_ERR_TOO_MANY_REPLICAS, "R = " + std::to_string(R) + ", must be 1..64");
    if (!d_summary) return fail(SDC_ERR_NULL, "d_summary is NULL");
    if (T && (!d_fp || !d_suspect || !d_mask)) return fail(SDC_ERR_NULL, "NULL table or output");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const sdc_status st = check_spans({{d_fp, (uint64_t)R * T * 16, "d_fp"},
                                       {d_suspect, (uint64_t)T * 4, "d_suspect"},
                                       {d_mask, (uint64_t)T * 8, "d_mask"},
                                       {d_summary, sizeof(sdc_vote_summary), "d_summary"}},
                                      dev);
    if (st != SDC_OK) return st;
    e = launch_vote(d_fp, R, T, d_suspect, d_mask, d_summary, (cudaStream_t)stream);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_vote launch");
}

sdc_status sdc_grad_scan(const sdc_plan *plan, sdc_grad_stats *d_stats, void *d_ws, size_t ws_bytes,
                         sdc_stream_t stream) {
    if (!plan) return fail(SDC_ERR_NULL, "plan is NULL");
    sdc_status st = check_plan_device(plan);
    if (st != SDC_OK) return st;
    if (!d_stats) return fail(SDC_ERR_NULL, "d_stats is NULL");
    if (!plan->all_float) return fail(SDC_ERR_BAD_DTYPE, "sdc_grad_scan needs F32, BF16 or F16 descriptors");
    st = check_device_range(d_stats, (uint64_t)plan->R * sizeof(sdc_grad_stats), plan->device, "d_stats");
    if (st == SDC_OK) st = check_ws(d_ws, ws_bytes, plan_ws_bytes(plan), plan->device);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    StatPartial *part = (StatPartial *)d_ws;
    StatGroup *groups = (StatGroup *)((char *)d_ws + plan_partials_bytes(plan));
    cudaError_t e = launch_grad_scan(plan, part, s);
    if (e == cudaSuccess) e = launch_stats_combine_plan(plan, part, groups, d_stats, s);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_grad_scan launch");
}

size_t sdc_grad_average_scan_workspace_size(uint64_t numel, uint32_t n_bufs, uint32_t dtype) {
    if (n_bufs == 0 || n_bufs > 8) return 0;
    if (dtype != SDC_DTYPE_F32 && dtype != SDC_DTYPE_BF16 && dtype != SDC_DTYPE_F16) return 0;
    const size_t nc = avg_chunks(numel, dtype);
    return round_up(nc * (n_bufs + 1) * sizeof(StatPartial), 256) +
           round_up((size_t)(n_bufs + 1) * kStatGroups * sizeof(StatGroup), 256);
}

}  // extern "C"

// ws_is_scratch: d_ws is this library's static scratch (sdc_noalloc.cu), whose
// extent needs no range query.
sdc_status sdc::grad_average_scan(const void *const *bufs, uint32_t n_bufs, void *d_avg, uint64_t numel,
                                  uint32_t dtype, sdc_grad_stats *d_pre, sdc_grad_stats *d_post, void *d_ws,
                                  size_t ws_bytes, bool ws_is_scratch, sdc_stream_t stream) {
    if (n_bufs == 0 || n_bufs > 8) return fail(SDC_ERR_TOO_MANY_REPLICAS, "n_bufs must be 1..8");
    if (dtype != SDC_DTYPE_F32 && dtype != SDC_DTYPE_BF16 && dtype != SDC_DTYPE_F16)
        return fail(SDC_ERR_BAD_DTYPE, "dtype must be F32, BF16 or F16");
    if (!bufs || !d_pre || !d_post) return fail(SDC_ERR_NULL, "NULL bufs or stats");
    const uint64_t es = dtype == SDC_DTYPE_F32 ? 4 : 2;
    if (numel > (~0ull) / es) return fail(SDC_ERR_BAD_ARG, "numel overflows");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    bool aligned = ((uint64_t)d_avg & 15u) == 0;
    const uint64_t bytes = numel * es;
    for (uint32_t b = 0; b < n_bufs; ++b) {
        if (numel && !bufs[b]) return fail(SDC_ERR_NULL, "bufs[" + std::to_string(b) + "] is NULL");
        if ((uint64_t)bufs[b] % es) return fail(SDC_ERR_BAD_POINTER, "bufs[] not aligned to the element size");
        std::string what = "bufs[" + std::to_string(b) + "]";
        sdc_status st = check_device_range(bufs[b], bytes, dev, what.c_str());
        if (st != SDC_OK) return st;
        aligned = aligned && ((uint64_t)bufs[b] & 15u) == 0;
        const uint64_t lo = (uint64_t)bufs[b], hi = lo + bytes, olo = (uint64_t)d_avg, ohi = olo + bytes;
        if (numel && lo < ohi && olo < hi) return fail(SDC_ERR_BAD_ARG, "d_avg overlaps an input");
    }
    if ((uint64_t)d_avg % es) return fail(SDC_ERR_BAD_POINTER, "d_avg not aligned to the element size");
    sdc_status st = check_spans({{d_avg, bytes, "d_avg"},
                                 {d_pre, (uint64_t)n_bufs * sizeof(sdc_grad_stats), "d_pre"},
                                 {d_post, sizeof(sdc_grad_stats), "d_post"}},
                                dev);
    if (st != SDC_OK) return st;
    const size_t nc = avg_chunks(numel, dtype);
    st = check_ws(d_ws, ws_bytes, sdc_grad_average_scan_workspace_size(numel, n_bufs, dtype), ws_is_scratch ? -1 : dev);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    StatPartial *part = (StatPartial *)d_ws;
    StatGroup *groups = (StatGroup *)((char *)d_ws + round_up(nc * (n_bufs + 1) * sizeof(StatPartial), 256));
    e = launch_avg_scan(bufs, n_bufs, d_avg, numel, dtype, part, nc, aligned, dev, s);
    if (e == cudaSuccess) e = launch_stats_combine_streams(part, groups, n_bufs + 1, nc, numel, d_pre, d_post, s);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_grad_average_scan launch");
}

extern "C" sdc_status sdc_grad_average_scan(const void *const *bufs, uint32_t n_bufs, void *d_avg, uint64_t numel,
                                            uint32_t dtype, sdc_grad_stats *d_pre, sdc_grad_stats *d_post,
                                            void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    return sdc::grad_average_scan(bufs, n_bufs, d_avg, numel, dtype, d_pre, d_post, d_ws, ws_bytes, false, stream);
}
