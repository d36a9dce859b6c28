// sdc_internal.cuh -- structures and device helpers shared by libsdc's
// translation units.  Not part of the public ABI (see include/sdc.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#include <string>
#include <vector>

#include "../../include/sdc.h"

namespace sdc {

// ---------------------------------------------------------------------------
// Device tables
// ---------------------------------------------------------------------------

// One warp task: a run of at most chunk_bytes bytes of one tensor copy.
// Interior chunk boundaries sit on absolute multiples of chunk_bytes, so every
// chunk except a tensor's first and last starts and ends 16-byte aligned.
struct Chunk {
    uint64_t addr;    // absolute device byte address of the chunk's first element
    uint32_t nbytes;  // bytes in the chunk, a multiple of the element size
    uint32_t tag;     // bits 0..27 descriptor index, 28..29 log2(elem size), 30..31 dtype
};
static_assert(sizeof(Chunk) == 16, "Chunk is 16 bytes");

constexpr uint32_t kDescBits = 28;
constexpr uint32_t kMaxDescs = 1u << kDescBits;

__host__ __device__ inline uint32_t chunk_desc(uint32_t tag) { return tag & (kMaxDescs - 1); }
__host__ __device__ inline uint32_t chunk_log2es(uint32_t tag) { return (tag >> 28) & 3u; }
__host__ __device__ inline uint32_t chunk_dtype(uint32_t tag) { return tag >> 30; }
__host__ __device__ inline uint32_t make_tag(uint32_t desc, uint32_t log2es, uint32_t dtype) {
    return desc | (log2es << 28) | (dtype << 30);
}

// Descriptor as the combine kernels see it.
struct DescDev {
    uint64_t ptr;          // device address of element 0
    uint64_t first_chunk;  // index of the descriptor's first chunk
    uint32_t n_chunks;     // chunks of this descriptor (0 when numel == 0)
    uint32_t log2es;       // log2(elem size)
};
static_assert(sizeof(DescDev) == 24, "DescDev is 24 bytes");

// Per-chunk partial of the fingerprint pass.
struct FpPartial {
    uint64_t s;  // sum of widened bits
    uint64_t w;  // sum of (local index + 1) * bits, local index from the chunk start
};

// Per-chunk (or per-stream) partial of a gradient scan.
struct StatPartial {
    double sumsq;  // sum of x^2 over finite elements
    uint32_t n_nan;
    uint32_t n_inf;
    uint32_t n_big;
    uint32_t pad;
};
static_assert(sizeof(StatPartial) == 24, "StatPartial is 24 bytes");

// One of the statistics combine's fixed groups: counts in 64 bits (a group
// may cover more than 2^32 elements of one stream).
struct StatGroup {
    double sumsq;
    uint64_t n_nan;
    uint64_t n_inf;
    uint64_t n_big;
};
static_assert(sizeof(StatGroup) == 32, "StatGroup is 32 bytes");

}  // namespace sdc

// The plan (opaque to callers).
struct sdc_plan {
    int device = -1;
    uint32_t T = 0, R = 0;
    uint32_t chunk_bytes = 0;
    uint64_t n_desc = 0;
    uint64_t n_chunks = 0;
    uint32_t grid = 0, block = 0;
    bool all_float = false;                 // every descriptor has a float dtype
    std::vector<sdc_tensor_desc> descs;     // host copy
    std::vector<uint64_t> replica_numel;    // elements per replica
    std::vector<uint64_t> replica_first_chunk;  // R + 1 entries
    sdc::Chunk *d_chunks = nullptr;
    sdc::DescDev *d_descs = nullptr;
    uint64_t *d_replica_first_chunk = nullptr;  // R + 1
    uint64_t *d_replica_numel = nullptr;        // R
};

namespace sdc {

// ---------------------------------------------------------------------------
// Host-side helpers (sdc_api.cu)
// ---------------------------------------------------------------------------
void set_error(const std::string &msg);
sdc_status fail(sdc_status st, const std::string &msg);
sdc_status cuda_fail(cudaError_t e, const char *what);
sdc_status check_plan_device(const sdc_plan *plan);
// Check [ptr, ptr + bytes) is device memory of `device` inside one allocation.
sdc_status check_device_range(const void *ptr, uint64_t bytes, int device, const char *what);
// One array a call reads or writes; ptr may be NULL only when bytes == 0.
struct DevSpan {
    const void *ptr;
    uint64_t bytes;
    const char *what;
};
// check_device_range for each span in order; the first failure is returned.
sdc_status check_spans(std::initializer_list<DevSpan> spans, int device);
// sdc_grad_average_scan; ws_is_scratch skips the workspace's range query (the
// no-allocation entry point passes this library's own static scratch).
sdc_status grad_average_scan(const void *const *bufs, uint32_t n_bufs, void *d_avg, uint64_t numel, uint32_t dtype,
                             sdc_grad_stats *d_pre, sdc_grad_stats *d_post, void *d_ws, size_t ws_bytes,
                             bool ws_is_scratch, sdc_stream_t stream);
int sm_count(int device);

// Launchers (one per translation unit that holds the kernel).
cudaError_t launch_fp_scan(const sdc_plan *plan, FpPartial *partials, cudaStream_t st);
cudaError_t launch_fp_combine(const sdc_plan *plan, const FpPartial *partials, uint64_t *out,
                              cudaStream_t st);
cudaError_t launch_xor_scan(const sdc_plan *plan, uint64_t *partials, cudaStream_t st);
cudaError_t launch_xor_combine(const sdc_plan *plan, const uint64_t *partials, uint64_t *out,
                               cudaStream_t st);
cudaError_t launch_grad_scan(const sdc_plan *plan, StatPartial *partials, cudaStream_t st);
cudaError_t launch_stats_combine_plan(const sdc_plan *plan, const StatPartial *partials, StatGroup *groups,
                                      sdc_grad_stats *out, cudaStream_t st);
cudaError_t launch_avg_scan(const void *const *bufs, uint32_t n_bufs, void *avg, uint64_t numel,
                            uint32_t dtype, StatPartial *partials, uint64_t n_chunks, bool vector_path,
                            int device, cudaStream_t st);
cudaError_t launch_stats_combine_streams(const StatPartial *partials, StatGroup *groups, uint32_t n_streams,
                                         uint64_t n_chunks, uint64_t numel, sdc_grad_stats *out_pre,
                                         sdc_grad_stats *out_post, cudaStream_t st);
cudaError_t launch_vote(const uint64_t *fp, uint32_t R, uint32_t T, int32_t *suspect, uint64_t *mask,
                        sdc_vote_summary *summary, cudaStream_t st);
cudaError_t launch_ring_audit(const uint64_t *table, uint32_t n, uint32_t L, uint32_t offset, uint8_t *mismatch,
                              uint32_t *hits, uint8_t *culprit, uint8_t *ambiguous, sdc_ring_summary *summary,
                              int device, cudaStream_t st);
cudaError_t launch_xor_compare(const uint64_t *a, const uint64_t *b, uint32_t n, uint8_t *mismatch,
                               uint64_t *diff, cudaStream_t st);

// Persistent-kernel block size and per-SM occupancy of the scan kernels.
constexpr int kScanBlock = 256;
int fp_scan_blocks_per_sm();
int grad_scan_blocks_per_sm();

// Bytes of one warp task in the fused average scan (per stream).
constexpr uint64_t kAvgChunkBytes = 16384;
// Fixed number of first-pass groups per stream in the statistics combine.
constexpr uint32_t kStatGroups = 128;

}  // namespace sdc

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
namespace sdc {

// Streaming 16-byte load: read-only path, no L1 allocation, 256-byte L2 fetch.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// L2 eviction policies for ld_stream_hint: evict_first for data read once
// (its lines are the first the L2 gives up), evict_normal for data read again.
__device__ __forceinline__ uint64_t l2_policy(bool read_once) {
    uint64_t p;
    if (read_once)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ld_stream with an L2 eviction policy from l2_policy.
__device__ __forceinline__ uint4 ld_stream_hint(const void *p, uint64_t policy) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(policy));
    return r;
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a
// multiple of 16); no data is returned and no completion is tracked.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch the line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Two-way 16x8-bit dot product with 32-bit accumulate, both halves signed.
__device__ __forceinline__ int dp2a_lo_s(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi_s(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Four-way 8x8-bit unsigned dot product with 32-bit accumulate.
__device__ __forceinline__ uint32_t dp4a_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Packed pair of float32 in one 64-bit register (low word = first element).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ uint64_t f2_pack_bits(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Error-free accumulation of a non-negative term on both lanes:
// s + y = s' + err exactly, and err is added to the compensation c.
// Dekker's Fast2Sum (s' = a + b, err = b - (s' - a)) is exact when |a| >= |b|;
// with s, y >= 0 the larger of the two is the larger bit pattern, so the
// ordering is two integer max/min per lane (integer pipe) and the floating
// point cost is four packed operations instead of TwoSum's seven.
// Requires s >= 0 and y >= 0 (NaN/Inf propagate into s).
__device__ __forceinline__ void f2_two_sum_acc(uint64_t &s, uint64_t &c, uint64_t y) {
    const uint32_t s0 = (uint32_t)s, s1 = (uint32_t)(s >> 32), y0 = (uint32_t)y, y1 = (uint32_t)(y >> 32);
    const uint64_t big = f2_pack_bits(max(s0, y0), max(s1, y1));
    const uint64_t small = f2_pack_bits(min(s0, y0), min(s1, y1));
    const uint64_t s2 = f2_add(big, small);
    const uint64_t err = f2_sub(small, f2_sub(s2, big));
    c = f2_add(c, err);
    s = s2;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ uint64_t warp_xor_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v ^= __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Fixed-shape butterfly: every lane ends with the same value, bit for bit.
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- mbarriers
// Shared-memory barriers that TMA copies and tcgen05.commit signal.  Every
// wait is bounded: after kSpinLimit polls the caller records an error and
// stops, so no kernel can hang on a barrier.
// A poll that finds the phase incomplete suspends the thread for ~3.76 us on
// GB300 (measured with sdc_selftest_bounded_wait), so 2^18 polls give up after
// about one second: far longer than any wait of these kernels (at most one
// tile's main loop, milliseconds), short enough to end a stall promptly.
constexpr uint32_t kSpinLimit = 1u << 18;

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    return done != 0;
}
// Bounded wait for the completion of phase `parity` of a barrier: at most
// `limit` polls (kSpinLimit unless given); false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, uint32_t limit = kSpinLimit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(mbar, parity)) return true;
    return false;
}

}  // namespace sdc

#endif  // __CUDACC__
