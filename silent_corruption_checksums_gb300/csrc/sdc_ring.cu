// sdc_ring.cu -- the ring replay audit's table comparison and localization.
//
// "Detecting and recovering from silent data corruption on Amazon SageMaker
// HyperPod", "Check 2: Ring replay, before the optimizer step": on an audit
// step rank r recomputes the micro-batch of its target (r + offset) mod n.
// Every rank contributes a row [its own result, its replay of its target],
// each a vector of L words (loss bits and gradient fingerprints).  The pair
// (target, replayer r) mismatches when the target's own result differs from
// r's replay in any word.  A rank in two or more mismatched pairs computed
// wrong in both of its comparisons: it is the culprit; a mismatched pair
// that touches no culprit is ambiguous (either side could be wrong).
#include "sdc_internal.cuh"

namespace sdc {

namespace {

constexpr int kRingBlock = 256;

// One warp per replayer r: compare table[t][0][:] with table[r][1][:].
__global__ void __launch_bounds__(kRingBlock) ring_compare_kernel(const uint64_t *__restrict__ table, uint32_t n,
                                                                  uint32_t L, uint32_t offset,
                                                                  uint8_t *__restrict__ mismatch,
                                                                  uint32_t *__restrict__ hits) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t r = warp; r < n; r += nwarps) {
        const uint32_t t = (uint32_t)((r + offset) % n);
        const uint64_t *own = table + ((uint64_t)t * 2 + 0) * L;
        const uint64_t *rep = table + ((uint64_t)r * 2 + 1) * L;
        uint32_t diff = 0;
        for (uint32_t i = lane; i < L; i += 32) diff |= own[i] != rep[i] ? 1u : 0u;
        diff = __any_sync(0xffffffffu, diff != 0) ? 1u : 0u;
        if (lane == 0) {
            mismatch[r] = (uint8_t)diff;
            if (diff) {
                atomicAdd(hits + t, 1u);
                atomicAdd(hits + r, 1u);  // a pair (r, r) counts r twice, as a count over pair members does
            }
        }
    }
}

// One thread per rank: culprit flags, ambiguous pairs (indexed by replayer), counts.
__global__ void __launch_bounds__(kRingBlock) ring_localize_kernel(uint32_t n, uint32_t offset,
                                                                   const uint8_t *__restrict__ mismatch,
                                                                   const uint32_t *__restrict__ hits,
                                                                   uint8_t *__restrict__ culprit,
                                                                   uint8_t *__restrict__ ambiguous,
                                                                   sdc_ring_summary *__restrict__ summary) {
    const uint32_t r = blockIdx.x * kRingBlock + threadIdx.x;
    uint32_t is_pair = 0, is_culprit = 0, is_amb = 0;
    if (r < n) {
        const uint32_t t = (uint32_t)(((uint64_t)r + offset) % n);
        is_culprit = hits[r] >= 2 ? 1u : 0u;
        is_pair = mismatch[r];
        is_amb = (is_pair && hits[t] < 2 && hits[r] < 2) ? 1u : 0u;
        culprit[r] = (uint8_t)is_culprit;
        ambiguous[r] = (uint8_t)is_amb;
    }
    const uint32_t wp = __reduce_add_sync(0xffffffffu, is_pair);
    const uint32_t wc = __reduce_add_sync(0xffffffffu, is_culprit);
    const uint32_t wa = __reduce_add_sync(0xffffffffu, is_amb);
    if ((threadIdx.x & 31u) == 0) {
        if (wp) atomicAdd(&summary->n_pairs, wp);
        if (wc) atomicAdd(&summary->n_culprits, wc);
        if (wa) atomicAdd(&summary->n_ambiguous, wa);
    }
}

}  // namespace

cudaError_t launch_ring_audit(const uint64_t *table, uint32_t n, uint32_t L, uint32_t offset, uint8_t *mismatch,
                              uint32_t *hits, uint8_t *culprit, uint8_t *ambiguous, sdc_ring_summary *summary,
                              int device, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(summary, 0, sizeof(sdc_ring_summary), st);
    if (e != cudaSuccess || n == 0) return e;
    e = cudaMemsetAsync(hits, 0, (size_t)n * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    uint64_t blocks = ((uint64_t)n * 32 + kRingBlock - 1) / kRingBlock;
    const uint64_t cap = (uint64_t)sm_count(device) * 8;
    if (blocks > cap) blocks = cap;
    ring_compare_kernel<<<(unsigned)blocks, kRingBlock, 0, st>>>(table, n, L, offset, mismatch, hits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    ring_localize_kernel<<<(n + kRingBlock - 1) / kRingBlock, kRingBlock, 0, st>>>(n, offset, mismatch, hits, culprit,
                                                                                 ambiguous, summary);
    return cudaGetLastError();
}

}  // namespace sdc

extern "C" sdc_status sdc_ring_audit(const uint64_t *d_table, uint32_t n, uint32_t L, uint32_t offset,
                                     uint8_t *d_mismatch, uint32_t *d_hits, uint8_t *d_culprit,
                                     uint8_t *d_ambiguous, sdc_ring_summary *d_summary, sdc_stream_t stream) {
    if (!d_summary) return sdc::fail(SDC_ERR_NULL, "d_summary is NULL");
    if (n && (!d_mismatch || !d_hits || !d_culprit || !d_ambiguous))
        return sdc::fail(SDC_ERR_NULL, "NULL output array");
    if (n && L && !d_table) return sdc::fail(SDC_ERR_NULL, "d_table is NULL");
    if (n && L == 0) return sdc::fail(SDC_ERR_BAD_ARG, "rows of L = 0 words");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return sdc::cuda_fail(e, "cudaGetDevice");
    const sdc_status st = sdc::check_spans({{d_table, (uint64_t)n * 2 * L * 8, "d_table"},
                                            {d_mismatch, n, "d_mismatch"},
                                            {d_hits, (uint64_t)n * 4, "d_hits"},
                                            {d_culprit, n, "d_culprit"},
                                            {d_ambiguous, n, "d_ambiguous"},
                                            {d_summary, sizeof(sdc_ring_summary), "d_summary"}},
                                           dev);
    if (st != SDC_OK) return st;
    const uint32_t off = n ? offset % n : 0;
    e = sdc::launch_ring_audit(d_table, n, L, off, d_mismatch, d_hits, d_culprit, d_ambiguous, d_summary, dev,
                               (cudaStream_t)stream);
    return e == cudaSuccess ? SDC_OK : sdc::cuda_fail(e, "sdc_ring_audit launch");
}
