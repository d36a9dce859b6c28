// sdc_vote.cu -- strict-majority vote over a fingerprint table, and the
// element-wise xorsum comparison.
//
// Vote: "Detecting and recovering from silent data corruption on Amazon
// SageMaker HyperPod", "Check 3: Weight fingerprints, after the optimizer
// step": per tensor, if the copies differ, the most common fingerprint is a
// majority only when more than half of the copies hold it; copies that differ
// from it are suspects.  With two copies or a split without a strict majority
// the disagreement is reported without naming a copy, and the page's result
// then has no suspects at all.
#include "sdc_internal.cuh"

namespace sdc {

namespace {

constexpr int kVoteBlock = 256;

// One thread per tensor.  The table is [R][T][2]: replica r's (S, W) of
// tensor k at fp[(r * T + k) * 2].  A value held by more than R/2 copies is
// unique, so the first copy found with a strict majority count is it.
__global__ void __launch_bounds__(kVoteBlock) vote_kernel(const uint64_t *__restrict__ fp, uint32_t R, uint32_t T,
                                                          int32_t *__restrict__ suspect, uint64_t *__restrict__ mask,
                                                          sdc_vote_summary *__restrict__ summary) {
    const uint32_t k = blockIdx.x * kVoteBlock + threadIdx.x;
    uint64_t my_mask = 0;
    uint32_t differs = 0, no_major = 0;
    if (k < T) {
        const ulonglong2 *tab = (const ulonglong2 *)fp;
        const ulonglong2 first = tab[k];
        bool all_eq = true;
        for (uint32_t r = 1; r < R; ++r) {
            const ulonglong2 v = tab[(uint64_t)r * T + k];
            all_eq = all_eq && v.x == first.x && v.y == first.y;
        }
        int32_t code = SDC_SUSPECT_AGREE;
        uint64_t m = 0;
        if (!all_eq) {
            differs = 1;
            int32_t major = -1;
            for (uint32_t r = 0; r < R && major < 0; ++r) {
                const ulonglong2 v = tab[(uint64_t)r * T + k];
                uint32_t cnt = 0;
                for (uint32_t q = 0; q < R; ++q) {
                    const ulonglong2 w = tab[(uint64_t)q * T + k];
                    cnt += (w.x == v.x && w.y == v.y) ? 1u : 0u;
                }
                if (2u * cnt > R) major = (int32_t)r;
            }
            if (major < 0) {
                code = SDC_SUSPECT_NO_MAJORITY;
                no_major = 1;
            } else {
                const ulonglong2 mv = tab[(uint64_t)major * T + k];
                for (uint32_t r = 0; r < R; ++r) {
                    const ulonglong2 v = tab[(uint64_t)r * T + k];
                    if (v.x != mv.x || v.y != mv.y) m |= 1ull << r;
                }
                code = (__popcll(m) == 1) ? (int32_t)(__ffsll((long long)m) - 1) : SDC_SUSPECT_SEVERAL;
                my_mask = m;
            }
        }
        suspect[k] = code;
        mask[k] = m;
    }
    // block-wide reduction, then one set of atomics per block (results are
    // order-independent: OR and integer add)
    __shared__ unsigned long long s_mask;
    __shared__ unsigned int s_diff, s_nomaj;
    if (threadIdx.x == 0) {
        s_mask = 0;
        s_diff = 0;
        s_nomaj = 0;
    }
    __syncthreads();
    const unsigned long long wm = __reduce_or_sync(0xffffffffu, (unsigned)(my_mask & 0xffffffffu)) |
                                  ((unsigned long long)__reduce_or_sync(0xffffffffu, (unsigned)(my_mask >> 32)) << 32);
    const unsigned wd = __reduce_add_sync(0xffffffffu, differs);
    const unsigned wn = __reduce_add_sync(0xffffffffu, no_major);
    if ((threadIdx.x & 31u) == 0) {
        if (wm) atomicOr(&s_mask, wm);
        if (wd) atomicAdd(&s_diff, wd);
        if (wn) atomicAdd(&s_nomaj, wn);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (s_mask) atomicOr((unsigned long long *)&summary->suspect_mask, s_mask);
        if (s_diff) {
            atomicAdd(&summary->n_differing, s_diff);
            atomicOr(&summary->diverged, 1u);
        }
        if (s_nomaj) {
            atomicAdd(&summary->n_no_majority, s_nomaj);
            atomicOr(&summary->no_majority, 1u);
        }
    }
}

__global__ void xor_compare_kernel(const uint64_t *__restrict__ a, const uint64_t *__restrict__ b, uint32_t n,
                                   uint8_t *__restrict__ mismatch, uint64_t *__restrict__ diff) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const uint64_t d = a[i] ^ b[i];
        mismatch[i] = d != 0 ? 1 : 0;
        if (diff) diff[i] = d;
    }
}

}  // namespace

cudaError_t launch_vote(const uint64_t *fp, uint32_t R, uint32_t T, int32_t *suspect, uint64_t *mask,
                        sdc_vote_summary *summary, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(summary, 0, sizeof(sdc_vote_summary), st);
    if (e != cudaSuccess) return e;
    if (T == 0) return cudaSuccess;
    vote_kernel<<<(T + kVoteBlock - 1) / kVoteBlock, kVoteBlock, 0, st>>>(fp, R, T, suspect, mask, summary);
    return cudaGetLastError();
}

cudaError_t launch_xor_compare(const uint64_t *a, const uint64_t *b, uint32_t n, uint8_t *mismatch, uint64_t *diff,
                               cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    xor_compare_kernel<<<(n + 255) / 256, 256, 0, st>>>(a, b, n, mismatch, diff);
    return cudaGetLastError();
}

}  // namespace sdc
