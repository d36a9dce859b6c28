// sdc_fp.cu -- fingerprint and xorsum passes over a plan's chunk table.
//
// Fingerprint ("Detecting and recovering from silent data corruption on
// Amazon SageMaker HyperPod", section "Compare by fingerprint"): per tensor,
// S = sum of the widened raw bits and W = sum of (index + 1) * bits, mod 2^64.
// Xorsum ("Safeguarding LLM Training at Scale ..." review, method section 4):
// XOR of the raw bits, zero-extended to 64 bits.
//
// Layout of the work: one warp task per chunk (<= 32 KiB of one tensor copy).
// A persistent grid of warps walks the chunk table; each warp reads its chunk
// with coalesced 16-byte streaming loads (512 contiguous bytes per warp
// instruction), reduces in registers and with shuffles, and writes one
// partial.  A second kernel, parallel over chunks, combines the partials per
// descriptor in integer arithmetic, so the result is exact and independent of
// the launch shape.
//
// Position weights without a 64-bit multiply per element: for a chunk whose
// first element has tensor index o, W = sum_j (o + j + 1) b_j
// = o * S_chunk + W_chunk, with W_chunk using chunk-local indices j.  Inside a
// chunk, lane l reads vectors v = l + 32 i, whose first element has local
// index h + e v (h = elements before the first aligned vector, e = elements
// per vector), so
//   W_chunk = sum_lanes [ (h + 1 + e l) S_l + 32 e I_l + L_l ]
// with S_l = sum of the lane's vector sums s_v, I_l = sum_i i s_v and
// L_l = sum of in-vector weighted sums sum_k k b_k.  For 1- and 2-byte
// elements s_v, L and I are formed with dp4a/dp2a byte-weighted dot products
// in 32-bit registers, which cannot overflow for <= 64 vectors per lane
// (chunk_bytes <= 32 KiB); they are widened once per chunk.
#include "sdc_internal.cuh"

namespace sdc {

namespace {

// Element i of a run starting at byte address `a`, widened the page's way:
// 1-byte zero-extended, wider sign-extended.
__device__ __forceinline__ uint64_t load_widened(uint64_t a, uint32_t l2) {
    switch (l2) {
        case 0: return (uint64_t)(*(const uint8_t *)a);
        case 1: return (uint64_t)(int64_t)(*(const int16_t *)a);
        case 2: return (uint64_t)(int64_t)(*(const int32_t *)a);
        default: return *(const uint64_t *)a;
    }
}
__device__ __forceinline__ uint64_t load_zext(uint64_t a, uint32_t l2) {
    switch (l2) {
        case 0: return (uint64_t)(*(const uint8_t *)a);
        case 1: return (uint64_t)(*(const uint16_t *)a);
        case 2: return (uint64_t)(*(const uint32_t *)a);
        default: return *(const uint64_t *)a;
    }
}

struct ChunkGeom {
    uint64_t addr;
    uint32_t head;  // bytes before the first 16-byte-aligned vector
    uint32_t nvec;  // aligned 16-byte vectors
    uint32_t tail;  // bytes after the last vector
    uint32_t l2;    // log2(elem size)
};

__device__ __forceinline__ ChunkGeom geom(const Chunk &ch) {
    ChunkGeom g;
    g.addr = ch.addr;
    g.l2 = chunk_log2es(ch.tag);
    uint32_t head = (uint32_t)((16u - (uint32_t)(ch.addr & 15u)) & 15u);
    if (head > ch.nbytes) head = ch.nbytes;
    g.head = head;
    g.nvec = (ch.nbytes - head) >> 4;
    g.tail = ch.nbytes - head - (g.nvec << 4);
    return g;
}

// Head and tail elements (fewer than 16 of each), one per lane: lanes 0..15
// take the head, lanes 16..31 the tail.  Returns the lane's element (widened
// or zero-extended) and its chunk-local index, or false.
template <bool kZext>
__device__ __forceinline__ bool edge_element(const ChunkGeom &g, uint32_t lane, uint64_t &b, uint64_t &j) {
    const uint32_t he = g.head >> g.l2, te = g.tail >> g.l2;
    uint64_t a;
    if (lane < 16) {
        if (lane >= he) return false;
        a = g.addr + ((uint64_t)lane << g.l2);
        j = lane;
    } else {
        const uint32_t t = lane - 16;
        if (t >= te) return false;
        const uint64_t off = (uint64_t)g.head + ((uint64_t)g.nvec << 4) + ((uint64_t)t << g.l2);
        a = g.addr + off;
        j = off >> g.l2;
    }
    b = kZext ? load_zext(a, g.l2) : load_widened(a, g.l2);
    return true;
}

// ---------------------------------------------------------------- fingerprint bodies
// Each returns the lane's (S, W) contribution over the aligned vectors, with
// W in chunk-local 1-based indices.

template <int U>
__device__ __forceinline__ void fp_body_1(const ChunkGeom &g, uint32_t lane, uint64_t &S, uint64_t &W) {
    const uint4 *vb = (const uint4 *)(g.addr + g.head);
    const uint32_t niter = (g.nvec + 31) >> 5;
    uint32_t S32 = 0, L32 = 0, I32 = 0;
    for (uint32_t i0 = 0; i0 < niter; i0 += U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t vi = lane + ((i0 + u) << 5);
            v[u] = vi < g.nvec ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t s = dp4a_u(v[u].x, 0x01010101u, 0u);
            s = dp4a_u(v[u].y, 0x01010101u, s);
            s = dp4a_u(v[u].z, 0x01010101u, s);
            s = dp4a_u(v[u].w, 0x01010101u, s);
            L32 = dp4a_u(v[u].x, 0x03020100u, L32);
            L32 = dp4a_u(v[u].y, 0x07060504u, L32);
            L32 = dp4a_u(v[u].z, 0x0B0A0908u, L32);
            L32 = dp4a_u(v[u].w, 0x0F0E0D0Cu, L32);
            S32 += s;
            I32 += (i0 + u) * s;
        }
    }
    const uint64_t h = g.head;  // 1-byte elements: head bytes == head elements
    S = S32;
    W = (h + 1 + 16ull * lane) * (uint64_t)S32 + 512ull * (uint64_t)I32 + (uint64_t)L32;
}

template <int U>
__device__ __forceinline__ void fp_body_2(const ChunkGeom &g, uint32_t lane, uint64_t &S, uint64_t &W) {
    const uint4 *vb = (const uint4 *)(g.addr + g.head);
    const uint32_t niter = (g.nvec + 31) >> 5;
    int S32 = 0, L32 = 0, I32 = 0;
    for (uint32_t i0 = 0; i0 < niter; i0 += U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t vi = lane + ((i0 + u) << 5);
            v[u] = vi < g.nvec ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            // sum of the 8 signed halves, and sum of k * half_k for k = 0..7
            int s = dp2a_lo_s(v[u].x, 0x0101u, 0);
            s = dp2a_lo_s(v[u].y, 0x0101u, s);
            s = dp2a_lo_s(v[u].z, 0x0101u, s);
            s = dp2a_lo_s(v[u].w, 0x0101u, s);
            L32 = dp2a_lo_s(v[u].x, 0x03020100u, L32);
            L32 = dp2a_hi_s(v[u].y, 0x03020100u, L32);
            L32 = dp2a_lo_s(v[u].z, 0x07060504u, L32);
            L32 = dp2a_hi_s(v[u].w, 0x07060504u, L32);
            S32 += s;
            I32 += (int)(i0 + u) * s;
        }
    }
    const uint64_t h = g.head >> 1;
    const uint64_t S64 = (uint64_t)(int64_t)S32;
    S = S64;
    W = (h + 1 + 8ull * lane) * S64 + 256ull * (uint64_t)(int64_t)I32 + (uint64_t)(int64_t)L32;
}

template <int U>
__device__ __forceinline__ void fp_body_4(const ChunkGeom &g, uint32_t lane, uint64_t &S, uint64_t &W) {
    const uint4 *vb = (const uint4 *)(g.addr + g.head);
    const uint32_t niter = (g.nvec + 31) >> 5;
    uint64_t S64 = 0, L64 = 0, I64 = 0;
    for (uint32_t i0 = 0; i0 < niter; i0 += U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t vi = lane + ((i0 + u) << 5);
            v[u] = vi < g.nvec ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t a = (int32_t)v[u].x, b = (int32_t)v[u].y, c = (int32_t)v[u].z, d = (int32_t)v[u].w;
            const int64_t s = a + b + c + d;           // |s| < 2^33: exact
            const int64_t l = b + 2 * c + 3 * d;       // |l| < 2^34: exact
            S64 += (uint64_t)s;
            L64 += (uint64_t)l;
            I64 += (uint64_t)((int64_t)(i0 + u) * s);  // |i s| < 2^39: exact
        }
    }
    const uint64_t h = g.head >> 2;
    S = S64;
    W = (h + 1 + 4ull * lane) * S64 + 128ull * I64 + L64;
}

template <int U>
__device__ __forceinline__ void fp_body_8(const ChunkGeom &g, uint32_t lane, uint64_t &S, uint64_t &W) {
    const uint4 *vb = (const uint4 *)(g.addr + g.head);
    const uint32_t niter = (g.nvec + 31) >> 5;
    uint64_t S64 = 0, L64 = 0, I64 = 0;
    for (uint32_t i0 = 0; i0 < niter; i0 += U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t vi = lane + ((i0 + u) << 5);
            v[u] = vi < g.nvec ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t b0 = ((uint64_t)v[u].y << 32) | v[u].x;
            const uint64_t b1 = ((uint64_t)v[u].w << 32) | v[u].z;
            const uint64_t s = b0 + b1;
            S64 += s;
            L64 += b1;
            I64 += (uint64_t)(i0 + u) * s;
        }
    }
    const uint64_t h = g.head >> 3;
    S = S64;
    W = (h + 1 + 2ull * lane) * S64 + 64ull * I64 + L64;
}

template <int U>
__global__ void __launch_bounds__(kScanBlock) fp_scan_kernel(const Chunk *__restrict__ chunks, uint64_t n_chunks,
                                                             FpPartial *__restrict__ partials) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    if (warp >= n_chunks) return;
    Chunk next = chunks[warp];
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const Chunk ch = next;
        if (c + nwarps < n_chunks) next = chunks[c + nwarps];  // prefetch the next task
        const ChunkGeom g = geom(ch);
        uint64_t S, W;
        switch (g.l2) {
            case 0: fp_body_1<U>(g, lane, S, W); break;
            case 1: fp_body_2<U>(g, lane, S, W); break;
            case 2: fp_body_4<U>(g, lane, S, W); break;
            default: fp_body_8<U>(g, lane, S, W); break;
        }
        uint64_t b, j;
        if (edge_element<false>(g, lane, b, j)) {
            S += b;
            W += (j + 1) * b;
        }
        S = warp_sum_u64(S);
        W = warp_sum_u64(W);
        if (lane == 0) partials[c] = FpPartial{S, W};
    }
}

// Second pass, parallel over chunks: thread i turns chunk i's partial into
// its tensor-level contribution (S_c, W_c + o_c S_c), o_c = the chunk's first
// tensor index; a segmented warp scan sums the contributions of each run of
// chunks that belong to one descriptor (the chunk table is in descriptor
// order), and the last lane of each run adds the run's sums to the output
// with one 64-bit atomic per sum.  Integer addition mod 2^64 is associative
// and commutative, so the result is exact and the same on every run.
// `out` must be zeroed first (descriptors without chunks stay (0, 0)).
__global__ void fp_combine_kernel(const Chunk *__restrict__ chunks, uint64_t n_chunks,
                                  const DescDev *__restrict__ descs, const FpPartial *__restrict__ partials,
                                  unsigned long long *__restrict__ out) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t d = 0xFFFFFFFFu;
    uint64_t S = 0, W = 0;
    if (i < n_chunks) {
        const Chunk ch = chunks[i];
        const FpPartial p = partials[i];
        d = chunk_desc(ch.tag);
        const uint64_t o = (ch.addr - descs[d].ptr) >> chunk_log2es(ch.tag);
        S = p.s;
        W = p.w + o * p.s;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t s_up = __shfl_up_sync(0xffffffffu, S, off);
        const uint64_t w_up = __shfl_up_sync(0xffffffffu, W, off);
        const uint32_t d_up = __shfl_up_sync(0xffffffffu, d, off);
        if (lane >= (uint32_t)off && d_up == d) {
            S += s_up;
            W += w_up;
        }
    }
    const uint32_t d_next = __shfl_down_sync(0xffffffffu, d, 1);
    if (d != 0xFFFFFFFFu && (lane == 31u || d_next != d)) {
        atomicAdd(out + 2ull * d, (unsigned long long)S);
        atomicAdd(out + 2ull * d + 1, (unsigned long long)W);
    }
}

// ---------------------------------------------------------------- xorsum
template <int U>
__global__ void __launch_bounds__(kScanBlock) xor_scan_kernel(const Chunk *__restrict__ chunks, uint64_t n_chunks,
                                                              uint64_t *__restrict__ partials) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const ChunkGeom g = geom(chunks[c]);
        const uint4 *vb = (const uint4 *)(g.addr + g.head);
        const uint32_t niter = (g.nvec + 31) >> 5;
        uint32_t xa = 0, xb = 0;  // XOR of words 0/2 and of words 1/3
        for (uint32_t i0 = 0; i0 < niter; i0 += U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t vi = lane + ((i0 + u) << 5);
                v[u] = vi < g.nvec ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                xa ^= v[u].x ^ v[u].z;
                xb ^= v[u].y ^ v[u].w;
            }
        }
        // fold the aligned words into one element-width value
        uint64_t X;
        if (g.l2 == 3) {
            X = ((uint64_t)xb << 32) | xa;
        } else {
            uint32_t x = xa ^ xb;
            if (g.l2 <= 1) x = (x ^ (x >> 16)) & 0xFFFFu;
            if (g.l2 == 0) x = (x ^ (x >> 8)) & 0xFFu;
            X = x;
        }
        uint64_t b, j;
        if (edge_element<true>(g, lane, b, j)) X ^= b;
        X = warp_xor_u64(X);
        if (lane == 0) partials[c] = X;
    }
}

// Same second pass for the xorsum: XOR is associative and commutative.
__global__ void xor_combine_kernel(const Chunk *__restrict__ chunks, uint64_t n_chunks,
                                   const uint64_t *__restrict__ partials, unsigned long long *__restrict__ out) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t d = 0xFFFFFFFFu;
    uint64_t X = 0;
    if (i < n_chunks) {
        d = chunk_desc(chunks[i].tag);
        X = partials[i];
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t x_up = __shfl_up_sync(0xffffffffu, X, off);
        const uint32_t d_up = __shfl_up_sync(0xffffffffu, d, off);
        if (lane >= (uint32_t)off && d_up == d) X ^= x_up;
    }
    const uint32_t d_next = __shfl_down_sync(0xffffffffu, d, 1);
    if (d != 0xFFFFFFFFu && (lane == 31u || d_next != d)) atomicXor(out + d, (unsigned long long)X);
}

constexpr int kFpUnroll = 4;

}  // namespace

int fp_scan_blocks_per_sm() {
    int n = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fp_scan_kernel<kFpUnroll>, kScanBlock, 0);
    return n > 0 ? n : 1;
}

cudaError_t launch_fp_scan(const sdc_plan *plan, FpPartial *partials, cudaStream_t st) {
    if (plan->n_chunks == 0) return cudaSuccess;
    fp_scan_kernel<kFpUnroll><<<plan->grid, plan->block, 0, st>>>(plan->d_chunks, plan->n_chunks, partials);
    return cudaGetLastError();
}

cudaError_t launch_fp_combine(const sdc_plan *plan, const FpPartial *partials, uint64_t *out, cudaStream_t st) {
    if (plan->n_desc == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(out, 0, plan->n_desc * 2 * sizeof(uint64_t), st);
    if (e != cudaSuccess || plan->n_chunks == 0) return e;
    const unsigned blocks = (unsigned)((plan->n_chunks + 255) / 256);
    fp_combine_kernel<<<blocks, 256, 0, st>>>(plan->d_chunks, plan->n_chunks, plan->d_descs, partials,
                                              (unsigned long long *)out);
    return cudaGetLastError();
}

cudaError_t launch_xor_scan(const sdc_plan *plan, uint64_t *partials, cudaStream_t st) {
    if (plan->n_chunks == 0) return cudaSuccess;
    xor_scan_kernel<kFpUnroll><<<plan->grid, plan->block, 0, st>>>(plan->d_chunks, plan->n_chunks, partials);
    return cudaGetLastError();
}

cudaError_t launch_xor_combine(const sdc_plan *plan, const uint64_t *partials, uint64_t *out, cudaStream_t st) {
    if (plan->n_desc == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(out, 0, plan->n_desc * sizeof(uint64_t), st);
    if (e != cudaSuccess || plan->n_chunks == 0) return e;
    const unsigned blocks = (unsigned)((plan->n_chunks + 255) / 256);
    xor_combine_kernel<<<blocks, 256, 0, st>>>(plan->d_chunks, plan->n_chunks, partials,
                                               (unsigned long long *)out);
    return cudaGetLastError();
}

}  // namespace sdc
