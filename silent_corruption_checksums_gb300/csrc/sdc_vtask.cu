// sdc_vtask.cu -- the replay context of the GEMM checksum and its replay.
//
// "Safeguarding LLM Training at Scale: Online SDC Detection and Insights from
// 35 Million GPU Hours" (review page), method sections 1 and 2: when a check
// fires, the sensor packs its evidence and the least context a replay needs
// into a vTask; a verifier replays it off the critical path and confirms.  For
// the forward (and dgrad) product the context is the flagged row of A and its
// output row; for the weight gradient, A's rows, B's columns and the matching
// results.
//
// Capture: the flagged indices in increasing order (one block scans the
// flags), then one block per captured row copies it (16-byte vectors), or per
// captured column gathers it (a strided column of a row-major matrix).
//
// Replay: the captured operands are recomputed by the same tensor-core GEMM
// kernel at the same position inside a tile (row i at lane i mod 128 of its
// own 128-row tile, column j at j mod 256 of its own 256-column tile, the
// other rows and columns zero), so a healthy GPU reproduces every accumulator
// bit and every rounding of the original output: a row of the product depends
// on its own row of A alone, and each output's accumulation order on its
// position in the tile and the contraction's blocks, not on the values beside
// it.  An output that is not reproduced bit for bit confirms a fault in the
// original computation (or in the replay: a confirming replay belongs on a
// second GPU).
#include <cuda_bf16.h>

#include "sdc_internal.cuh"

namespace sdc {

namespace {

constexpr uint32_t kRowTile = 128, kColTile = 256;  // the GEMM kernel's output tile
constexpr uint32_t kMaxCapture = 1024;              // captured rows (forward replay)
constexpr uint32_t kMaxPairs = 64;                  // captured rows and columns (the pairs replays)

// idx[0 .. min(total, cap)) = the positions of the non-zero flags in increasing order; *count = total.
// One block of 1024 threads, each over a contiguous run of the flags, an exclusive scan of the runs'
// counts between them.
__global__ void __launch_bounds__(1024) capture_scan_kernel(const uint8_t *__restrict__ flag, uint32_t n, uint32_t cap,
                                                            uint32_t *__restrict__ idx, uint32_t *__restrict__ count) {
    __shared__ uint32_t warp_tot[32];
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t per = (n + 1023) / 1024, b0 = tid * per < n ? tid * per : n, b1 = b0 + per < n ? b0 + per : n;
    uint32_t mine = 0;
    for (uint32_t i = b0; i < b1; ++i) mine += flag[i] != 0;
    uint32_t incl = mine;  // inclusive scan in the warp, then over the warps
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= (uint32_t)off) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_tot[lane], wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= (uint32_t)off) wi += v;
        }
        warp_tot[lane] = wi - w;  // exclusive: the warps before this one
    }
    __syncthreads();
    uint32_t pos = warp_tot[warp] + incl - mine;
    for (uint32_t i = b0; i < b1 && pos < cap; ++i)
        if (flag[i] != 0) idx[pos++] = i;
    if (tid == 1023) *count = warp_tot[31] + incl;
}

// dst[r][0 .. n) = src[idx[r]][0 .. n) for r < min(count, cap); one block per row, 16-byte vectors
// (n a multiple of 8 bf16).
__global__ void __launch_bounds__(256) capture_rows_kernel(const __nv_bfloat16 *__restrict__ src, uint32_t n,
                                                           const uint32_t *__restrict__ idx,
                                                           const uint32_t *__restrict__ count, uint32_t cap,
                                                           __nv_bfloat16 *__restrict__ dst) {
    const uint32_t r = blockIdx.x;
    if (r >= min(*count, cap)) return;
    const uint4 *s = (const uint4 *)(src + (uint64_t)idx[r] * n);
    uint4 *d = (uint4 *)(dst + (uint64_t)r * n);
    for (uint32_t v = threadIdx.x; v < n / 8; v += blockDim.x) d[v] = s[v];
}

// dst[c][0 .. rows) = src[0 .. rows)[idx[c]] for c < min(count, cap): column idx[c] of the row-major
// src [rows][ld]; block (x, c) gathers rows 256 x .. 256 x + 255.
__global__ void __launch_bounds__(256) capture_cols_kernel(const uint16_t *__restrict__ src, uint32_t rows,
                                                           uint32_t ld, const uint32_t *__restrict__ idx,
                                                           const uint32_t *__restrict__ count, uint32_t cap,
                                                           uint16_t *__restrict__ dst) {
    const uint32_t c = blockIdx.y, i = blockIdx.x * 256 + threadIdx.x;
    if (c >= min(*count, cap) || i >= rows) return;
    dst[(uint64_t)c * rows + i] = src[(uint64_t)i * ld + idx[c]];
}

// staged[r * tile + idx[r] % tile][0 .. K) = rows[r][0 .. K) for r < min(count, cap) (the rest of
// staged is zero): each captured row of A at its own lane of its own 128-row tile (tile = 128), or
// each captured row of W at its own column of its own 256-column tile of the product (tile = 256).
__global__ void __launch_bounds__(256) stage_rows_kernel(const __nv_bfloat16 *__restrict__ rows, uint32_t K,
                                                         const uint32_t *__restrict__ idx,
                                                         const uint32_t *__restrict__ count, uint32_t cap,
                                                         uint32_t tile, __nv_bfloat16 *__restrict__ staged) {
    const uint32_t r = blockIdx.x;
    if (r >= min(*count, cap)) return;
    const uint4 *s = (const uint4 *)(rows + (uint64_t)r * K);
    uint4 *d = (uint4 *)(staged + ((uint64_t)r * tile + idx[r] % tile) * K);
    for (uint32_t v = threadIdx.x; v < K / 8; v += blockDim.x) d[v] = s[v];
}

// ndiff[r] = how many of the n outputs of captured row r the replay does not reproduce bit for bit
// (0 for r past the captured rows); n_differ counts the rows with any.  One block per row.
__global__ void __launch_bounds__(256) compare_rows_kernel(const uint16_t *__restrict__ replay,
                                                           const uint16_t *__restrict__ saved, uint32_t n,
                                                           const uint32_t *__restrict__ idx,
                                                           const uint32_t *__restrict__ count, uint32_t cap,
                                                           uint32_t *__restrict__ ndiff,
                                                           uint32_t *__restrict__ n_differ) {
    __shared__ uint32_t part[8];
    const uint32_t r = blockIdx.x;
    uint32_t d = 0;
    if (r < min(*count, cap)) {
        const uint16_t *a = replay + ((uint64_t)r * kRowTile + idx[r] % kRowTile) * n;
        const uint16_t *b = saved + (uint64_t)r * n;
        for (uint32_t j = threadIdx.x; j < n; j += blockDim.x) d += a[j] != b[j];
    }
    d = warp_sum_u32(d);
    if ((threadIdx.x & 31u) == 0) part[threadIdx.x >> 5] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < 8; ++w) t += part[w];
        ndiff[r] = t;
        if (t) atomicAdd(n_differ, 1u);
    }
}

// Weight-gradient replay operands: column (r * tile + idx[r] % tile) of the token-major staged
// [T][cap * tile] holds captured column r (cols[r][0 .. T)), for r < min(count, cap); the rest is
// zero.  Block (x, r) covers tokens 256 x .. 256 x + 255.
__global__ void __launch_bounds__(256) stage_cols_kernel(const uint16_t *__restrict__ cols, uint32_t T,
                                                         const uint32_t *__restrict__ idx,
                                                         const uint32_t *__restrict__ count, uint32_t cap,
                                                         uint32_t tile, uint16_t *__restrict__ staged) {
    const uint32_t r = blockIdx.y, t = blockIdx.x * 256 + threadIdx.x;
    if (r >= min(*count, cap) || t >= T) return;
    staged[(uint64_t)t * cap * tile + (uint64_t)r * tile + idx[r] % tile] = cols[(uint64_t)r * T + t];
}

// differs[r][c] = 1 unless the replayed dW[n_r][k_c] equals, bit for bit, both saved copies of it
// (row r's element k_c and column c's element n_r); pairs past the captured rows or columns are 0.
// n_differ counts the pairs that differ.
__global__ void __launch_bounds__(256) compare_pairs_kernel(const uint16_t *__restrict__ replay, uint32_t cap_r,
                                                            uint32_t cap_c, uint32_t N, uint32_t K,
                                                            const uint32_t *__restrict__ row_idx,
                                                            const uint16_t *__restrict__ row_dW,
                                                            const uint32_t *__restrict__ col_idx,
                                                            const uint16_t *__restrict__ col_dW,
                                                            const uint32_t *__restrict__ counts,
                                                            uint8_t *__restrict__ differs,
                                                            uint32_t *__restrict__ n_differ) {
    const uint32_t p = blockIdx.x * 256 + threadIdx.x;
    if (p >= cap_r * cap_c) return;
    const uint32_t r = p / cap_c, c = p % cap_c;
    uint8_t f = 0;
    if (r < min(counts[0], cap_r) && c < min(counts[1], cap_c)) {
        const uint32_t n = row_idx[r], k = col_idx[c];
        const uint16_t v = replay[((uint64_t)r * kRowTile + n % kRowTile) * ((uint64_t)cap_c * kColTile) +
                                  (uint64_t)c * kColTile + k % kColTile];
        f = (v != row_dW[(uint64_t)r * K + k] || v != col_dW[(uint64_t)c * N + n]) ? 1 : 0;
        if (f) atomicAdd(n_differ, 1u);
    }
    differs[p] = f;
}

// Aborted flag of the replay's GEMM into summary[1].
__global__ void copy_word_kernel(const uint32_t *__restrict__ src, uint32_t *__restrict__ dst) { *dst = *src; }

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Forward replay workspace: staged rows [cap * 128][K] | replayed C [cap * 128][N] | row checksums
// [cap * 128] double | aborted word | the GEMM's workspace.
struct ReplayWs {
    size_t staged, out, rowsum, aborted, gemm, gemm_bytes, total;
};
ReplayWs replay_ws(uint32_t cap, uint32_t N, uint32_t K) {
    ReplayWs w;
    const size_t M = (size_t)cap * kRowTile;
    w.staged = 0;
    w.out = round_up256(M * K * 2);
    w.rowsum = w.out + round_up256(M * N * 2);
    w.aborted = w.rowsum + round_up256(M * 8);
    w.gemm = w.aborted + 256;
    w.gemm_bytes = sdc_abft_workspace_size((uint32_t)M, N, K);
    w.total = w.gemm + round_up256(w.gemm_bytes);
    return w;
}

// Forward pairs replay workspace: staged A rows [cap_r * 128][K] | staged W rows [cap_c * 256][K] |
// replayed C [cap_r * 128][cap_c * 256] | row checksums [cap_r * 128] double | aborted word | the GEMM's
// workspace.
struct ReplayPairsWs {
    size_t sa, sw, out, rowsum, aborted, gemm, gemm_bytes, total;
};
ReplayPairsWs replay_pairs_ws(uint32_t K, uint32_t cap_r, uint32_t cap_c) {
    ReplayPairsWs w;
    const size_t m = (size_t)cap_r * kRowTile, n = (size_t)cap_c * kColTile;
    w.sa = 0;
    w.sw = round_up256(m * K * 2);
    w.out = w.sw + round_up256(n * K * 2);
    w.rowsum = w.out + round_up256(m * n * 2);
    w.aborted = w.rowsum + round_up256(m * 8);
    w.gemm = w.aborted + 256;
    w.gemm_bytes = sdc_abft_workspace_size((uint32_t)m, (uint32_t)n, K);
    w.total = w.gemm + round_up256(w.gemm_bytes);
    return w;
}

// Weight-gradient replay workspace: staged dY [T][cap_r * 128] | staged X [T][cap_c * 256] |
// replayed dW [cap_r * 128][cap_c * 256] | row checksums [cap_r * 128] double | aborted word | the
// GEMM's workspace.
struct ReplayWgWs {
    size_t sdy, sx, out, rowsum, aborted, gemm, gemm_bytes, total;
};
ReplayWgWs replay_wg_ws(uint32_t T, uint32_t cap_r, uint32_t cap_c) {
    ReplayWgWs w;
    const size_t n = (size_t)cap_r * kRowTile, k = (size_t)cap_c * kColTile;
    w.sdy = 0;
    w.sx = round_up256((size_t)T * n * 2);
    w.out = w.sx + round_up256((size_t)T * k * 2);
    w.rowsum = w.out + round_up256(n * k * 2);
    w.aborted = w.rowsum + round_up256(n * 8);
    w.gemm = w.aborted + 256;
    w.gemm_bytes = sdc_abft_wgrad_workspace_size(T, (uint32_t)n, (uint32_t)k);
    w.total = w.gemm + round_up256(w.gemm_bytes);
    return w;
}

}  // namespace

}  // namespace sdc

using namespace sdc;

extern "C" {

// One capture: the flagged indices of `flag` [n] (at most cap), then the rows of `rows_src`
// [n][row_len] and the columns of `cols_src` [col_rows][n] they name.
static cudaError_t capture_side(const uint8_t *flag, uint32_t n, uint32_t cap, uint32_t *idx, uint32_t *count,
                                const void *rows_src, uint32_t row_len, void *rows_dst, const void *cols_src,
                                uint32_t col_rows, void *cols_dst, cudaStream_t s) {
    capture_scan_kernel<<<1, 1024, 0, s>>>(flag, n, cap, idx, count);
    if (cap && rows_src)
        capture_rows_kernel<<<cap, 256, 0, s>>>((const __nv_bfloat16 *)rows_src, row_len, idx, count, cap,
                                                (__nv_bfloat16 *)rows_dst);
    if (cap && cols_src)
        capture_cols_kernel<<<dim3((col_rows + 255) / 256, cap), 256, 0, s>>>(
            (const uint16_t *)cols_src, col_rows, n, idx, count, cap, (uint16_t *)cols_dst);
    return cudaGetLastError();
}

sdc_status sdc_abft_capture(const void *d_A, const void *d_W, const void *d_C, uint32_t M, uint32_t N, uint32_t K,
                            const uint8_t *d_flag, const uint8_t *d_flag_col, uint32_t cap_rows, uint32_t *d_row_idx,
                            void *d_row_A, void *d_row_C, uint32_t cap_cols, uint32_t *d_col_idx, void *d_col_W,
                            void *d_col_C, uint32_t *d_counts, sdc_stream_t stream) {
    if (!d_A || !d_W || !d_C || !d_flag || !d_counts) return fail(SDC_ERR_NULL, "NULL argument");
    if (M == 0 || N == 0 || K == 0 || N % 8 || K % 8) return fail(SDC_ERR_BAD_ARG, "M positive, N and K multiples of 8");
    const bool cols = d_flag_col != nullptr;
    if ((cap_rows && (!d_row_idx || !d_row_A || !d_row_C)) ||
        (cols && cap_cols && (!d_col_idx || !d_col_W || !d_col_C)))
        return fail(SDC_ERR_NULL, "NULL capture buffer");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const uint64_t cc = cols ? cap_cols : 0;
    sdc_status st = check_spans({{d_A, (uint64_t)M * K * 2, "d_A"},
                                 {d_W, (uint64_t)N * K * 2, "d_W"},
                                 {d_C, (uint64_t)M * N * 2, "d_C"},
                                 {d_flag, M, "d_flag"},
                                 {d_flag_col, cols ? N : 0, "d_flag_col"},
                                 {d_row_idx, (uint64_t)cap_rows * 4, "d_row_idx"},
                                 {d_row_A, (uint64_t)cap_rows * K * 2, "d_row_A"},
                                 {d_row_C, (uint64_t)cap_rows * N * 2, "d_row_C"},
                                 {d_col_idx, cc * 4, "d_col_idx"},
                                 {d_col_W, cc * K * 2, "d_col_W"},
                                 {d_col_C, cc * M * 2, "d_col_C"},
                                 {d_counts, 8, "d_counts"}},
                                dev);
    if (st != SDC_OK) return st;
    if (((uint64_t)d_A | (uint64_t)d_W | (uint64_t)d_C | (uint64_t)d_row_A | (uint64_t)d_row_C |
         (uint64_t)(cols ? d_col_W : nullptr)) & 15u)
        return fail(SDC_ERR_BAD_POINTER, "matrices and row buffers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    // rows: A's row and C's row; columns: W's row j (B's column j) and C's column j
    e = capture_side(d_flag, M, cap_rows, d_row_idx, d_counts, d_A, K, d_row_A, nullptr, 0, nullptr, s);
    if (e == cudaSuccess && cap_rows)
        capture_rows_kernel<<<cap_rows, 256, 0, s>>>((const __nv_bfloat16 *)d_C, N, d_row_idx, d_counts, cap_rows,
                                                     (__nv_bfloat16 *)d_row_C);
    if (e == cudaSuccess && cols)
        e = capture_side(d_flag_col, N, cap_cols, d_col_idx, d_counts + 1, d_W, K, d_col_W, d_C, M, d_col_C, s);
    if (e == cudaSuccess && !cols) e = cudaMemsetAsync(d_counts + 1, 0, 4, s);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_capture launch");
}

sdc_status sdc_abft_capture_wgrad(const void *d_dY, const void *d_X, const void *d_dW, uint32_t T, uint32_t N,
                                  uint32_t K, const uint8_t *d_flag, const uint8_t *d_flag_col, uint32_t cap_rows,
                                  uint32_t *d_row_idx, void *d_row_dY, void *d_row_dW, uint32_t cap_cols,
                                  uint32_t *d_col_idx, void *d_col_X, void *d_col_dW, uint32_t *d_counts,
                                  sdc_stream_t stream) {
    if (!d_dY || !d_X || !d_dW || !d_flag || !d_counts) return fail(SDC_ERR_NULL, "NULL argument");
    if (T == 0 || N == 0 || K == 0 || N % 8 || K % 8) return fail(SDC_ERR_BAD_ARG, "T positive, N and K multiples of 8");
    const bool cols = d_flag_col != nullptr;
    if ((cap_rows && (!d_row_idx || !d_row_dY || !d_row_dW)) ||
        (cols && cap_cols && (!d_col_idx || !d_col_X || !d_col_dW)))
        return fail(SDC_ERR_NULL, "NULL capture buffer");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const uint64_t cc = cols ? cap_cols : 0;
    sdc_status st = check_spans({{d_dY, (uint64_t)T * N * 2, "d_dY"},
                                 {d_X, (uint64_t)T * K * 2, "d_X"},
                                 {d_dW, (uint64_t)N * K * 2, "d_dW"},
                                 {d_flag, N, "d_flag"},
                                 {d_flag_col, cols ? K : 0, "d_flag_col"},
                                 {d_row_idx, (uint64_t)cap_rows * 4, "d_row_idx"},
                                 {d_row_dY, (uint64_t)cap_rows * T * 2, "d_row_dY"},
                                 {d_row_dW, (uint64_t)cap_rows * K * 2, "d_row_dW"},
                                 {d_col_idx, cc * 4, "d_col_idx"},
                                 {d_col_X, cc * T * 2, "d_col_X"},
                                 {d_col_dW, cc * N * 2, "d_col_dW"},
                                 {d_counts, 8, "d_counts"}},
                                dev);
    if (st != SDC_OK) return st;
    if (((uint64_t)d_dW | (uint64_t)d_row_dW) & 15u) return fail(SDC_ERR_BAD_POINTER, "dW and d_row_dW must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    // rows of dW: dY's column n (A's row) and dW's row n; columns: X's column k (B's column) and dW's column k
    e = capture_side(d_flag, N, cap_rows, d_row_idx, d_counts, d_dW, K, d_row_dW, nullptr, 0, nullptr, s);
    if (e == cudaSuccess && cap_rows)
        capture_cols_kernel<<<dim3((T + 255) / 256, cap_rows), 256, 0, s>>>((const uint16_t *)d_dY, T, N, d_row_idx,
                                                                            d_counts, cap_rows, (uint16_t *)d_row_dY);
    if (e == cudaSuccess && cols) {
        e = capture_side(d_flag_col, K, cap_cols, d_col_idx, d_counts + 1, nullptr, 0, nullptr, d_dW, N, d_col_dW, s);
        if (e == cudaSuccess && cap_cols)
            capture_cols_kernel<<<dim3((T + 255) / 256, cap_cols), 256, 0, s>>>(
                (const uint16_t *)d_X, T, K, d_col_idx, d_counts + 1, cap_cols, (uint16_t *)d_col_X);
    }
    if (e == cudaSuccess && !cols) e = cudaMemsetAsync(d_counts + 1, 0, 4, s);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_capture_wgrad launch");
}

size_t sdc_abft_replay_workspace_size(uint32_t cap_rows, uint32_t N, uint32_t K) {
    if (cap_rows == 0 || cap_rows > kMaxCapture || N == 0 || K == 0 || N % 8 || K % 8) return 0;
    return replay_ws(cap_rows, N, K).total;
}

sdc_status sdc_abft_replay(const void *d_W, uint32_t N, uint32_t K, uint32_t cap_rows, const uint32_t *d_row_idx,
                           const void *d_row_A, const void *d_row_C, const uint32_t *d_counts, uint32_t *d_ndiff,
                           uint32_t *d_summary, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    if (!d_W || !d_row_idx || !d_row_A || !d_row_C || !d_counts || !d_ndiff || !d_summary || !d_ws)
        return fail(SDC_ERR_NULL, "NULL argument");
    if (cap_rows == 0 || cap_rows > kMaxCapture || N == 0 || K == 0 || N % 8 || K % 8)
        return fail(SDC_ERR_BAD_ARG, "cap_rows in 1..1024, N and K positive multiples of 8");
    const ReplayWs w = replay_ws(cap_rows, N, K);
    if (ws_bytes < w.total) return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_replay_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    if (((uint64_t)d_row_A | (uint64_t)d_row_C) & 15u) return fail(SDC_ERR_BAD_POINTER, "row buffers must be 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_spans({{d_W, (uint64_t)N * K * 2, "d_W"},
                                 {d_row_idx, (uint64_t)cap_rows * 4, "d_row_idx"},
                                 {d_row_A, (uint64_t)cap_rows * K * 2, "d_row_A"},
                                 {d_row_C, (uint64_t)cap_rows * N * 2, "d_row_C"},
                                 {d_counts, 4, "d_counts"},
                                 {d_ndiff, (uint64_t)cap_rows * 4, "d_ndiff"},
                                 {d_summary, 8, "d_summary"},
                                 {d_ws, w.total, "d_ws"}},
                                dev);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)d_ws;
    const uint32_t M = cap_rows * kRowTile;
    e = cudaMemsetAsync(ws + w.staged, 0, (size_t)M * K * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_summary, 0, 8, s);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_replay setup");
    stage_rows_kernel<<<cap_rows, 256, 0, s>>>((const __nv_bfloat16 *)d_row_A, K, d_row_idx, d_counts, cap_rows,
                                               kRowTile, (__nv_bfloat16 *)(ws + w.staged));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_replay launch");
    st = sdc_abft_gemm(ws + w.staged, d_W, ws + w.out, M, N, K, (double *)(ws + w.rowsum), nullptr,
                       (uint32_t *)(ws + w.aborted), ws + w.gemm, w.gemm_bytes, stream);
    if (st != SDC_OK) return st;
    compare_rows_kernel<<<cap_rows, 256, 0, s>>>((const uint16_t *)(ws + w.out), (const uint16_t *)d_row_C, N,
                                                 d_row_idx, d_counts, cap_rows, d_ndiff, d_summary);
    copy_word_kernel<<<1, 1, 0, s>>>((const uint32_t *)(ws + w.aborted), d_summary + 1);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_replay launch");
}

size_t sdc_abft_replay_wgrad_workspace_size(uint32_t T, uint32_t cap_rows, uint32_t cap_cols) {
    if (T == 0 || cap_rows == 0 || cap_cols == 0 || cap_rows > kMaxPairs || cap_cols > kMaxPairs) return 0;
    return replay_wg_ws(T, cap_rows, cap_cols).total;
}

sdc_status sdc_abft_replay_wgrad(uint32_t T, uint32_t N, uint32_t K, uint32_t cap_rows, uint32_t cap_cols,
                                 const uint32_t *d_row_idx, const void *d_row_dY, const void *d_row_dW,
                                 const uint32_t *d_col_idx, const void *d_col_X, const void *d_col_dW,
                                 const uint32_t *d_counts, uint8_t *d_differs, uint32_t *d_summary, void *d_ws,
                                 size_t ws_bytes, sdc_stream_t stream) {
    if (!d_row_idx || !d_row_dY || !d_row_dW || !d_col_idx || !d_col_X || !d_col_dW || !d_counts || !d_differs ||
        !d_summary || !d_ws)
        return fail(SDC_ERR_NULL, "NULL argument");
    if (T == 0 || T > (1u << 20) || N == 0 || K == 0 || N % 8 || K % 8 || cap_rows == 0 || cap_cols == 0 ||
        cap_rows > kMaxPairs || cap_cols > kMaxPairs)
        return fail(SDC_ERR_BAD_ARG, "T in 1..2^20, N and K multiples of 8, cap_rows and cap_cols in 1..64");
    const ReplayWgWs w = replay_wg_ws(T, cap_rows, cap_cols);
    if (ws_bytes < w.total) return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_replay_wgrad_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_spans({{d_row_idx, (uint64_t)cap_rows * 4, "d_row_idx"},
                                 {d_row_dY, (uint64_t)cap_rows * T * 2, "d_row_dY"},
                                 {d_row_dW, (uint64_t)cap_rows * K * 2, "d_row_dW"},
                                 {d_col_idx, (uint64_t)cap_cols * 4, "d_col_idx"},
                                 {d_col_X, (uint64_t)cap_cols * T * 2, "d_col_X"},
                                 {d_col_dW, (uint64_t)cap_cols * N * 2, "d_col_dW"},
                                 {d_counts, 8, "d_counts"},
                                 {d_differs, (uint64_t)cap_rows * cap_cols, "d_differs"},
                                 {d_summary, 8, "d_summary"},
                                 {d_ws, w.total, "d_ws"}},
                                dev);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)d_ws;
    const uint32_t n = cap_rows * kRowTile, k = cap_cols * kColTile;
    e = cudaMemsetAsync(ws + w.sdy, 0, w.out - w.sdy, s);  // both staged operands
    if (e == cudaSuccess) e = cudaMemsetAsync(d_summary, 0, 8, s);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_replay_wgrad setup");
    stage_cols_kernel<<<dim3((T + 255) / 256, cap_rows), 256, 0, s>>>((const uint16_t *)d_row_dY, T, d_row_idx,
                                                                      d_counts, cap_rows, kRowTile,
                                                                      (uint16_t *)(ws + w.sdy));
    stage_cols_kernel<<<dim3((T + 255) / 256, cap_cols), 256, 0, s>>>((const uint16_t *)d_col_X, T, d_col_idx,
                                                                      d_counts + 1, cap_cols, kColTile,
                                                                      (uint16_t *)(ws + w.sx));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_replay_wgrad launch");
    st = sdc_abft_gemm_wgrad(ws + w.sdy, ws + w.sx, ws + w.out, T, n, k, (double *)(ws + w.rowsum), nullptr,
                             (uint32_t *)(ws + w.aborted), ws + w.gemm, w.gemm_bytes, stream);
    if (st != SDC_OK) return st;
    compare_pairs_kernel<<<(cap_rows * cap_cols + 255) / 256, 256, 0, s>>>(
        (const uint16_t *)(ws + w.out), cap_rows, cap_cols, N, K, d_row_idx, (const uint16_t *)d_row_dW, d_col_idx,
        (const uint16_t *)d_col_dW, d_counts, d_differs, d_summary);
    copy_word_kernel<<<1, 1, 0, s>>>((const uint32_t *)(ws + w.aborted), d_summary + 1);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_replay_wgrad launch");
}

size_t sdc_abft_replay_pairs_workspace_size(uint32_t K, uint32_t cap_rows, uint32_t cap_cols) {
    if (K == 0 || K % 8 || K > (1u << 20) || cap_rows == 0 || cap_cols == 0 || cap_rows > kMaxPairs ||
        cap_cols > kMaxPairs)
        return 0;
    return replay_pairs_ws(K, cap_rows, cap_cols).total;
}

sdc_status sdc_abft_replay_pairs(uint32_t M, uint32_t N, uint32_t K, uint32_t cap_rows, uint32_t cap_cols,
                                 const uint32_t *d_row_idx, const void *d_row_A, const void *d_row_C,
                                 const uint32_t *d_col_idx, const void *d_col_W, const void *d_col_C,
                                 const uint32_t *d_counts, uint8_t *d_differs, uint32_t *d_summary, void *d_ws,
                                 size_t ws_bytes, sdc_stream_t stream) {
    if (!d_row_idx || !d_row_A || !d_row_C || !d_col_idx || !d_col_W || !d_col_C || !d_counts || !d_differs ||
        !d_summary || !d_ws)
        return fail(SDC_ERR_NULL, "NULL argument");
    if (M == 0 || N == 0 || K == 0 || N % 8 || K % 8 || K > (1u << 20) || cap_rows == 0 || cap_cols == 0 ||
        cap_rows > kMaxPairs || cap_cols > kMaxPairs)
        return fail(SDC_ERR_BAD_ARG, "M positive, N and K multiples of 8, K <= 2^20, cap_rows and cap_cols in 1..64");
    const ReplayPairsWs w = replay_pairs_ws(K, cap_rows, cap_cols);
    if (ws_bytes < w.total) return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_replay_pairs_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    if (((uint64_t)d_row_A | (uint64_t)d_col_W) & 15u) return fail(SDC_ERR_BAD_POINTER, "row buffers must be 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_spans({{d_row_idx, (uint64_t)cap_rows * 4, "d_row_idx"},
                                 {d_row_A, (uint64_t)cap_rows * K * 2, "d_row_A"},
                                 {d_row_C, (uint64_t)cap_rows * N * 2, "d_row_C"},
                                 {d_col_idx, (uint64_t)cap_cols * 4, "d_col_idx"},
                                 {d_col_W, (uint64_t)cap_cols * K * 2, "d_col_W"},
                                 {d_col_C, (uint64_t)cap_cols * M * 2, "d_col_C"},
                                 {d_counts, 8, "d_counts"},
                                 {d_differs, (uint64_t)cap_rows * cap_cols, "d_differs"},
                                 {d_summary, 8, "d_summary"},
                                 {d_ws, w.total, "d_ws"}},
                                dev);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)d_ws;
    const uint32_t m = cap_rows * kRowTile, n = cap_cols * kColTile;
    e = cudaMemsetAsync(ws + w.sa, 0, w.out - w.sa, s);  // both staged operands
    if (e == cudaSuccess) e = cudaMemsetAsync(d_summary, 0, 8, s);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_replay_pairs setup");
    // row i of A at lane i mod 128 of tile r, row j of W (B's column j) at column j mod 256 of tile c
    stage_rows_kernel<<<cap_rows, 256, 0, s>>>((const __nv_bfloat16 *)d_row_A, K, d_row_idx, d_counts, cap_rows,
                                               kRowTile, (__nv_bfloat16 *)(ws + w.sa));
    stage_rows_kernel<<<cap_cols, 256, 0, s>>>((const __nv_bfloat16 *)d_col_W, K, d_col_idx, d_counts + 1, cap_cols,
                                               kColTile, (__nv_bfloat16 *)(ws + w.sw));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_replay_pairs launch");
    st = sdc_abft_gemm(ws + w.sa, ws + w.sw, ws + w.out, m, n, K, (double *)(ws + w.rowsum), nullptr,
                       (uint32_t *)(ws + w.aborted), ws + w.gemm, w.gemm_bytes, stream);
    if (st != SDC_OK) return st;
    // the output at (row i, column j): row r's element j (d_row_C [cap_r][N]) and column c's element i
    // (d_col_C [cap_c][M]), the layouts the weight-gradient pairs have with N, K in place of M, N
    compare_pairs_kernel<<<(cap_rows * cap_cols + 255) / 256, 256, 0, s>>>(
        (const uint16_t *)(ws + w.out), cap_rows, cap_cols, M, N, d_row_idx, (const uint16_t *)d_row_C, d_col_idx,
        (const uint16_t *)d_col_C, d_counts, d_differs, d_summary);
    copy_word_kernel<<<1, 1, 0, s>>>((const uint32_t *)(ws + w.aborted), d_summary + 1);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_replay_pairs launch");
}

}  // extern "C"
