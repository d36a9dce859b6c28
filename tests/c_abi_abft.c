/* A plain C caller of libsdc's GEMM checksum calls (include/sdc.h), used by
 * tests/test_gpu_c_abi.py.
 *
 * Reads A [M][K], W [N][K] (the weights the check trusts) and Wp [N][K] (the
 * weights the product reads: W itself, or a copy with a fault in it), all
 * bfloat16 bits, from a file.  Runs, on the default stream:
 *   1. the product with row and column checksums (sdc_abft_gemm on A, Wp),
 *      then the verifier against A and W (sdc_abft_verify);
 *   2. W's column sums and the product with its row check fused into it
 *      (sdc_abft_weight_sums on W, sdc_abft_gemm_checked on A, Wp);
 *   3. the replay context of what step 1 flagged and its (row, column) pair
 *      replay (sdc_abft_capture, sdc_abft_replay_pairs), caps of CAP each.
 * Prints what each step returned; writes step 1's C to the output file so the
 * test can form the oracle's capture from the same bits.
 *
 * Input file (little-endian): uint32 M, N, K; then the bits of A, W and Wp.
 * Output lines: "gemm aborted", "rowsum i hexfloat", "colsum j hexfloat",
 * "verify n_flagged n_flagged_cols", "flag i", "flagcol j",
 * "checked aborted n_flagged n_flagged_cols c_equal", "checkedflag i",
 * "capture n_rows n_cols", "rowidx r i", "colidx c j", "differs r c v",
 * "replay n_differ aborted".
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "sdc.h"

#define CAP 4u

#define SDC(call)                                                                                     \
    do {                                                                                              \
        sdc_status st_ = (call);                                                                      \
        if (st_ != SDC_OK) {                                                                          \
            fprintf(stderr, "%s: %s (%s)\n", #call, sdc_status_string(st_), sdc_last_error());      \
            return 1;                                                                                 \
        }                                                                                             \
    } while (0)
#define CUDA(call)                                                                                    \
    do {                                                                                              \
        cudaError_t e_ = (call);                                                                      \
        if (e_ != cudaSuccess) {                                                                      \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                              \
            return 1;                                                                                 \
        }                                                                                             \
    } while (0)

static int read_exact(FILE *f, void *dst, size_t n) { return fread(dst, 1, n, f) == n ? 0 : 1; }

/* a device buffer of at least one byte */
static void *dev_alloc(size_t bytes) {
    void *p = NULL;
    return cudaMalloc(&p, bytes ? bytes : 1) == cudaSuccess ? p : NULL;
}

static size_t max_size(size_t a, size_t b) { return a > b ? a : b; }

int main(int argc, char **argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s input.bin c_out.bin\n", argv[0]);
        return 2;
    }
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 2;
    uint32_t M = 0, N = 0, K = 0;
    if (read_exact(f, &M, 4) || read_exact(f, &N, 4) || read_exact(f, &K, 4)) return 2;
    const size_t a_bytes = (size_t)M * K * 2, w_bytes = (size_t)N * K * 2, c_bytes = (size_t)M * N * 2;
    uint16_t *hA = malloc(a_bytes), *hW = malloc(w_bytes), *hWp = malloc(w_bytes);
    if (!hA || !hW || !hWp) return 2;
    if (read_exact(f, hA, a_bytes) || read_exact(f, hW, w_bytes) || read_exact(f, hWp, w_bytes)) return 2;
    fclose(f);

    void *dA = dev_alloc(a_bytes), *dW = dev_alloc(w_bytes), *dWp = dev_alloc(w_bytes);
    void *dC = dev_alloc(c_bytes), *dC2 = dev_alloc(c_bytes);
    double *d_rowsum = dev_alloc((size_t)M * 8), *d_colsum = dev_alloc((size_t)N * 8);
    double *d_res = dev_alloc((size_t)M * 8), *d_bnd = dev_alloc((size_t)M * 8);
    double *d_res_col = dev_alloc((size_t)N * 8), *d_bnd_col = dev_alloc((size_t)N * 8);
    uint8_t *d_flag = dev_alloc(M), *d_flag_col = dev_alloc(N), *d_flag2 = dev_alloc(M);
    double *d_rowsum2 = dev_alloc((size_t)M * 8), *d_res2 = dev_alloc((size_t)M * 8), *d_bnd2 = dev_alloc((size_t)M * 8);
    sdc_abft_summary *d_summ = dev_alloc(sizeof(sdc_abft_summary)), *d_summ2 = dev_alloc(sizeof(sdc_abft_summary));
    uint32_t *d_aborted = dev_alloc(4), *d_aborted2 = dev_alloc(4);
    float *d_wsums = dev_alloc((size_t)K * 2 * sizeof(float));
    const size_t ws_bytes = max_size(sdc_abft_workspace_size(M, N, K),
                                     max_size(sdc_abft_weight_sums_workspace_size(N, K),
                                              sdc_abft_gemm_checked_workspace_size(M, N, K)));
    const size_t rp_bytes = sdc_abft_replay_pairs_workspace_size(K, CAP, CAP);
    void *d_ws = dev_alloc(ws_bytes), *d_rpws = dev_alloc(rp_bytes);
    uint32_t *d_row_idx = dev_alloc(CAP * 4), *d_col_idx = dev_alloc(CAP * 4), *d_counts = dev_alloc(8);
    void *d_row_A = dev_alloc((size_t)CAP * K * 2), *d_row_C = dev_alloc((size_t)CAP * N * 2);
    void *d_col_W = dev_alloc((size_t)CAP * K * 2), *d_col_C = dev_alloc((size_t)CAP * M * 2);
    uint8_t *d_differs = dev_alloc(CAP * CAP);
    uint32_t *d_rsumm = dev_alloc(8);
    if (!dA || !dW || !dWp || !dC || !dC2 || !d_rowsum || !d_colsum || !d_res || !d_bnd || !d_res_col ||
        !d_bnd_col || !d_flag || !d_flag_col || !d_flag2 || !d_rowsum2 || !d_res2 || !d_bnd2 || !d_summ ||
        !d_summ2 || !d_aborted || !d_aborted2 || !d_wsums || !d_ws || !d_rpws || !d_row_idx || !d_col_idx ||
        !d_counts || !d_row_A || !d_row_C || !d_col_W || !d_col_C || !d_differs || !d_rsumm) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 1;
    }
    CUDA(cudaMemcpy(dA, hA, a_bytes, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dW, hW, w_bytes, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dWp, hWp, w_bytes, cudaMemcpyHostToDevice));
    if (ws_bytes == 0 || rp_bytes == 0) {
        fprintf(stderr, "shape rejected by a workspace query\n");
        return 1;
    }

    /* 1. product with both checksums, then the verifier against the trusted W */
    SDC(sdc_abft_gemm(dA, dWp, dC, M, N, K, d_rowsum, d_colsum, d_aborted, d_ws, ws_bytes, NULL));
    SDC(sdc_abft_verify(dA, dW, M, N, K, d_rowsum, d_colsum, 1.0f, d_res, d_bnd, d_flag, d_res_col, d_bnd_col,
                        d_flag_col, d_summ, d_ws, ws_bytes, NULL));
    /* 2. the fused row check */
    SDC(sdc_abft_weight_sums(dW, N, K, d_wsums, d_ws, ws_bytes, NULL));
    SDC(sdc_abft_gemm_checked(dA, dWp, dC2, M, N, K, d_wsums, 1.0f, d_rowsum2, d_res2, d_bnd2, d_flag2, d_summ2,
                              d_aborted2, d_ws, ws_bytes, NULL));
    /* 3. the replay context of step 1's flags and its pair replay */
    SDC(sdc_abft_capture(dA, dW, dC, M, N, K, d_flag, d_flag_col, CAP, d_row_idx, d_row_A, d_row_C, CAP, d_col_idx,
                         d_col_W, d_col_C, d_counts, NULL));
    SDC(sdc_abft_replay_pairs(M, N, K, CAP, CAP, d_row_idx, d_row_A, d_row_C, d_col_idx, d_col_W, d_col_C, d_counts,
                              d_differs, d_rsumm, d_rpws, rp_bytes, NULL));
    CUDA(cudaDeviceSynchronize());

    uint16_t *hC = malloc(c_bytes ? c_bytes : 1), *hC2 = malloc(c_bytes ? c_bytes : 1);
    double *rowsum = malloc((size_t)M * 8), *colsum = malloc((size_t)N * 8);
    uint8_t *flag = malloc(M), *flag_col = malloc(N), *flag2 = malloc(M);
    if (!hC || !hC2 || !rowsum || !colsum || !flag || !flag_col || !flag2) return 1;
    sdc_abft_summary summ, summ2;
    uint32_t aborted, aborted2, counts[2], row_idx[CAP], col_idx[CAP], rsumm[2];
    uint8_t differs[CAP * CAP];
    CUDA(cudaMemcpy(hC, dC, c_bytes, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(hC2, dC2, c_bytes, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(rowsum, d_rowsum, (size_t)M * 8, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(colsum, d_colsum, (size_t)N * 8, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(flag, d_flag, M, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(flag_col, d_flag_col, N, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(flag2, d_flag2, M, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&summ, d_summ, sizeof(summ), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&summ2, d_summ2, sizeof(summ2), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&aborted, d_aborted, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&aborted2, d_aborted2, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(counts, d_counts, 8, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(row_idx, d_row_idx, CAP * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(col_idx, d_col_idx, CAP * 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(differs, d_differs, CAP * CAP, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(rsumm, d_rsumm, 8, cudaMemcpyDeviceToHost));

    FILE *out = fopen(argv[2], "wb");
    if (!out || fwrite(hC, 1, c_bytes, out) != c_bytes) return 2;
    fclose(out);

    printf("gemm %u\n", aborted);
    for (uint32_t i = 0; i < M; ++i) printf("rowsum %u %a\n", i, rowsum[i]);
    for (uint32_t j = 0; j < N; ++j) printf("colsum %u %a\n", j, colsum[j]);
    printf("verify %u %u\n", summ.n_flagged, summ.n_flagged_cols);
    for (uint32_t i = 0; i < M; ++i)
        if (flag[i]) printf("flag %u\n", i);
    for (uint32_t j = 0; j < N; ++j)
        if (flag_col[j]) printf("flagcol %u\n", j);
    printf("checked %u %u %u %d\n", aborted2, summ2.n_flagged, summ2.n_flagged_cols, memcmp(hC, hC2, c_bytes) == 0);
    for (uint32_t i = 0; i < M; ++i)
        if (flag2[i]) printf("checkedflag %u\n", i);
    printf("capture %u %u\n", counts[0], counts[1]);
    const uint32_t nr = counts[0] < CAP ? counts[0] : CAP, nc = counts[1] < CAP ? counts[1] : CAP;
    for (uint32_t r = 0; r < nr; ++r) printf("rowidx %u %u\n", r, row_idx[r]);
    for (uint32_t c = 0; c < nc; ++c) printf("colidx %u %u\n", c, col_idx[c]);
    for (uint32_t r = 0; r < CAP; ++r)
        for (uint32_t c = 0; c < CAP; ++c) printf("differs %u %u %u\n", r, c, differs[r * CAP + c]);
    printf("replay %u %u\n", rsumm[0], rsumm[1]);

    void *bufs[] = {dA, dW, dWp, dC, dC2, d_rowsum, d_colsum, d_res, d_bnd, d_res_col, d_bnd_col, d_flag,
                    d_flag_col, d_flag2, d_rowsum2, d_res2, d_bnd2, d_summ, d_summ2, d_aborted, d_aborted2,
                    d_wsums, d_ws, d_rpws, d_row_idx, d_col_idx, d_counts, d_row_A, d_row_C, d_col_W, d_col_C,
                    d_differs, d_rsumm};
    for (size_t b = 0; b < sizeof(bufs) / sizeof(bufs[0]); ++b) CUDA(cudaFree(bufs[b]));
    free(hA);
    free(hW);
    free(hWp);
    free(hC);
    free(hC2);
    free(rowsum);
    free(colsum);
    free(flag);
    free(flag_col);
    free(flag2);
    return 0;
}
