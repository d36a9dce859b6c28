/* A plain C caller of libsdc (include/sdc.h), used by tests/test_gpu_c_abi.py.
 *
 * Reads R replicas of T tensors from a file, copies every tensor into its own
 * device allocation, builds a plan, fingerprints the copies and votes, and
 * prints the fingerprint table, the per-tensor suspects and the summary.  The
 * test compares what it prints with the oracle on the same bytes.
 *
 * Input file (little-endian): uint32 R, uint32 T; T x {uint64 numel, uint32
 * elem_size}; then the bytes of tensor 0..T-1 of replica 0, of replica 1, ...
 * Output lines: "fp r t S W" (S, W in hex), "suspect t code mask",
 * "summary diverged no_majority suspect_mask".
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "sdc.h"

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

int main(int argc, char **argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s input.bin\n", argv[0]);
        return 2;
    }
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 2;
    uint32_t R = 0, T = 0;
    if (read_exact(f, &R, 4) || read_exact(f, &T, 4)) return 2;
    uint64_t *numel = calloc(T ? T : 1, sizeof(uint64_t));
    uint32_t *esize = calloc(T ? T : 1, sizeof(uint32_t));
    for (uint32_t t = 0; t < T; ++t)
        if (read_exact(f, &numel[t], 8) || read_exact(f, &esize[t], 4)) return 2;

    /* every copy in a device allocation of its own, as separate framework tensors would be */
    sdc_tensor_desc *desc = calloc((size_t)R * T + 1, sizeof(sdc_tensor_desc));
    void **dptr = calloc((size_t)R * T + 1, sizeof(void *));
    for (uint32_t r = 0; r < R; ++r) {
        for (uint32_t t = 0; t < T; ++t) {
            const size_t bytes = (size_t)numel[t] * esize[t];
            void *host = malloc(bytes ? bytes : 1);
            if (read_exact(f, host, bytes)) return 2;
            void *d = NULL;
            if (bytes) {
                CUDA(cudaMalloc(&d, bytes));
                CUDA(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
            }
            free(host);
            dptr[(size_t)r * T + t] = d;
            desc[(size_t)r * T + t].ptr = d;
            desc[(size_t)r * T + t].numel = numel[t];
            desc[(size_t)r * T + t].elem_size = esize[t];
            desc[(size_t)r * T + t].dtype = SDC_DTYPE_RAW;
        }
    }
    fclose(f);

    sdc_plan *plan = NULL;
    SDC(sdc_plan_create(desc, T, R, NULL, &plan));
    const size_t ws_bytes = sdc_workspace_size(plan);
    void *d_ws = NULL;
    uint64_t *d_fp = NULL, *d_mask = NULL;
    int32_t *d_suspect = NULL;
    sdc_vote_summary *d_summary = NULL;
    CUDA(cudaMalloc(&d_ws, ws_bytes ? ws_bytes : 256));
    CUDA(cudaMalloc((void **)&d_fp, (size_t)R * T * 2 * sizeof(uint64_t) + 16));
    CUDA(cudaMalloc((void **)&d_suspect, (size_t)T * sizeof(int32_t) + 16));
    CUDA(cudaMalloc((void **)&d_mask, (size_t)T * sizeof(uint64_t) + 16));
    CUDA(cudaMalloc((void **)&d_summary, sizeof(sdc_vote_summary)));
    SDC(sdc_fingerprint(plan, d_fp, d_ws, ws_bytes, NULL));
    SDC(sdc_vote(d_fp, R, T, d_suspect, d_mask, d_summary, NULL));
    CUDA(cudaDeviceSynchronize());

    uint64_t *fp = malloc((size_t)R * T * 2 * sizeof(uint64_t) + 16);
    int32_t *suspect = malloc((size_t)T * sizeof(int32_t) + 16);
    uint64_t *mask = malloc((size_t)T * sizeof(uint64_t) + 16);
    sdc_vote_summary summary;
    CUDA(cudaMemcpy(fp, d_fp, (size_t)R * T * 2 * sizeof(uint64_t), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(suspect, d_suspect, (size_t)T * sizeof(int32_t), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(mask, d_mask, (size_t)T * sizeof(uint64_t), cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&summary, d_summary, sizeof(summary), cudaMemcpyDeviceToHost));
    for (uint32_t r = 0; r < R; ++r)
        for (uint32_t t = 0; t < T; ++t)
            printf("fp %u %u %llx %llx\n", r, t, (unsigned long long)fp[((size_t)r * T + t) * 2],
                   (unsigned long long)fp[((size_t)r * T + t) * 2 + 1]);
    for (uint32_t t = 0; t < T; ++t)
        printf("suspect %u %d %llx\n", t, suspect[t], (unsigned long long)mask[t]);
    printf("summary %u %u %llx\n", summary.diverged, summary.no_majority, (unsigned long long)summary.suspect_mask);

    SDC(sdc_plan_destroy(plan));
    for (size_t i = 0; i < (size_t)R * T; ++i)
        if (dptr[i]) CUDA(cudaFree(dptr[i]));
    CUDA(cudaFree(d_ws));
    CUDA(cudaFree(d_fp));
    CUDA(cudaFree(d_suspect));
    CUDA(cudaFree(d_mask));
    CUDA(cudaFree(d_summary));
    free(fp);
    free(suspect);
    free(mask);
    free(desc);
    free(dptr);
    free(numel);
    free(esize);
    return 0;
}
