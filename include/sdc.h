/*
 * sdc.h -- C ABI of libsdc, the replica-integrity scan for one GB300 GPU.
 *
 * The method comes from "Detecting and recovering from silent data corruption
 * on Amazon SageMaker HyperPod" (AWS Machine Learning Blog; cited below as
 * [AWS]) and, for the xorsum, from the review page "Safeguarding LLM Training
 * at Scale: Online SDC Detection and Insights from 35 Million GPU Hours"
 * (cited as [AEGIS]).  Data-parallel training keeps R copies ("replicas") of
 * every weight tensor; after each optimizer step the copies must be identical
 * bit for bit.  This library reduces every copy of every tensor to a small
 * fingerprint, votes on the fingerprints, and scans gradient buffers for NaN,
 * Inf and float32 overflow while computing their L2 norm.
 *
 * Conventions shared by every call:
 *  - All data pointers named d_* point to device memory of the CURRENT device
 *    (cudaGetDevice() when the call is made); the caller allocates and owns
 *    them.  Host arrays are named host_* or documented as host arrays.
 *  - Every compute call is asynchronous: it validates its arguments on the
 *    host, enqueues its kernels on `stream` and returns; results appear in
 *    device memory in stream order.  No compute call synchronises the device
 *    or allocates device memory; only sdc_plan_create and
 *    sdc_opt_state_create allocate (their tables, uploaded with a synchronous
 *    cudaMemcpy), and only their destroy calls free (cudaFree, which may wait
 *    for work queued on the device).
 *  - `stream` is a cudaStream_t (same type; NULL = the legacy default stream).
 *  - Errors are returned as sdc_status codes, checked before anything is
 *    enqueued; nothing is enqueued when a call fails.  Every d_* array a call
 *    reads or writes, and its workspace, is checked against the allocation
 *    that holds it (SDC_ERR_BAD_POINTER when it is not device memory of the
 *    current device or the bytes the call touches run past its end).  sdc_last_error()
 *    returns a one-line detail for the calling thread's last failure.  No
 *    kernel traps or asserts.
 *  - A workspace (d_ws) holds a call's intermediate values and counters,
 *    which the call resets itself: calls that share one workspace must not
 *    overlap on the GPU (order them on one stream, or give each its own).
 *  - Tensors are contiguous (the page fingerprints t.contiguous()) and their
 *    element order is the flat row-major order.  Start addresses need only be
 *    aligned to the element size.
 *  - Replica-major layout: the fingerprint table of R replicas x T tensors is
 *    uint64 out[R][T][2]; entry (r, k) describes replica r's copy of tensor k.
 */
#ifndef SDC_H
#define SDC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *sdc_stream_t;

typedef int sdc_status;
enum {
    SDC_OK = 0,
    SDC_ERR_NULL = 1,              /* a required pointer argument is NULL */
    SDC_ERR_BAD_ELEM_SIZE = 2,     /* element size not in {1, 2, 4, 8} or not matching dtype */
    SDC_ERR_SHAPE_MISMATCH = 3,    /* replicas of one tensor differ in numel/elem_size/dtype */
    SDC_ERR_TOO_MANY_REPLICAS = 4, /* R == 0 or R > SDC_MAX_REPLICAS, or too many buffers */
    SDC_ERR_WS_TOO_SMALL = 5,      /* workspace smaller than the size query returned */
    SDC_ERR_CUDA = 6,              /* a CUDA runtime call failed (see sdc_last_error) */
    SDC_ERR_BAD_DTYPE = 7,         /* dtype code unknown, or not a float type where one is needed */
    SDC_ERR_BAD_POINTER = 8,       /* not device memory of the current device, misaligned,
                                      or [ptr, ptr + bytes) leaves its allocation */
    SDC_ERR_BAD_ARG = 9,           /* any other invalid argument (sizes, options) */
    SDC_ERR_WRONG_DEVICE = 10      /* plan used on a device other than the one it was built on */
};

#define SDC_MAX_REPLICAS 64

/* dtype codes.  RAW: fingerprint/xorsum only (bits are bits).  The grad calls
 * need a float dtype: F32 (elem_size 4), BF16 or F16 (elem_size 2). */
enum { SDC_DTYPE_RAW = 0, SDC_DTYPE_F32 = 1, SDC_DTYPE_BF16 = 2, SDC_DTYPE_F16 = 3 };

/* One tensor copy.  ptr: device address of element 0 (may be NULL only if
 * numel == 0); numel: number of elements; elem_size: 1, 2, 4 or 8 bytes;
 * dtype: one of SDC_DTYPE_*. */
typedef struct {
    const void *ptr;
    uint64_t numel;
    uint32_t elem_size;
    uint32_t dtype;
} sdc_tensor_desc;

/* Plan options; a zero field takes its default.  chunk_bytes: bytes of one
 * warp task, a power of two in [4096, 32768] (default 16384, halved down to
 * 4096 while the plan would give fewer than 16 tasks per warp of the
 * persistent grid: 32 warps per SM); ctas_per_sm:
 * resident CTAs per SM of the persistent kernels (default: the occupancy
 * limit); skip_pointer_checks: 1 skips the driver queries that check every
 * descriptor's range lies inside one device allocation of this device. */
typedef struct {
    uint32_t chunk_bytes;
    uint32_t ctas_per_sm;
    uint32_t skip_pointer_checks;
    uint32_t reserved;
} sdc_plan_opts;

/* Opaque plan: the validated descriptor table and its chunk table, resident
 * in device memory.  Built once per parameter set -- training frameworks keep
 * parameter storage fixed between steps. */
typedef struct sdc_plan sdc_plan;

/* Gradient statistics of one buffer (or one replica's tensors).
 *  n_nan, n_inf: NaN and +-Inf elements;
 *  n_big: finite elements whose exact square exceeds FLT_MAX (|x| > ~1.8e19);
 *  n_elems: elements scanned;
 *  sumsq_finite: sum of x^2 over finite elements, float64;
 *  norm: sqrt(sumsq_finite), except NaN if any element is NaN, else +Inf if
 *        any element is +-Inf (IEEE propagation, as clip_grad_norm_ reports);
 *  nonfinite_fp32: 1 if the float32 squared norm would not be finite:
 *        n_nan > 0 or n_inf > 0 or sumsq_finite > FLT_MAX -- [AWS] "Decide
 *        what the alarm means": a norm above about 1.8e19 counts as non-finite. */
typedef struct {
    uint64_t n_nan;
    uint64_t n_inf;
    uint64_t n_big;
    uint64_t n_elems;
    double sumsq_finite;
    double norm;
    uint32_t nonfinite_fp32;
    uint32_t reserved;
} sdc_grad_stats;

/* Vote summary.  diverged: some tensor's copies differ; no_majority: some
 * differing tensor has no strict majority; suspect_mask: bit r set when
 * replica r differs from a strict majority on some tensor that has one;
 * n_differing / n_no_majority: tensor counts.  The page's result
 * {"diverged", "suspects"} is: not diverged -> suspects = [];
 * no_majority -> suspects = None; otherwise suspects = bits of suspect_mask. */
typedef struct {
    uint32_t diverged;
    uint32_t no_majority;
    uint64_t suspect_mask;
    uint32_t n_differing;
    uint32_t n_no_majority;
} sdc_vote_summary;

/* Per-tensor suspect codes written by sdc_vote. */
#define SDC_SUSPECT_AGREE (-1)       /* every copy agrees */
#define SDC_SUSPECT_SEVERAL (-2)     /* several copies differ from a strict majority (see mask) */
#define SDC_SUSPECT_NO_MAJORITY (-3) /* copies differ and no value has a strict majority */

/* ---------------------------------------------------------------- plan */

/* Build a plan over R replicas x T tensors.  host_descs: host array of R*T
 * descriptors in replica-major order (entry r*T + k is replica r's copy of
 * tensor k); every replica's copy of tensor k must have the same numel,
 * elem_size and dtype.  The descriptors are copied; the plan does not keep
 * host_descs.  Allocates the plan's device tables on the current device.
 * opts may be NULL.  On success *out receives the plan.
 * [AWS] "Compare by fingerprint": the fingerprint function allocates one row
 * of two int64 per tensor; "Check 3": every rank fingerprints every weight. */
sdc_status sdc_plan_create(const sdc_tensor_desc *host_descs, uint32_t T, uint32_t R,
                           const sdc_plan_opts *opts, sdc_plan **out);

/* Free a plan and its device tables with cudaFree (which may wait for work
 * queued on the device); the caller must not destroy a plan whose work is
 * still queued or will be.  NULL is accepted. */
sdc_status sdc_plan_destroy(sdc_plan *plan);

/* Bytes of device workspace the plan's compute calls need: per-chunk partials
 * plus the group sums of the statistics combine.  Any 256-byte-aligned device
 * buffer at least this large works; its contents need no initialisation.
 * Calls that share one workspace must not overlap on the GPU. */
size_t sdc_workspace_size(const sdc_plan *plan);

/* Plan facts for reporting: chunk count, persistent grid and block size. */
sdc_status sdc_plan_info(const sdc_plan *plan, uint64_t *n_chunks, uint32_t *grid, uint32_t *block);

/* ---------------------------------------------------------------- fingerprint */

/* Weight fingerprints.  [AWS] "Compare by fingerprint": each tensor is
 * reduced to two 64-bit sums of its raw bit patterns, one plain and one
 * weighted by position.  The element bits b_i are read through the integer
 * type of the element width (unsigned 8-bit, or signed 16/32/64-bit) and
 * widened to 64 bits (zero-extension for 1-byte, sign-extension otherwise):
 *     S = sum_i b_i  mod 2^64,     W = sum_i (i + 1) * b_i  mod 2^64.
 * d_out: device uint64[R][T][2], (S, W) of replica r's copy of tensor k at
 * d_out[(r*T + k)*2 + {0, 1}]; the bits equal the page's int64 values.
 * d_ws: device workspace of ws_bytes >= sdc_workspace_size(plan).
 * Results are exact integers: identical on every run and any launch shape. */
sdc_status sdc_fingerprint(const sdc_plan *plan, uint64_t *d_out, void *d_ws, size_t ws_bytes,
                           sdc_stream_t stream);

/* Xorsum fingerprints.  [AEGIS] method section 4: an original and a
 * recomputed result are each reduced to an xorsum fingerprint; any differing
 * bit is an anomaly.  Read here as the XOR over elements of each element's
 * raw bits zero-extended to 64 bits.  d_out: device uint64[R][T]. */
sdc_status sdc_xorsum(const sdc_plan *plan, uint64_t *d_out, void *d_ws, size_t ws_bytes,
                      sdc_stream_t stream);

/* Compare two xorsum vectors of n entries: d_mismatch[p] = (d_a[p] != d_b[p]),
 * d_diff[p] = d_a[p] ^ d_b[p].  d_mismatch: device uint8[n]; d_diff: device
 * uint64[n] (may be NULL).  n == 0 is a no-op. */
sdc_status sdc_xorsum_compare(const uint64_t *d_a, const uint64_t *d_b, uint32_t n,
                              uint8_t *d_mismatch, uint64_t *d_diff, sdc_stream_t stream);

/* ---------------------------------------------------------------- vote */

/* Strict-majority vote over a fingerprint table.  [AWS] "Check 3: Weight
 * fingerprints, after the optimizer step": a copy is named only when it
 * differs from a strict majority (more than half of the copies); with two
 * copies, or a split with no strict majority, a disagreement is reported
 * without naming anyone.  d_fp: device uint64[R][T][2] (as sdc_fingerprint
 * writes it); 1 <= R <= SDC_MAX_REPLICAS.  Outputs: d_suspect: device
 * int32[T] (SDC_SUSPECT_* or the one replica that differs); d_mask: device
 * uint64[T], bit r set when replica r differs from the majority (0 when all
 * agree or no majority exists); d_summary: device sdc_vote_summary. */
sdc_status sdc_vote(const uint64_t *d_fp, uint32_t R, uint32_t T, int32_t *d_suspect, uint64_t *d_mask,
                    sdc_vote_summary *d_summary, sdc_stream_t stream);

/* ---------------------------------------------------------------- optimizer step + fingerprint */

/* AdamW hyperparameters of one step.  step: the step number, counting from 1
 * (for the bias corrections); clip: 1 scales the gradient by
 * min(1, max_grad_norm / (norm + 1e-6)) with `norm` the reduced gradient's
 * global L2 norm (as clip_grad_norm_ does). */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    float max_grad_norm;
    uint32_t step;
    uint32_t clip;
} sdc_adamw_hparams;

/* Opaque per-plan table of each weight's averaged gradient and AdamW moments. */
typedef struct sdc_opt_state sdc_opt_state;

/* Attach optimizer tensors to a plan whose descriptors are F32 weights (R
 * replicas x T tensors).  host_grads: HOST array of T device pointers, the
 * averaged gradient of tensor k (shared by all replicas: every replica applies
 * the same average), each numel elements of grad_dtype (F32, BF16 or F16);
 * host_exp_avg, host_exp_avg_sq: HOST arrays of R*T device pointers to float32
 * moments, replica-major like the plan.  Copies the pointers to a device
 * table (allocated here).  The tensors must outlive the state. */
sdc_status sdc_opt_state_create(const sdc_plan *plan, const void *const *host_grads, uint32_t grad_dtype,
                                void *const *host_exp_avg, void *const *host_exp_avg_sq, sdc_opt_state **out);
sdc_status sdc_opt_state_destroy(sdc_opt_state *state);

/* One pass over every replica's weights: clip, AdamW step, and the weight
 * fingerprint of the values written.  [AWS] `train()`: clip the reduced
 * gradient, skip the step when it is NaN/Inf, step the optimizer; "Check 3":
 * fingerprint every replica's weights after the update; the use case trains
 * with AdamW (betas 0.9/0.95, weight decay 0.1, clipping at 1.0).
 * d_post: device sdc_grad_stats of the reduced (averaged) gradient, as
 * sdc_grad_average_scan writes it; when its nonfinite_fp32 is set nothing is
 * updated (the step is skipped on the device, no host round trip) and the
 * fingerprints are those of the unchanged weights.  May be NULL when clip is
 * 0 (no gate).  Per element, in float32 with every operation separately
 * rounded: g = grad * coef; p = p * (1 - lr*wd); m = m + (1 - beta1) * (g - m);
 * v = v * beta2 + (g*g) * (1 - beta2); d = sqrt(v) / sqrt(1 - beta2^step) + eps;
 * p = p - (lr / (1 - beta1^step)) * (m / d); the scalars in parentheses are
 * formed in double and rounded once to float32.  d_fp_out: device
 * uint64[R][T][2] as sdc_fingerprint.  d_ws: the plan's workspace.  This
 * fingerprints values as written; a separate sdc_fingerprint re-read of the
 * stored weights still checks corruption after the write. */
sdc_status sdc_adamw_fingerprint(const sdc_plan *plan, const sdc_opt_state *state, const sdc_adamw_hparams *hp,
                                 const sdc_grad_stats *d_post, uint64_t *d_fp_out, void *d_ws, size_t ws_bytes,
                                 sdc_stream_t stream);

/* ---------------------------------------------------------------- GEMM checksums (AEGIS) */

/* Counts written by sdc_abft_verify and sdc_attn_dv_check. */
typedef struct {
    uint32_t n_flagged;      /* GEMM: flagged rows; attention: flagged (head, column) pairs */
    uint32_t n_flagged_cols; /* GEMM: flagged columns (0 without the column check); attention: 0 */
} sdc_abft_summary;

/* Workspace bytes of sdc_abft_gemm / sdc_abft_verify (one buffer may serve both
 * when they are ordered on one stream). */
size_t sdc_abft_workspace_size(uint32_t M, uint32_t N, uint32_t K);

/* The checksum sensor: C = A . W^T on the tensor cores (tcgen05, accumulator
 * in TMEM, operands staged by TMA) with each output row's checksum formed
 * from the float32 accumulator before the bfloat16 store.  [AEGIS] method
 * section 2: compare (AB)1 with A(B1), with the checksum taken from the fp32
 * accumulator inside the kernel.  d_A: device bf16 [M][K]; d_W: device bf16
 * [N][K] (both row-major, K contiguous, 16-byte aligned); d_C: device bf16
 * [M][N].  M >= 1; N and K positive multiples of 8 (row strides of 16-byte
 * multiples), K <= 2^20; tiles past M, N or K are filled with zeros, which add
 * nothing to C or to a checksum, and only C itself is written.  d_rowsum: device double
 * [M], sum over j of the fp32 accumulator of C[i][j] (float32 pairs per
 * 256-column tile, tile partials added in a fixed order in float64).
 * d_colsum: NULL, or device double [N] for the page's row + column
 * configuration: sum over i of the fp32 accumulator of C[i][j] (float32 pairs
 * per 32 rows, merged per 128-row tile in a fixed order, tile partials added
 * in a fixed order in float64).  d_aborted: device uint32,
 * 1 if a bounded wait of the GEMM gave up (results then invalid). */
sdc_status sdc_abft_gemm(const void *d_A, const void *d_W, void *d_C, uint32_t M, uint32_t N, uint32_t K,
                         double *d_rowsum, double *d_colsum, uint32_t *d_aborted, void *d_ws, size_t ws_bytes,
                         sdc_stream_t stream);

/* The checksum verifier: per row, the reference A(W^T 1) (float32 pairs,
 * about 48 bits, returned in float64), the residual d_residual[i] =
 * d_rowsum[i] - reference, the rounding bound
 * d_bound[i] = (g (1 + g) + 20 2^-24 + (N + K + 64) 2^-44) mag + 2 K N 2^-126 with
 * g = K 2^-22 and mag an upper bound on sum_k |A[i][k]| sum_j |W[j][k]|
 * (summed in plain float32 and raised by twice its chains' length in units of
 * 2^-24, at most 2 (N/8 + K/4 + 32) 2^-24 of itself).  Each float32
 * accumulation step may lose two units in the last place of its partial sum;
 * the check's own sums and flushed subnormals are covered; so a correct
 * product stays inside the bound.  d_flag[i] = 1 unless
 * |residual| <= tol_scale * bound (a NaN residual flags; tol_scale > 0; the
 * page's adaptive threshold has no published constants).  With d_colsum
 * (from sdc_abft_gemm) the columns are checked too, against (1^T A) W^T:
 * d_residual_col[j], d_bound_col[j] (the same bound with M, the rows summed,
 * in place of N and mag = sum_k sum_i |A[i][k]| |W[j][k]|) and d_flag_col[j];
 * with d_colsum NULL the three column outputs are not touched.  d_summary
 * counts the flagged rows and columns.  Same shapes and workspace as
 * sdc_abft_gemm; K <= 2^20.
 * Errors: SDC_ERR_BAD_ARG for shapes, SDC_ERR_BAD_POINTER for misalignment,
 * SDC_ERR_WS_TOO_SMALL, SDC_ERR_WRONG_DEVICE. */
sdc_status sdc_abft_verify(const void *d_A, const void *d_W, uint32_t M, uint32_t N, uint32_t K, const double *d_rowsum,
                           const double *d_colsum, float tol_scale, double *d_residual, double *d_bound,
                           uint8_t *d_flag, double *d_residual_col, double *d_bound_col, uint8_t *d_flag_col,
                           sdc_abft_summary *d_summary, void *d_ws, size_t ws_bytes, sdc_stream_t stream);

/* Workspace bytes of sdc_abft_weight_sums (0 for shapes it rejects). */
size_t sdc_abft_weight_sums_workspace_size(uint32_t N, uint32_t K);

/* W's column sums for the fused check: d_wsums[2k] = h, the float nearest
 * sum_j W[j][k] (float32 pairs over 8-row chains), d_wsums[2k + 1] = the
 * plain float32 sum of |W[j][k]|.  d_W: device bf16 [N][K] (16-byte aligned);
 * d_wsums: device float [K][2].  They depend on W alone: one call serves
 * every product with the same weights (a training step's micro-batches, its
 * forward and dgrad products) until the weights change. */
sdc_status sdc_abft_weight_sums(const void *d_W, uint32_t N, uint32_t K, float *d_wsums, void *d_ws, size_t ws_bytes,
                                sdc_stream_t stream);

/* The GEMM with its row check fused into it: C = A . W^T with each row's
 * accumulator checksum (as sdc_abft_gemm), and the reference A[i][:] (W^T 1)
 * formed in the same kernel by four more warps on the CUDA cores from the
 * A tiles the product stages in shared memory (one tile of each tile row,
 * against d_wsums from sdc_abft_weight_sums for this W).  [AEGIS] method
 * section 2: the checksum and its check inside the GEMM kernel.  The check
 * reads no operand again from HBM; its reference covers the tensor cores and
 * the accumulator, not the copies into shared memory (which sdc_abft_verify,
 * reading A and W from HBM, also covers).  d_residual, d_bound, d_flag and
 * d_summary->n_flagged as sdc_abft_verify's rows, with the same bound (the
 * magnitude's raise from W's column sums and a 32-term chain per 64-column
 * stage); d_summary->n_flagged_cols = 0.  Tile (m, n) of the product forms
 * the references of its 128 rows over the K blocks kb with
 * kb mod ceil(N/256) = n, so the work spreads over all tiles; the partials
 * are merged per row in a fixed order (eight interleaved runs of tiles, then
 * the runs in order).  Shapes, d_rowsum and d_aborted as
 * sdc_abft_gemm; tol_scale > 0; the workspace is
 * sdc_abft_gemm_checked_workspace_size bytes. */
size_t sdc_abft_gemm_checked_workspace_size(uint32_t M, uint32_t N, uint32_t K);
sdc_status sdc_abft_gemm_checked(const void *d_A, const void *d_W, void *d_C, uint32_t M, uint32_t N, uint32_t K,
                                 const float *d_wsums, float tol_scale, double *d_rowsum, double *d_residual,
                                 double *d_bound, uint8_t *d_flag, sdc_abft_summary *d_summary, uint32_t *d_aborted,
                                 void *d_ws, size_t ws_bytes, sdc_stream_t stream);

/* Workspace bytes of sdc_abft_gemm_wgrad / sdc_abft_verify_wgrad (one buffer
 * may serve both when they are ordered on one stream). */
size_t sdc_abft_wgrad_workspace_size(uint32_t T, uint32_t N, uint32_t K);

/* The checksum sensor on the weight-gradient product: dW = dY^T . X on the
 * tensor cores, with row and column checksums from the float32 accumulator.
 * [AEGIS] method section 2: the row configuration leaves wgrad partly
 * uncovered; the row + column configuration covers every matmul class.
 * d_dY: device bf16 [T][N], the layer's output gradient; d_X: device bf16
 * [T][K], its input (both token-major, as the backward pass holds them:
 * row-major, 16-byte aligned; the operands reach the tensor cores MN-major,
 * no transposed copy is made); d_dW: device bf16 [N][K].  T >= 1 tokens (the
 * contraction), T <= 2^20; N and K positive multiples of 8.  d_rowsum: device
 * double [N], sum over k of the fp32 accumulator of dW[n][k]; d_colsum: NULL
 * (rows only) or device double [K], sum over n (the same orders as
 * sdc_abft_gemm).  d_aborted: device uint32, 1 if a bounded wait gave up. */
sdc_status sdc_abft_gemm_wgrad(const void *d_dY, const void *d_X, void *d_dW, uint32_t T, uint32_t N, uint32_t K,
                               double *d_rowsum, double *d_colsum, uint32_t *d_aborted, void *d_ws, size_t ws_bytes,
                               sdc_stream_t stream);

/* The checksum verifier of the weight-gradient product.  Rows: X's row sums
 * r[t] = sum_k X[t][k] weight dY's column sums, the reference of row n is
 * sum_t dY[t][n] r[t] = (dY^T (X 1))[n] and its magnitude
 * sum_t |dY[t][n]| sum_k |X[t][k]|.  Columns (d_colsum given): dY's row sums
 * q[t] weight X's column sums, reference sum_t q[t] X[t][k] and magnitude
 * sum_t (sum_n |dY[t][n]|) |X[t][k]|.  Both in float32 pairs (8-term chains
 * folded in with TwoSum), the magnitudes in plain float32 raised to an upper
 * bound.  The bound is sdc_abft_verify's with the T tokens as the contraction
 * and the outputs a checksum sums (K for a row, N for a column):
 * (g (1 + g) + 20 2^-24 + (n_sum + T + 64) 2^-44) mag + 2 T n_sum 2^-126,
 * g = T 2^-22.  Flags, residuals and d_summary as sdc_abft_verify (rows: N
 * entries; columns: K).  Same shapes and workspace as sdc_abft_gemm_wgrad.
 * Errors: SDC_ERR_BAD_ARG for shapes or tol_scale <= 0, SDC_ERR_NULL,
 * SDC_ERR_BAD_POINTER for misalignment, SDC_ERR_WS_TOO_SMALL,
 * SDC_ERR_WRONG_DEVICE. */
sdc_status sdc_abft_verify_wgrad(const void *d_dY, const void *d_X, uint32_t T, uint32_t N, uint32_t K,
                                 const double *d_rowsum, const double *d_colsum, float tol_scale, double *d_residual,
                                 double *d_bound, uint8_t *d_flag, double *d_residual_col, double *d_bound_col,
                                 uint8_t *d_flag_col, sdc_abft_summary *d_summary, void *d_ws, size_t ws_bytes,
                                 sdc_stream_t stream);

/* ---------------------------------------------------------------- replay context and replay (AEGIS) */

/* The replay context of a checked product C = A . W^T.  [AEGIS] method
 * sections 1 and 2: a check that fires packs its evidence and the least
 * context a replay needs into a vTask; for the forward (and dgrad) product
 * that is the flagged row of A and its output row; with the row + column
 * configuration also each flagged column's operand (W's row j, which is B's
 * column j) and output column.  d_flag: device uint8 [M] (sdc_abft_verify's
 * d_flag, or any selection); d_flag_col: device uint8 [N] or NULL (no
 * columns).  The first cap_rows flagged rows in increasing index are copied:
 * d_row_idx [cap_rows] uint32, d_row_A [cap_rows][K] bf16 (A[i][:]),
 * d_row_C [cap_rows][N] bf16 (C[i][:]); the first cap_cols flagged columns:
 * d_col_idx [cap_cols], d_col_W [cap_cols][K] (W[j][:]), d_col_C
 * [cap_cols][M] (C[:][j]).  d_counts: device uint32 [2], how many rows and
 * columns were flagged (all of them, also past the caps; 0 columns without
 * d_flag_col).  Entries past the counts are not written.  Shapes as
 * sdc_abft_gemm; A, W, C, d_row_A, d_row_C and d_col_W 16-byte aligned. */
sdc_status sdc_abft_capture(const void *d_A, const void *d_W, const void *d_C, uint32_t M, uint32_t N, uint32_t K,
                            const uint8_t *d_flag, const uint8_t *d_flag_col, uint32_t cap_rows, uint32_t *d_row_idx,
                            void *d_row_A, void *d_row_C, uint32_t cap_cols, uint32_t *d_col_idx, void *d_col_W,
                            void *d_col_C, uint32_t *d_counts, sdc_stream_t stream);

/* The replay context of a checked weight gradient dW = dY^T . X (see
 * sdc_abft_gemm_wgrad): per flagged row n of dW, dY's column n (A's row:
 * d_row_dY [cap_rows][T]) and dW[n][:] (d_row_dW [cap_rows][K]); per flagged
 * column k, X's column k (B's column: d_col_X [cap_cols][T]) and dW[:][k]
 * (d_col_dW [cap_cols][N]).  d_flag [N], d_flag_col [K] or NULL; indices,
 * caps and d_counts as sdc_abft_capture.  dW and d_row_dW 16-byte aligned. */
sdc_status sdc_abft_capture_wgrad(const void *d_dY, const void *d_X, const void *d_dW, uint32_t T, uint32_t N,
                                  uint32_t K, const uint8_t *d_flag, const uint8_t *d_flag_col, uint32_t cap_rows,
                                  uint32_t *d_row_idx, void *d_row_dY, void *d_row_dW, uint32_t cap_cols,
                                  uint32_t *d_col_idx, void *d_col_X, void *d_col_dW, uint32_t *d_counts,
                                  sdc_stream_t stream);

/* Workspace bytes of sdc_abft_replay (0 for cap_rows outside 1..1024 or bad
 * N, K): cap_rows x 128 staged rows of K and of N bf16, plus a GEMM's. */
size_t sdc_abft_replay_workspace_size(uint32_t cap_rows, uint32_t N, uint32_t K);

/* The replay of captured rows (the verifier's confirmation): each captured
 * row of A is recomputed against W (the same weights: [N][K] bf16) by the
 * same tensor-core GEMM at the same lane of a 128-row tile (the rest of the
 * tile zero), so a healthy GPU reproduces its output row bit for bit.
 * d_ndiff [cap_rows] uint32: per captured row, how many of its N outputs
 * differ from the captured d_row_C (0 for rows past the count).  d_summary:
 * device uint32 [2], the rows with any difference, and 1 if a bounded wait
 * of the replay's GEMM gave up.  d_row_idx, d_row_A, d_row_C and d_counts
 * (its first word) as sdc_abft_capture wrote them with the same cap_rows. */
sdc_status sdc_abft_replay(const void *d_W, uint32_t N, uint32_t K, uint32_t cap_rows, const uint32_t *d_row_idx,
                           const void *d_row_A, const void *d_row_C, const uint32_t *d_counts, uint32_t *d_ndiff,
                           uint32_t *d_summary, void *d_ws, size_t ws_bytes, sdc_stream_t stream);

/* Workspace bytes of sdc_abft_replay_pairs (0 for caps outside 1..64 or a
 * bad K). */
size_t sdc_abft_replay_pairs_workspace_size(uint32_t K, uint32_t cap_rows, uint32_t cap_cols);

/* The replay of a forward product's captured rows and columns (the row +
 * column configuration): every (row i_r, column j_c) pair's output C[i_r][j_c]
 * is recomputed from the captured row of A and the captured row of W (B's
 * column) alone, by the same tensor-core kernel at the same position in its
 * tile.  d_differs [cap_rows][cap_cols] uint8: 1 unless the replay equals, bit
 * for bit, both captured copies of that output (d_row_C's element j_c and
 * d_col_C's element i_r); 0 past the counts.  d_summary [2]: the pairs that
 * differ, and the replay GEMM's abort flag.  The captured buffers and
 * d_counts as sdc_abft_capture wrote them for this M, N, K with the same caps
 * (1..64 each). */
sdc_status sdc_abft_replay_pairs(uint32_t M, uint32_t N, uint32_t K, uint32_t cap_rows, uint32_t cap_cols,
                                 const uint32_t *d_row_idx, const void *d_row_A, const void *d_row_C,
                                 const uint32_t *d_col_idx, const void *d_col_W, const void *d_col_C,
                                 const uint32_t *d_counts, uint8_t *d_differs, uint32_t *d_summary, void *d_ws,
                                 size_t ws_bytes, sdc_stream_t stream);

/* Workspace bytes of sdc_abft_replay_wgrad (0 for caps outside 1..64). */
size_t sdc_abft_replay_wgrad_workspace_size(uint32_t T, uint32_t cap_rows, uint32_t cap_cols);

/* The replay of a weight gradient's captured rows and columns: every
 * (row n_r, column k_c) pair's output dW[n_r][k_c] is recomputed from the
 * captured dY column and X column alone, by the same tensor-core kernel at
 * the same position in its tile.  d_differs [cap_rows][cap_cols] uint8: 1
 * unless the replay equals, bit for bit, both captured copies of that output
 * (row r's element k_c and column c's element n_r); 0 past the counts.
 * d_summary [2]: the pairs that differ, and the replay GEMM's abort flag.
 * The captured buffers and d_counts as sdc_abft_capture_wgrad wrote them
 * with the same caps (1..64 each). */
sdc_status sdc_abft_replay_wgrad(uint32_t T, uint32_t N, uint32_t K, uint32_t cap_rows, uint32_t cap_cols,
                                 const uint32_t *d_row_idx, const void *d_row_dY, const void *d_row_dW,
                                 const uint32_t *d_col_idx, const void *d_col_X, const void *d_col_dW,
                                 const uint32_t *d_counts, uint8_t *d_differs, uint32_t *d_summary, void *d_ws,
                                 size_t ws_bytes, sdc_stream_t stream);

/* ---------------------------------------------------------------- attention invariant (AEGIS) */

/* Workspace bytes of sdc_attn_dv_check (0 unless D == 128). */
size_t sdc_attn_workspace_size(uint32_t BH, uint32_t L, uint32_t D);

/* The dV half of the attention backward with the invariant 1^T dV = 1^T dO.
 * [AEGIS] method section 3: dV = P^T dO and every row of the softmax P sums
 * to 1, so dV's column sums (taken from the float32 accumulator) equal dO's;
 * P is rebuilt from Q K^T, the softmax and the forward's log-sum-exp, so an
 * upstream error that breaks the row sums breaks the invariant too.
 *
 * Inputs (device): d_Q, d_K, d_dO bf16 [BH][L][D] (BH heads, L tokens, row-
 * major, 16-byte aligned); d_lse float [BH][L], the forward's natural-log
 * log-sum-exp of scale * q_i . k_j over the keys each query attends; scale
 * (> 0, e.g. 1/sqrt(D)); causal (1: query i attends keys j <= i).  D must be
 * 128 and L a positive multiple of 4 (the last 128-token block may be
 * partial: keys and queries past L take no probability).
 * Computes P[i][j] = exp(scale q_i . k_j - lse_i) (bf16 for the product, as a
 * flash-attention backward does), d_dV = P^T dO (bf16 [BH][L][D], float32
 * accumulation on the tensor cores), and per head h and column c:
 *   d_colsum_dv[h][c] = sum_j of dV's float32 accumulator [j][c],
 *   d_colsum_do[h][c] = sum_i dO[i][c],
 *   d_residual = colsum_dv - colsum_do,
 *   d_bound = (2^-8 rho + g (1 + g) rho + own) A (1 + 2^-21) + 2^-100,
 *     A = sum_i |dO[i][c]| (as summed here), g = L 2^-22, rho = 1 + 2^-7
 *     (each probability within 2^-8 of itself: its bf16 rounding and up to
 *     2^-9 for the recomputed scores, exp and the float32 log-sum-exp; each
 *     float32 accumulation step within two ulps); own = 2^-40 + 2^-20 covers
 *     this library's own column sums (float32 pairs of plain 8-row chains),
 *     and the factor 1 + 2^-21 keeps A above the exact sum,
 *   d_flag[h][c] = 1 unless |residual| <= tol_scale * bound (NaN flags),
 * all double/uint8 [BH][D]; d_summary counts the flagged columns; *d_aborted
 * = 1 if a bounded wait gave up (results then invalid).
 * Errors: SDC_ERR_NULL, SDC_ERR_BAD_ARG (shapes, scale, tol_scale, causal),
 * SDC_ERR_BAD_POINTER (alignment), SDC_ERR_WRONG_DEVICE, SDC_ERR_WS_TOO_SMALL.
 * The workspace (256-byte aligned) holds per-block partial sums, -lse log2(e)
 * and the kernels' abort word and work counter. */
sdc_status sdc_attn_dv_check(const void *d_Q, const void *d_K, const void *d_dO, const float *d_lse, uint32_t BH,
                             uint32_t L, uint32_t D, float scale, uint32_t causal, float tol_scale, void *d_dV,
                             double *d_colsum_dv, double *d_colsum_do, double *d_residual, double *d_bound,
                             uint8_t *d_flag, sdc_abft_summary *d_summary, uint32_t *d_aborted, void *d_ws,
                             size_t ws_bytes, sdc_stream_t stream);

/* The same for grouped-query attention: `group` query heads share each K/V
 * head (group = 1 is sdc_attn_dv_check).  BH query heads, a multiple of
 * group; query head h uses K/V head h / group.  d_Q, d_dO bf16 [BH][L][D] and
 * d_lse float [BH][L] as above; d_K bf16 [BH / group][L][D].  dV of a K/V head
 * sums over its group's query heads, as the backward of grouped attention
 * does: d_dV[v] = sum over h in v's group of P_h^T dO_h (bf16 [BH / group][L][D],
 * float32 accumulation over group * L query rows).  Per K/V head v and column c:
 *   d_colsum_dv[v][c] = sum_j of dV's float32 accumulator [j][c],
 *   d_colsum_do[v][c] = sum over h in v's group and i of dO_h[i][c],
 *   d_residual, d_bound, d_flag as above with g = group L 2^-22 and the sum of
 *     |dO| over the group, all [BH / group][D].
 * Errors as above; SDC_ERR_BAD_ARG also when group is 0 or does not divide BH,
 * or when group * ceil(L / 128) (the steps of one work item) exceeds 2^19.
 * The workspace is sdc_attn_workspace_size(BH, L, D). */
sdc_status sdc_attn_dv_check_grouped(const void *d_Q, const void *d_K, const void *d_dO, const float *d_lse,
                                     uint32_t BH, uint32_t group, uint32_t L, uint32_t D, float scale, uint32_t causal,
                                     float tol_scale, void *d_dV, double *d_colsum_dv, double *d_colsum_do,
                                     double *d_residual, double *d_bound, uint8_t *d_flag, sdc_abft_summary *d_summary,
                                     uint32_t *d_aborted, void *d_ws, size_t ws_bytes, sdc_stream_t stream);

/* ---------------------------------------------------------------- self-test */

/* Self-test of the bounded barrier wait with which the TMA / tensor-core
 * kernels (sdc_abft_gemm, sdc_attn_dv_check) turn a stall into an abort flag
 * instead of a hang.  No page counterpart: it tests this library's own
 * failure handling.  One thread waits up to `polls` polls (1 .. 2^24) on a
 * shared-memory barrier phase that nothing completes, then completes it itself
 * and waits again.  *d_status (device uint32) = bit 0: the first wait gave up;
 * bit 1: the second wait succeeded; 3 is the correct outcome.  The kernel ends
 * in every case. */
sdc_status sdc_selftest_bounded_wait(uint32_t polls, uint32_t *d_status, sdc_stream_t stream);

/* ---------------------------------------------------------------- ring replay audit */

/* Counts written by sdc_ring_audit. */
typedef struct {
    uint32_t n_pairs;      /* mismatched (target, replayer) pairs */
    uint32_t n_culprits;   /* ranks in two or more mismatched pairs */
    uint32_t n_ambiguous;  /* mismatched pairs that touch no culprit */
    uint32_t reserved;
} sdc_ring_summary;

/* The ring replay audit's comparison and localization, on device.
 * [AWS] "Check 2: Ring replay, before the optimizer step": on an audit step
 * rank r replays the micro-batch of its target t = (r + offset) mod n; each
 * rank's row holds [its own result, its replay of its target], and the pair
 * (t, r) mismatches when t's own result differs from r's replay in any word.
 * A rank in two or more mismatched pairs is a culprit; a mismatched pair that
 * touches no culprit is ambiguous and needs the page's confirmation replay.
 * d_table: device uint64[n][2][L] (row 0 = own result, row 1 = replay of the
 * target), e.g. loss bits followed by per-parameter (S, W) gradient
 * fingerprints; offset is taken mod n.  Outputs (device): d_mismatch uint8[n]
 * and d_ambiguous uint8[n], indexed by the replayer r of pair (t, r);
 * d_hits uint32[n], mismatched pairs containing each rank (a pair (r, r)
 * counts r twice, as a count over pair members does); d_culprit uint8[n];
 * d_summary the counts.  n == 0 writes a zero summary. */
sdc_status sdc_ring_audit(const uint64_t *d_table, uint32_t n, uint32_t L, uint32_t offset, uint8_t *d_mismatch,
                          uint32_t *d_hits, uint8_t *d_culprit, uint8_t *d_ambiguous, sdc_ring_summary *d_summary,
                          sdc_stream_t stream);

/* ---------------------------------------------------------------- gradients */

/* Non-finite scan and squared norm of each replica's gradient tensors.
 * [AWS] "Check 1: NaN/Inf gradients, before and after the all-reduce": each
 * rank's local gradient is checked for NaN/Inf before the all-reduce.  Here
 * replica r of the plan is one local gradient made of T tensors; every
 * descriptor must have a float dtype.  d_stats: device sdc_grad_stats[R].
 * Counts are exact; sumsq_finite is within 2e-11 relative of the exact sum
 * and identical on every run (fixed reduction order). */
sdc_status sdc_grad_scan(const sdc_plan *plan, sdc_grad_stats *d_stats, void *d_ws, size_t ws_bytes,
                         sdc_stream_t stream);

/* Workspace bytes for sdc_grad_average_scan with these sizes (0 when n_bufs or
 * dtype is invalid). */
size_t sdc_grad_average_scan_workspace_size(uint64_t numel, uint32_t n_bufs, uint32_t dtype);

/* One fused pass: scan n_bufs local gradient buffers, write their average,
 * and scan the average -- the one-device stand-in for the page's check 1
 * around the all-reduce ([AWS] "Step 1: Detect": the all-reduce averages the
 * replicas' gradients; "Check 1": check each local gradient before it and the
 * reduced gradient after it, whose norm clip_grad_norm_ already computes).
 * bufs: HOST array of n_bufs (1..8) device pointers, each to numel elements
 * of `dtype` (F32, BF16 or F16); d_avg: device output of numel elements of
 * the same dtype (must not overlap the inputs).  Average, per element: the
 * float32 sum of the inputs in buffer order, divided by n_bufs in float32
 * (correctly rounded), rounded to dtype ties-to-even; every NaN result is the
 * canonical quiet NaN (0x7FC0 bf16, 0x7E00 f16, 0x7FC00000 f32).
 * d_pre: device sdc_grad_stats[n_bufs] of the inputs; d_post: device
 * sdc_grad_stats of the average (its `norm` is the global L2 norm and
 * its nonfinite_fp32 is the reduced-gradient alarm).  Pointers aligned to 16
 * bytes take the vector path; others take a slower element path. */
sdc_status sdc_grad_average_scan(const void *const *bufs, uint32_t n_bufs, void *d_avg, uint64_t numel,
                                 uint32_t dtype, sdc_grad_stats *d_pre, sdc_grad_stats *d_post,
                                 void *d_ws, size_t ws_bytes, sdc_stream_t stream);

/* Size of the library's fixed device scratch used by
 * sdc_grad_average_scan_noalloc (16 MiB on every GPU that loads libsdc). */
#define SDC_NOALLOC_SCRATCH_BYTES (16u << 20)

/* sdc_grad_average_scan without a workspace argument and without any device
 * allocation.  (The pages have no counterpart: this is an interface choice of
 * this library, not a step of the method.)  It is for callers that cannot
 * call cudaMalloc or take memory from a caching allocator -- code running in
 * a host callback or inside an allocator's hooks, a tool injected into a job
 * whose device memory is owned and capped by another framework -- but still
 * want the non-finite scan and average of their gradient buffers.
 * Arguments, results and errors are those of sdc_grad_average_scan.  The
 * scratch is a fixed __device__ array of SDC_NOALLOC_SCRATCH_BYTES inside the
 * library: sizes whose sdc_grad_average_scan_workspace_size(numel, n_bufs,
 * dtype) exceeds it are rejected with SDC_ERR_BAD_ARG and a message giving
 * the limit (with 4 bf16 buffers that is about 1.14e9 elements).  The first
 * call on each device looks up the array's device address (a
 * cudaGetSymbolAddress with that device current) and caches it with the ID
 * of the current context; a call that finds another context current (after
 * cudaDeviceReset, for example, which loads the library's device code anew)
 * looks it up again.  Make the first call on a device, and the first after
 * such a reset, before any stream capture.  All calls share the one array and
 * it keeps the last call's contents (nothing in it needs to start at zero):
 * calls whose GPU work overlaps -- on different streams, or from several host
 * threads -- race on it and must be ordered by the caller. */
sdc_status sdc_grad_average_scan_noalloc(const void *const *bufs, uint32_t n_bufs, void *d_avg, uint64_t numel,
                                         uint32_t dtype, sdc_grad_stats *d_pre, sdc_grad_stats *d_post,
                                         sdc_stream_t stream);

/* ---------------------------------------------------------------- errors */

/* Static name of a status code. */
const char *sdc_status_string(sdc_status status);

/* Detail of the calling thread's most recent failed call ("" if none). */
const char *sdc_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SDC_H */
