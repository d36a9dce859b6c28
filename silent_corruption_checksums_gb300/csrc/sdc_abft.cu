// sdc_abft.cu -- a bf16 GEMM on the 5th-generation tensor cores whose
// epilogue checksums every output row from the float32 accumulator.
//
// "Safeguarding LLM Training at Scale: Online SDC Detection and Insights from
// 35 Million GPU Hours" (review page), method section 2: the classic matrix
// checksum compares (AB)1 with A(B1); AEGIS forms the checksum inside the GEMM
// kernel from the float32 accumulator, before the bfloat16 output is rounded,
// so the check's noise is far below that of a checksum of the bf16 output.
//
// Here C[M, N] = A[M, K] . W[N, K]^T (the forward product of a linear layer,
// both operands K-contiguous), bf16 in, fp32 accumulate, bf16 out.  Row i's
// checksum sum_j acc[i, j] is summed in float64 from the TMEM accumulator by
// the epilogue (one partial per 256-column tile, reduced in a fixed order);
// the reference A (W^T 1) comes from a column-sum and a float64 row dot
// product.  A row whose residual exceeds tol_scale times a bound on the
// rounding error is flagged.  With mag = sum_k |A[i, k]| * sum_j |W[j, k]| and
// g = K * 2^-22 the bound is
//   g (1 + g) mag  +  (N + K + 64) 2^-52 mag  +  2 K N 2^-126:
// the first term lets each of the K float32 accumulation steps of an output
// lose up to two units in the last place of its partial sum's magnitude (so it
// holds for round-to-nearest and for truncating adders alike), the second
// covers the float64 sums of the check, the third subnormals flushed to zero.
// A clean product is thus not flagged with tol_scale >= 1; AEGIS adapts its
// threshold online and the page gives no constants, so the residual is
// returned too.
//
// Kernel layout (one 128 x 256 output tile per CTA, 6 warps):
//   warp 0 lane 0: TMA producer -- per 64-wide K block, 8 + 8 tiled bulk
//     tensor copies (boxes of 8 K-elements x 128 or 256 rows) lay A and W out
//     in the tensor core's core-matrix order (no swizzle) in one of kStages
//     shared-memory stages, completing on the stage's `full` mbarrier;
//   warp 1 lane 0: MMA issuer -- 4 tcgen05.mma (M=128, N=256, K=16) per stage
//     into a 256-column TMEM accumulator, tcgen05.commit releases the stage
//     (`empty`) and, after the last block, signals the epilogue (`acc`);
//   warps 2..5: epilogue -- each thread owns one row (TMEM lane), reads its
//     256 fp32 accumulators with tcgen05.ld, sums them in float64, rounds to
//     bf16 and stores.
// Every wait is bounded; a wait that gives up sets the call's abort flag.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "sdc_internal.cuh"

namespace sdc {

namespace {

constexpr uint32_t kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kStageA = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kStageW = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kGemmThreads = 192;
constexpr uint32_t kGemmSmem = kStages * (kStageA + kStageW) + 2048;  // + alignment slack, barriers, TMEM slot
constexpr uint32_t kMaxK = 1u << 20;

// Shared-memory matrix descriptor, no swizzle: start address, the byte stride
// between core matrices along K (lbo) and along M/N (sbo), version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N and M.
__host__ __device__ constexpr uint32_t umma_idesc(uint32_t m, uint32_t n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                            uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(map), "r"(c0), "r"(c1), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            tmem),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    abft_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapW,
                     __nv_bfloat16 *__restrict__ C, uint32_t M, uint32_t N, uint32_t K, double *__restrict__ rowsum_part,
                     int *__restrict__ err) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    const uint32_t tile_n = blockIdx.x, tile_m = blockIdx.y;
    const uint32_t base = smem_addr(smem), pad = ((base + 1023u) & ~1023u) - base;
    const uint32_t sA = base + pad;                 // kStages x 16 KiB, 1 KiB aligned
    const uint32_t sW = sA + kStages * kStageA;     // kStages x 32 KiB
    const uint32_t bars = sW + kStages * kStageW;   // full[S], empty[S], acc
    uint32_t *tmem_slot = (uint32_t *)(smem + pad + kStages * (kStageA + kStageW) + 8 * (2 * kStages + 1));
    const uint32_t full = bars, empty = bars + 8 * kStages, acc = bars + 16 * kStages;
    const uint32_t nkb = K / kBK;

    if (warp == 1) {  // the MMA warp owns the accumulator's TMEM columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        mbar_init(acc, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------ TMA producer
            uint32_t issued = 0;
            for (uint32_t kb = 0; kb < nkb && ok; ++kb) {
                const uint32_t s = kb % kStages;
                if (kb >= (uint32_t)kStages && !mbar_wait(empty + 8 * s, ((kb / kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                issued = kb + 1;
                mbar_arrive_expect_tx(full + 8 * s, kStageA + kStageW);
                for (uint32_t j = 0; j < kBK / 8; ++j) {
                    const int32_t k0 = (int32_t)(kb * kBK + 8 * j);
                    tma_load_2d(sA + s * kStageA + j * (kBM * 16), &mapA, k0, (int32_t)(tile_m * kBM), full + 8 * s);
                    tma_load_2d(sW + s * kStageW + j * (kBN * 16), &mapW, k0, (int32_t)(tile_n * kBN), full + 8 * s);
                }
            }
            // Let no copy land in shared memory after the block has left: wait
            // (bounded) for the last stages issued to complete.
            const uint32_t first = issued > (uint32_t)kStages ? issued - kStages : 0;
            for (uint32_t kb = first; kb < issued; ++kb)
                if (!mbar_wait(full + 8 * (kb % kStages), (kb / kStages) & 1)) ok = false;
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ------------------------------------------ MMA issuer
            constexpr uint32_t idesc = umma_idesc(kBM, kBN);
            for (uint32_t kb = 0; kb < nkb && ok; ++kb) {
                const uint32_t s = kb % kStages;
                if (!mbar_wait(full + 8 * s, (kb / kStages) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (uint32_t ks = 0; ks < kBK / 16; ++ks) {
                    // one K16 step = two core-matrix columns: 2 x (rows x 16 B)
                    const uint64_t da = umma_desc(sA + s * kStageA + ks * 2 * (kBM * 16), kBM * 16, 128);
                    const uint64_t dw = umma_desc(sW + s * kStageW + ks * 2 * (kBN * 16), kBN * 16, 128);
                    tc_mma(tmem, da, dw, idesc, (kb | ks) != 0 ? 1u : 0u);
                }
                tc_commit(empty + 8 * s);  // the stage is free once these MMAs have read it
            }
            // Always signal: the barrier then tracks every MMA this thread
            // issued, and the TMEM owner waits on it before freeing.
            tc_commit(acc);
            if (!ok) atomicOr(err, 1);
        }
    } else {  // ------------------------------------------------------- epilogue
        const uint32_t quarter = warp & 3u;  // TMEM lanes this warp may read
        const uint32_t row = tile_m * kBM + quarter * 32 + lane;
        const bool got = mbar_wait(acc, 0);
        if (__any_sync(0xffffffffu, !got)) {
            if (lane == 0) atomicOr(err, 1);
        } else {
            tc_fence_after();
            double rs = 0.0;
            __nv_bfloat16 *crow = C + (uint64_t)row * N + tile_n * kBN;
            for (uint32_t c = 0; c < kBN; c += 32) {
                uint32_t r[32];
                tc_ld32(tmem + ((quarter * 32) << 16) + c, r);
                uint32_t packed[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float lo = __uint_as_float(r[j]), hi = __uint_as_float(r[j + 1]);
                    rs = __dadd_rn(rs, (double)lo);
                    rs = __dadd_rn(rs, (double)hi);
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed[j / 2]) : "f"(hi), "f"(lo));
                }
                uint4 *dst = (uint4 *)(crow + c);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
            }
            rowsum_part[(uint64_t)tile_n * M + row] = rs;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && !mbar_wait(acc, 0)) atomicOr(err, 1);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBN) : "memory");
    }
}

// w1[k] = sum_j W[j, k] and wabs[k] = sum_j |W[j, k]| in float64, one thread per k
// column, rows in order.
__global__ void abft_colsum_kernel(const __nv_bfloat16 *__restrict__ W, uint32_t N, uint32_t K, double *__restrict__ w1,
                                   double *__restrict__ wabs) {
    const uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    double s = 0.0, a = 0.0;
    for (uint32_t j = 0; j < N; ++j) {
        const double x = (double)__bfloat162float(W[(uint64_t)j * K + k]);
        s = __dadd_rn(s, x);
        a = __dadd_rn(a, fabs(x));
    }
    w1[k] = s;
    wabs[k] = a;
}

// Row checksums: the tile partials of each row summed in tile order.
__global__ void abft_rowsum_kernel(const double *__restrict__ rowsum_part, uint32_t M, uint32_t n_tiles,
                                   double *__restrict__ rowsum) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M) return;
    double cs = 0.0;
    for (uint32_t t = 0; t < n_tiles; ++t) cs = __dadd_rn(cs, rowsum_part[(uint64_t)t * M + i]);
    rowsum[i] = cs;
}

// Per row: the reference A (W^T 1), the rounding bound, the residual against
// the accumulator checksum, and the flag.  One warp per row.
__global__ void abft_check_kernel(const __nv_bfloat16 *__restrict__ A, uint32_t M, uint32_t N, uint32_t K,
                                  const double *__restrict__ rowsum, const double *__restrict__ w1,
                                  const double *__restrict__ wabs, float tol_scale, double *__restrict__ residual,
                                  double *__restrict__ bound, uint8_t *__restrict__ flag,
                                  sdc_abft_summary *__restrict__ summary) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= M) return;
    const uint32_t i = (uint32_t)warp;
    double ref = 0.0, mag = 0.0;
    for (uint32_t k = lane; k < K; k += 32) {
        const double a = (double)__bfloat162float(A[(uint64_t)i * K + k]);
        ref = fma(a, w1[k], ref);
        mag = fma(fabs(a), wabs[k], mag);
    }
    ref = warp_sum_f64(ref);
    mag = warp_sum_f64(mag);
    if (lane == 0) {
        const double cs = rowsum[i];
        const double g = (double)K * 0x1p-22;
        const double b = (g * (1.0 + g) + (double)(N + K + 64) * 0x1p-52) * mag + 2.0 * (double)K * (double)N * 0x1p-126;
        const double d = cs - ref;
        residual[i] = d;
        bound[i] = b;
        const uint8_t f = fabs(d) <= (double)tol_scale * b ? 0 : 1;  // NaN flags
        flag[i] = f;
        if (f) atomicAdd(&summary->n_flagged, 1u);
    }
}

__global__ void abft_finish_kernel(const int *__restrict__ err, uint32_t *__restrict__ aborted) {
    *aborted = *err != 0 ? 1u : 0u;
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled encode_fn() {
    static std::once_flag once;
    static PFN_encodeTiled fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_encodeTiled)p;
    });
    return fn;
}

// 2-D map over a [rows, K] bf16 matrix: boxes of 8 K-elements (16 bytes) x box_rows.
sdc_status make_map(CUtensorMap *map, const void *ptr, uint32_t rows, uint32_t K, uint32_t box_rows) {
    PFN_encodeTiled fn = encode_fn();
    if (!fn) return fail(SDC_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {8, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SDC_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return SDC_OK;
}

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

}  // namespace sdc

using namespace sdc;

extern "C" {

size_t sdc_abft_workspace_size(uint32_t M, uint32_t N, uint32_t K) {
    const size_t tiles_n = N / kBN;
    return round_up256(tiles_n * M * sizeof(double)) + 2 * round_up256((size_t)K * sizeof(double)) + 256;
}

static sdc_status abft_args(const void *d_A, const void *d_W, uint32_t M, uint32_t N, uint32_t K, void *d_ws,
                            size_t ws_bytes, int *dev) {
    if (!d_A || !d_W) return fail(SDC_ERR_NULL, "NULL operand");
    if (M == 0 || N == 0 || K == 0 || M % kBM || N % kBN || K % kBK || K > kMaxK)
        return fail(SDC_ERR_BAD_ARG, "M must be a multiple of 128, N of 256 and K of 64 (all > 0, K <= 2^20)");
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_device_range(d_A, (uint64_t)M * K * 2, *dev, "d_A");
    if (st == SDC_OK) st = check_device_range(d_W, (uint64_t)N * K * 2, *dev, "d_W");
    if (st != SDC_OK) return st;
    if (((uint64_t)d_A | (uint64_t)d_W) & 15u) return fail(SDC_ERR_BAD_POINTER, "A and W must be 16-byte aligned");
    if (!d_ws || ws_bytes < sdc_abft_workspace_size(M, N, K))
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    return SDC_OK;
}

sdc_status sdc_abft_gemm(const void *d_A, const void *d_W, void *d_C, uint32_t M, uint32_t N, uint32_t K,
                         double *d_rowsum, uint32_t *d_aborted, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    int dev = -1;
    sdc_status st = abft_args(d_A, d_W, M, N, K, d_ws, ws_bytes, &dev);
    if (st != SDC_OK) return st;
    if (!d_C || !d_rowsum || !d_aborted) return fail(SDC_ERR_NULL, "NULL output");
    st = check_device_range(d_C, (uint64_t)M * N * 2, dev, "d_C");
    if (st != SDC_OK) return st;
    if ((uint64_t)d_C & 15u) return fail(SDC_ERR_BAD_POINTER, "C must be 16-byte aligned");
    CUtensorMap mapA, mapW;
    st = make_map(&mapA, d_A, M, K, kBM);
    if (st == SDC_OK) st = make_map(&mapW, d_W, N, K, kBN);
    if (st != SDC_OK) return st;
    const uint32_t tiles_n = N / kBN;
    double *part = (double *)d_ws;
    int *err = (int *)((char *)d_ws + round_up256((size_t)tiles_n * M * sizeof(double)) +
                       2 * round_up256((size_t)K * sizeof(double)));
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(abft_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm setup");
    abft_gemm_kernel<<<dim3(tiles_n, M / kBM), kGemmThreads, kGemmSmem, s>>>(mapA, mapW, (__nv_bfloat16 *)d_C, M, N, K,
                                                                           part, err);
    abft_rowsum_kernel<<<(M + 255) / 256, 256, 0, s>>>(part, M, tiles_n, d_rowsum);
    abft_finish_kernel<<<1, 1, 0, s>>>(err, d_aborted);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_gemm launch");
}

sdc_status sdc_abft_verify(const void *d_A, const void *d_W, uint32_t M, uint32_t N, uint32_t K, const double *d_rowsum,
                           float tol_scale, double *d_residual, double *d_bound, uint8_t *d_flag,
                           sdc_abft_summary *d_summary, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    int dev = -1;
    sdc_status st = abft_args(d_A, d_W, M, N, K, d_ws, ws_bytes, &dev);
    if (st != SDC_OK) return st;
    if (!d_rowsum || !d_residual || !d_bound || !d_flag || !d_summary) return fail(SDC_ERR_NULL, "NULL output");
    if (!(tol_scale > 0.0f)) return fail(SDC_ERR_BAD_ARG, "tol_scale must be positive");
    const uint32_t tiles_n = N / kBN;
    double *w1 = (double *)((char *)d_ws + round_up256((size_t)tiles_n * M * sizeof(double)));
    double *wabs = (double *)((char *)w1 + round_up256((size_t)K * sizeof(double)));
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(d_summary, 0, sizeof(sdc_abft_summary), s);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_verify setup");
    abft_colsum_kernel<<<(K + 255) / 256, 256, 0, s>>>((const __nv_bfloat16 *)d_W, N, K, w1, wabs);
    abft_check_kernel<<<(unsigned)(((uint64_t)M * 32 + 255) / 256), 256, 0, s>>>(
        (const __nv_bfloat16 *)d_A, M, N, K, d_rowsum, w1, wabs, tol_scale, d_residual, d_bound, d_flag, d_summary);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_verify launch");
}

}  // extern "C"
