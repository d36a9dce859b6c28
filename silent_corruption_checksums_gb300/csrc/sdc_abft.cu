// sdc_abft.cu -- a bf16 GEMM on the 5th-generation tensor cores whose
// epilogue checksums every output row from the float32 accumulator, and the
// check of those checksums.
//
// "Safeguarding LLM Training at Scale: Online SDC Detection and Insights from
// 35 Million GPU Hours" (review page), method section 2: the classic matrix
// checksum compares (AB)1 with A(B1); AEGIS forms the checksum inside the GEMM
// kernel from the float32 accumulator, before the bfloat16 output is rounded,
// so the check's noise is far below that of a checksum of the bf16 output.
//
// Here C[M, N] = A[M, K] . W[N, K]^T (the forward product of a linear layer,
// both operands K-contiguous), bf16 in, fp32 accumulate, bf16 out.  Row i's
// checksum sum_j acc[i, j] is summed by the epilogue from the TMEM accumulator
// (one partial per 256-column tile, reduced in a fixed order); the reference
// A (W^T 1) comes from a column-sum and a row dot product.  A row whose
// residual exceeds tol_scale times a bound on the rounding error is flagged.
// With mag = sum_k |A[i, k]| * sum_j |W[j, k]| and g = K * 2^-22 the bound is
//   g (1 + g) mag  +  (N + K + 64) 2^-44 mag  +  2 K N 2^-126:
// the first term lets each of the K float32 accumulation steps of an output
// lose up to two units in the last place of its partial sum's magnitude (so it
// holds for round-to-nearest and for truncating adders alike), the second
// covers the sums of the check (float32 pairs, ~2^-48 per step), the third
// subnormals flushed to zero.  A clean product is thus not flagged with
// tol_scale >= 1; AEGIS adapts its threshold online and the page gives no
// constants, so the residual is returned too.
//
// The check's sums run on float32 pairs (an error-free TwoSum, products split
// with a fused multiply-add) rather than float64: this GPU's float64 rate is a
// small fraction of its float32 rate, and a pair carries ~48 bits, far more
// than the check needs.
//
// GEMM kernel (persistent, one CTA per SM, 6 warps, 128 x 256 output tiles):
//   warp 0 lane 0: TMA producer -- per 64-wide K block one tiled bulk tensor
//     copy of A (64 x 128) and one of W (64 x 256) into a kStages-deep ring of
//     shared-memory stages, 128-byte swizzled (the tensor core's canonical
//     K-major layout), completing on the stage's `full` mbarrier;
//   warp 1 lane 0: MMA issuer -- 4 tcgen05.mma (M=128, N=256, K=16) per stage
//     into one of two 256-column TMEM accumulators; tcgen05.commit frees the
//     stage (`empty`) and, after a tile's last block, hands the accumulator to
//     the epilogue (`tfull`);
//   warps 2..5: epilogue -- each thread owns one row (TMEM lane), reads its
//     256 fp32 accumulators with tcgen05.ld, sums them (float32 pair), rounds
//     to bf16 and stores, then frees the accumulator (`tempty`), so the
//     epilogue of one tile overlaps the main loop of the next.
// Every wait is bounded; a wait that gives up sets the call's abort flag, and
// the block still waits (bounded) for its copies and MMAs in flight and frees
// its TMEM before it exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "sdc_internal.cuh"
#include "sdc_tc.cuh"

namespace sdc {

int sm_count(int device);

namespace {

constexpr uint32_t kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kStageA = kBM * kBK * 2;  // 16 KiB
constexpr uint32_t kStageW = kBN * kBK * 2;  // 32 KiB
constexpr uint32_t kAccCols = 256;           // one accumulator; two are allocated
constexpr uint32_t kMnBlock = kBK * 128;      // 8 KiB: kBK contraction rows of 64 bf16 (MN-major operands)
constexpr uint32_t kGemmThreads = 192;
constexpr uint32_t kRefThreads = 128;  // the fused check's reference warps (one row of the tile each)
constexpr uint32_t kNumBars = 2 * kStages + 5;  // full[S], empty[S], tfull[2], tempty[2], done
constexpr uint32_t kGemmSmem = kStages * (kStageA + kStageW) + 1024 + 8 * kNumBars + 16;
// with the reference warps: a selected K block's column sums (64 x {h, m}, 512 bytes) after the barriers
// and the TMEM slot, at a 16-byte boundary (128-bit loads)
constexpr uint32_t kRefSumsOff = (kStages * (kStageA + kStageW) + 8 * kNumBars + 16 + 15) / 16 * 16;
constexpr uint32_t kGemmSmemRef = 1024 + kRefSumsOff + kBK * 8;
static_assert(kRefSumsOff % 16 == 0 && kGemmSmemRef <= 232448, "reference sums: alignment and shared memory");
constexpr uint32_t kColTileFloats = 32 * 33;  // one epilogue warp's column-sum tile (row pitch 33)
// with columns: the four epilogue warps' column tiles, then their per-tile column partials [4][kBN]
// (merged in the CTA, so one partial row per tile row reaches global memory)
constexpr uint32_t kGemmSmemCols = kGemmSmem + 4 * kColTileFloats * 4 + 4 * kBN * 8;
static_assert(kGemmSmemCols <= 232448, "shared memory per block");
constexpr uint32_t kMaxK = 1u << 20;
constexpr uint32_t kMaxSlabs = 64;

// Converts 32 accumulators to bf16 (round to nearest even), stores them at
// dst (64 bytes, 16-byte aligned) and adds them to the row's pair sum.
// valid: how many of the chunk's 32 columns lie inside C (a multiple of 8; 0 for a row past M)
__device__ __forceinline__ void epilogue_chunk(const uint32_t (&r)[32], __nv_bfloat16 *dst, float &s, float &c,
                                               uint32_t valid) {
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float lo = __uint_as_float(r[j]), hi = __uint_as_float(r[j + 1]);
        pair_add(s, c, lo);
        pair_add(s, c, hi);
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed[j / 2]) : "f"(hi), "f"(lo));
    }
    uint4 *d = (uint4 *)dst;
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
        if (8 * q < valid) d[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
}

// Tile t of the schedule -> (tile row, tile column).  Tiles go in bands of
// band_m tile rows; inside a band the row index runs fastest, so the CTAs in
// flight share a few W tiles while the band's rows of A (sized on the host to
// stay resident in L2) are reused by every column of the band.
__device__ __forceinline__ void tile_coords(uint32_t t, uint32_t tiles_m, uint32_t tiles_n, uint32_t band_m,
                                            uint32_t &tm, uint32_t &tn) {
    const uint32_t band_tiles = band_m * tiles_n;
    const uint32_t band = t / band_tiles, r = t - band * band_tiles;
    const uint32_t m0 = band * band_m;
    const uint32_t bm = tiles_m - m0 < band_m ? tiles_m - m0 : band_m;
    tm = m0 + r % bm;
    tn = r / bm;
}

// The sum over the warp's 32 rows (lanes) of 32 accumulator columns: the warp
// writes its 32 x 32 block into its own padded shared-memory tile (row pitch
// 33 words: conflict-free both ways), then lane k sums column k in row order as
// a float32 pair.  Each column is summed by one lane in a fixed order, so the
// result is reproducible.
__device__ __forceinline__ double warp_column_sum(const uint32_t (&r)[32], uint32_t lane, float *tile) {
#pragma unroll
    for (int k = 0; k < 32; ++k) tile[lane * 33 + k] = __uint_as_float(r[k]);
    __syncwarp();
    float s = 0.0f, c = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) pair_add(s, c, tile[i * 33 + lane]);
    __syncwarp();  // the tile is reused by the next chunk
    return (double)s + (double)c;
}

// Barrier over `count` threads that also ORs `pred` across them: every warp of the group takes the
// same branch afterwards.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// kMN: both operands MN-major (the weight-gradient form, below); otherwise both K-major.
// kRef (K-major only): four more warps form the check's reference of each row, A[i, :] (W^T 1), on
// the CUDA cores beside the product, against W's column sums wsums[k] = {h, m}.  Tile (m, n) takes
// the K blocks kb with kb mod tiles_n = n, so every K block of every tile row is taken once and the
// work spreads over all tiles; ref[n][i] = {s, c, mh, ml} is the tile's partial (the reference and
// the magnitude, each a float32 pair).  They read A's rows from global memory (Ag), where the
// banded schedule keeps them in L2 for the product's copies, and touch none of its barriers.
template <bool kCols, bool kMN, bool kRef>
__global__ void __launch_bounds__(kRef ? kGemmThreads + kRefThreads : kGemmThreads, 1)
    abft_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapW,
                     __nv_bfloat16 *__restrict__ C, uint32_t M, uint32_t N, uint32_t K, uint32_t band_m,
                     double *__restrict__ rowsum_part, double *__restrict__ colsum_part, int *__restrict__ err,
                     const float2 *__restrict__ wsums, float4 *__restrict__ ref, const __nv_bfloat16 *__restrict__ Ag,
                     uint32_t *__restrict__ zero, uint32_t n_zero) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    // zero[0 .. n_zero): counts that only a later launch on the stream adds to (the fused check's summary)
    if (blockIdx.x == 0 && tid < n_zero) zero[tid] = 0u;
    const uint32_t base = smem_addr(smem), pad = ((base + 1023u) & ~1023u) - base;
    const uint32_t sA = base + pad;                // kStages x 16 KiB, 1 KiB aligned (the swizzle atom)
    const uint32_t sW = sA + kStages * kStageA;    // kStages x 32 KiB
    const uint32_t bars = sW + kStages * kStageW;  // full[S], empty[S], tfull[2], tempty[2], done
    const uint32_t full = bars, empty = bars + 8 * kStages, tfull = bars + 16 * kStages, tempty = tfull + 16,
                   done = tempty + 16;
    uint32_t *tmem_slot = (uint32_t *)(smem + pad + kStages * (kStageA + kStageW) + 8 * kNumBars);
    // tiles cover C with zeros past M, N and K: the copies fill the rows and columns outside A and
    // W with zeros, which add nothing to a product or a checksum; the epilogue stores only inside C
    const uint32_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN, nkb = (K + kBK - 1) / kBK;
    const uint32_t n_units = tiles_m * tiles_n, unit0 = blockIdx.x, ustep = gridDim.x;
    auto coords = [&](uint32_t u, uint32_t &tm, uint32_t &tn) { tile_coords(u, tiles_m, tiles_n, band_m, tm, tn); };

    if (warp == 1) {  // the MMA warp owns both accumulators' TMEM columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(2 * kAccCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + 8 * b, 1);
            mbar_init(tempty + 8 * b, 4);  // one arrival per epilogue warp
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------ TMA producer
            uint32_t it = 0;
            for (uint32_t u = unit0; u < n_units && ok; u += ustep) {
                uint32_t tm, tn;
                coords(u, tm, tn);
                const int32_t row_a = (int32_t)(tm * kBM), row_w = (int32_t)(tn * kBN);
                for (uint32_t kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    if (it >= (uint32_t)kStages && !mbar_wait(empty + 8 * s, ((it / kStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + 8 * s, kStageA + kStageW);
                    if constexpr (kMN) {  // 64 x 64 boxes: kBK contraction rows of 64 output rows or columns
#pragma unroll
                        for (uint32_t j = 0; j < kBM / 64; ++j)
                            tma_load_2d(sA + s * kStageA + j * kMnBlock, &mapA, row_a + (int32_t)(64 * j),
                                        (int32_t)(kb * kBK), full + 8 * s);
#pragma unroll
                        for (uint32_t j = 0; j < kBN / 64; ++j)
                            tma_load_2d(sW + s * kStageW + j * kMnBlock, &mapW, row_w + (int32_t)(64 * j),
                                        (int32_t)(kb * kBK), full + 8 * s);
                    } else {
                        tma_load_2d(sA + s * kStageA, &mapA, (int32_t)(kb * kBK), row_a, full + 8 * s);
                        tma_load_2d(sW + s * kStageW, &mapW, (int32_t)(kb * kBK), row_w, full + 8 * s);
                    }
                }
            }
            // Let no copy land in shared memory after the block has left: wait
            // (bounded) for the last stages issued to complete.
            const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
            for (uint32_t j = first; j < it; ++j)
                if (!mbar_wait(full + 8 * (j % kStages), (j / kStages) & 1)) ok = false;
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ------------------------------------------ MMA issuer
            constexpr uint32_t idesc = kMN ? umma_idesc_mn(kBM, kBN) : umma_idesc(kBM, kBN);
            uint32_t it = 0, lt = 0;
            for (uint32_t u = unit0; u < n_units && ok; u += ustep, ++lt) {
                const uint32_t b = lt & 1u;
                if (lt >= 2 && !mbar_wait(tempty + 8 * b, ((lt >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + b * kAccCols;
                for (uint32_t kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % kStages;
                    if (!mbar_wait(full + 8 * s, (it / kStages) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (uint32_t ks = 0; ks < kBK / 16; ++ks) {
                        // K-major: a K16 step is 32 bytes inside each 128-byte row; MN-major: 16 rows of
                        // 128 bytes (2 KiB), the 64-wide blocks kMnBlock apart
                        const uint64_t da = kMN ? umma_desc_sw128_mn(sA + s * kStageA + ks * 2048, kMnBlock)
                                                : umma_desc_sw128(sA + s * kStageA + ks * 32);
                        const uint64_t db = kMN ? umma_desc_sw128_mn(sW + s * kStageW + ks * 2048, kMnBlock)
                                                : umma_desc_sw128(sW + s * kStageW + ks * 32);
                        tc_mma(d, da, db, idesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty + 8 * s);  // the stage is free once these MMAs have read it
                }
                if (ok) tc_commit(tfull + 8 * b);
            }
            // Tracks every MMA this thread issued; the TMEM owner waits on it before freeing.
            tc_commit(done);
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp < kGemmThreads / 32) {  // ------------------------ epilogue
        const uint32_t quarter = warp & 3u;  // the TMEM lanes this warp may read
        const uint32_t lane_base = (quarter * 32) << 16;
        float *coltile = (float *)(smem + pad + kStages * (kStageA + kStageW) + 8 * kNumBars + 16) + quarter * kColTileFloats;
        double *cq = (double *)(smem + pad + kStages * (kStageA + kStageW) + 8 * kNumBars + 16 + 4 * kColTileFloats * 4);
        const uint32_t et = tid - 64;  // thread index within the epilogue (warps 2-5)
        uint32_t lt = 0;
        for (uint32_t u = unit0; u < n_units; u += ustep, ++lt) {
            const uint32_t b = lt & 1u;
            const bool got = mbar_wait(tfull + 8 * b, (lt >> 1) & 1);
            // with columns the four warps meet at barriers below: they leave together
            if (kCols ? bar_any(1, 128, !got) : __any_sync(0xffffffffu, !got)) {
                if (lane == 0) atomicOr(err, 1);
                break;
            }
            tc_fence_after();
            uint32_t tm, tile_n;
            coords(u, tm, tile_n);
            const uint32_t row = tm * kBM + quarter * 32 + lane;
            const uint32_t col0 = tile_n * kBN;  // the tile's first column
            __nv_bfloat16 *crow = C + (uint64_t)row * N + col0;
            const uint32_t acc = tmem + lane_base + b * kAccCols;
            float s = 0.0f, c = 0.0f;

            for (uint32_t c0 = 0; c0 < kBN; c0 += 64) {
                uint32_t r0[32], r1[32];
                tc_ld32(acc + c0, r0);
                tc_ld32(acc + c0 + 32, r1);
                tc_wait_ld();
                // columns of the two chunks inside C (none for a row past M)
                const uint32_t v0 = row >= M || col0 + c0 >= N ? 0u : min(32u, N - col0 - c0);
                const uint32_t v1 = row >= M || col0 + c0 + 32 >= N ? 0u : min(32u, N - col0 - c0 - 32);
                epilogue_chunk(r0, crow + c0, s, c, v0);
                epilogue_chunk(r1, crow + c0 + 32, s, c, v1);
                if (kCols) {  // this warp's 32 rows of the chunk's columns
                    cq[quarter * kBN + c0 + lane] = warp_column_sum(r0, lane, coltile);
                    cq[quarter * kBN + c0 + 32 + lane] = warp_column_sum(r1, lane, coltile);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tempty + 8 * b) : "memory");
            if (row < M) rowsum_part[(uint64_t)tile_n * M + row] = (double)s + (double)c;
            if (kCols) {  // the tile's column partials: the four lane quarters merged in order, one row per tile row
                named_bar_sync(1, 128);
#pragma unroll
                for (uint32_t h = 0; h < kBN / 128; ++h) {
                    const uint32_t cc = et + 128 * h;
                    const double v = ((cq[cc] + cq[kBN + cc]) + cq[2 * kBN + cc]) + cq[3 * kBN + cc];
                    if (col0 + cc < N) colsum_part[(uint64_t)tm * N + col0 + cc] = v;
                }
                named_bar_sync(1, 128);  // read before the next tile's partials overwrite them
            }
        }
    } else if constexpr (kRef) {  // ----------------------------------- reference warps
        // Thread rt takes row rt of each tile; the tiles come in the CTA's order.  Per selected K block
        // the group stages the block's 64 column sums in shared memory (one word per thread), each
        // thread reads its row's 64 values of A (eight 16-byte loads of one 128-byte line) and forms
        // its part of the reference.  The named barriers keep the staged sums whole while they are read.
        const uint32_t rt = tid - kGemmThreads;
        float *hsm = (float *)(smem + pad + kRefSumsOff);
        const uint32_t hm = smem_addr(hsm);  // {h, m, h, m}: two columns per 16 bytes
        for (uint32_t u = unit0; u < n_units; u += ustep) {
            uint32_t tm, tn;
            coords(u, tm, tn);
            const uint32_t row = tm * kBM + rt;
            const uint4 *arow = (const uint4 *)(Ag + (uint64_t)(row < M ? row : 0) * K);
            // packed float32 pairs over even and odd columns: the reference (s2, c2), the magnitude (a2, e2)
            uint64_t s2 = 0ull, c2 = 0ull, a2 = 0ull, e2 = 0ull;
            for (uint32_t kb = tn; kb < nkb; kb += tiles_n) {
                named_bar_sync(2, kRefThreads);  // the previous block's sums have been read
                hsm[rt] = kb * kBK + rt / 2 < K ? __ldg((const float *)(wsums + (uint64_t)kb * kBK) + rt) : 0.0f;
                uint4 av[kBK / 8];
#pragma unroll
                for (uint32_t q = 0; q < kBK / 8; ++q)  // past M or K (a multiple of 8): zero
                    av[q] = row < M && kb * kBK + 8 * q < K ? __ldg(arow + kb * (kBK / 8) + q) : make_uint4(0, 0, 0, 0);
                named_bar_sync(2, kRefThreads);  // the staged sums are whole
                uint64_t m2 = 0ull;  // this block's magnitude: a plain chain of 32 terms per half
#pragma unroll
                for (uint32_t q = 0; q < kBK / 8; ++q) {  // 8 columns: a chain of 4 per half
                    uint64_t t = 0ull;
#pragma unroll
                    for (uint32_t e = 0; e < 4; ++e) {
                        const uint32_t w = (&av[q].x)[e];
                        const uint64_t x = f2_pack_bits(w << 16, w & 0xFFFF0000u);
                        const uint4 h = ld_shared_u4(hm + (4 * q + e) * 16);
                        t = f2_fma(x, f2_pack_bits(h.x, h.z), t);
                        m2 = f2_fma(x & kF2Abs, f2_pack_bits(h.y, h.w), m2);
                    }
                    pair2_add(s2, c2, t);
                }
                pair2_add(a2, e2, m2);
            }
            float s0, s1, c0, c1, a0, a1, e0, e1;
            f2_unpack(s2, s0, s1);
            f2_unpack(c2, c0, c1);
            f2_unpack(a2, a0, a1);
            f2_unpack(e2, e0, e1);
            pair_merge(s0, c0, s1, c1);
            pair_merge(a0, e0, a1, e1);
            if (row < M) ref[(uint64_t)tn * M + row] = make_float4(s0, c0, a0, e0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1 && lane == 0 && !mbar_wait(done, 0)) atomicOr(err, 1);
    __syncwarp();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kAccCols) : "memory");
    }
}

// out[j] = sum over p < count of parts[p * n + j] (row checksums from the tile
// partials, or column checksums from the 32-row partials), in a fixed order:
// block = 32 outputs (one per lane) x 8 warps; warp w sums the partials
// p = w, w + 8, ... in turn, then the 8 warp sums are added in warp order.
// Thread 0 also publishes the GEMM's abort flag when `aborted` is given.
__global__ void __launch_bounds__(256) abft_sum_parts_kernel(const double *__restrict__ parts, uint32_t n,
                                                             uint32_t count, double *__restrict__ out,
                                                             const int *__restrict__ err,
                                                             uint32_t *__restrict__ aborted) {
    __shared__ double part[8][32];
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t j = blockIdx.x * 32 + lane;
    if (aborted && blockIdx.x == 0 && threadIdx.x == 0) *aborted = *err != 0 ? 1u : 0u;
    double acc = 0.0;
    if (j < n) {
#pragma unroll 4
        for (uint32_t p = warp; p < count; p += 8) acc = __dadd_rn(acc, parts[(uint64_t)p * n + j]);
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && j < n) {
        double t = part[0][lane];
        for (int w = 1; w < 8; ++w) t = __dadd_rn(t, part[w][lane]);
        out[j] = t;
    }
}

// ---------------------------------------------------------------- the check
//
// The check's sums need far less than float32-pair precision: it compares a
// checksum with a reference under a bound of about K 2^-22 of the magnitude
// mag = sum_k |A[i, k]| sum_j |W[j, k]|, so its own rounding only has to stay
// well below that and be counted in the bound.  Plain float32 chains of at
// most 8 terms are folded into float32 pairs with TwoSum:
//  - W's column sums: 8-row chains per lane, each off by at most 8.01 2^-24
//    of its rows' |W| sum;
//  - the reference A (W^T 1): 8-term fused multiply-add chains (one vector
//    of 8 columns), each off by at most 8.01 2^-24 of its |a| |w| sum, against
//    the column sums rounded to float32 (2^-24 more);
//  - the pairs and their merges: below (n + K + 64) 2^-44 of the magnitude.
// Together the reference is within (20 2^-24 + (n_sum + K + 64) 2^-44) mag of
// A (W^T 1), and that term is added to the bound.  The magnitude itself is
// summed in plain float32 and raised by 1 + 2 (L1 + L2 + S + 8) 2^-24, where L1
// is the longest plain float32 chain of the column sums of |W|, L2 that of a
// lane's magnitude dot product and S the K splits merged after them.  Each
// chain of non-negative terms is off by at most (its length) 2^-24 of its sum,
// so the raised value is an upper bound on the exact magnitude, and the bound
// stays rigorous.
constexpr uint32_t kChain = 8;  // terms of a plain float32 chain before it is folded into a pair

// Column sums of X [rows][K] over one slab of its rows: block (x, y) covers
// columns 256x .. 256x + 255 (8 per lane, one 16-byte load per row) and slab
// y; the 8 warps take the slab's rows in turn.  Writes slabs[y][k] =
// {s, c, a, e}: the float32 pair of sum_j X[j, k], and the plain float32 sum of
// |X[j, k]| (its chain: the warp's rows) as a pair a + e after the warps'
// merge; warps merged in order.  The last block of each column block (a
// counter per column block in `done`, zero at launch) merges the slabs into
// split[] = {h, m} per column.
//
// The weight-gradient check (kWeighted) runs the same kernel over dY or X [T][n] with a weight
// wt[t] = {h, m} per token row (X's or dY's row sums, below): s + c = sum_t X[t, k] h_t from 8-term
// fused multiply-add chains, a = sum_t |X[t, k]| m_t, and its last block compares the merged sums
// with the accumulator checksums (ColCheck) instead of writing split[].
struct ColCheck {
    const float2 *wt;  // {h, m} per row
    const double *checksum;
    double *residual, *bound;
    uint8_t *flag;
    uint32_t *n_flagged;
    double delta;      // the magnitude's raise
    float tol_scale;
    uint32_t n_sum;    // outputs each checksum sums
};

// One launch serves one or two independent column sums (the two sides of a check): column blocks
// below cb0 are side s0's, the rest side s1's; each side has its own slabs and counters, and a
// block whose slab index is past its side's slab count leaves at once.
struct SlabSide {
    const __nv_bfloat16 *X;
    uint32_t rows, K, n_slabs;
    float4 *slabs;
    float2 *split;   // unweighted: the output
    uint32_t *done;  // a counter per column block
    ColCheck o;      // weighted: the check
    uint32_t keep = 1;    // 0: X is read once here, and its lines are the first the L2 gives up
    uint32_t planar = 0;  // unweighted: split[] in the check's planar layout instead of {h, m} per column
};

// zero[0 .. n_zero) and zero2[0 .. n_zero2) are set to 0 by block (0, 0) first: counters and counts
// that only a later launch on the stream uses (null when there are none).
template <bool kWeighted>
__global__ void __launch_bounds__(256, 3) abft_colsum_slab_kernel(const SlabSide s0, const SlabSide s1, uint32_t cb0,
                                                                  uint32_t *__restrict__ zero, uint32_t n_zero,
                                                                  uint32_t *__restrict__ zero2, uint32_t n_zero2) {
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        for (uint32_t z = threadIdx.x; z < n_zero; z += blockDim.x) zero[z] = 0u;
        for (uint32_t z = threadIdx.x; z < n_zero2; z += blockDim.x) zero2[z] = 0u;
    }
    const bool second = blockIdx.x >= cb0;
    const uint32_t bx = second ? blockIdx.x - cb0 : blockIdx.x, by = blockIdx.y;
    const __nv_bfloat16 *__restrict__ X = second ? s1.X : s0.X;
    const uint32_t rows = second ? s1.rows : s0.rows, K = second ? s1.K : s0.K,
                   n_slabs = second ? s1.n_slabs : s0.n_slabs;
    float4 *__restrict__ slabs = second ? s1.slabs : s0.slabs;
    float2 *__restrict__ split = second ? s1.split : s0.split;
    uint32_t *__restrict__ done = second ? s1.done : s0.done;
    const ColCheck o = second ? s1.o : s0.o;
    if (by >= n_slabs) return;  // the whole block
    __shared__ float4 part[8][256];
    __shared__ uint32_t last;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint64_t policy = l2_policy(!(second ? s1.keep : s0.keep));
    const uint32_t k = bx * 256 + lane * 8;
    const uint32_t j0 = (uint32_t)((uint64_t)by * rows / n_slabs),
                   j1 = (uint32_t)((uint64_t)(by + 1) * rows / n_slabs);
    // columns 2q and 2q + 1 of the lane's 8 share packed registers: the pair (s, c) of the sum,
    // the running chain t of up to kChain rows folded into it, the plain sum a of |x|
    uint64_t s[4], c[4], a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) s[q] = c[q] = a[q] = 0ull;
    // n <= kChain rows from row j0r on (every 8th row), in row order
    auto add_rows = [&](const uint4 (&v)[kChain], uint32_t n, uint32_t j0r) {
        uint64_t t[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (uint32_t u = 0; u < kChain; ++u) {
            if (u < n) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                uint64_t hh = 0ull, mm = 0ull;
                if constexpr (kWeighted) {
                    const float2 wt = __ldg(o.wt + j0r + 8 * u);
                    hh = f2_pack_bits(__float_as_uint(wt.x), __float_as_uint(wt.x));
                    mm = f2_pack_bits(__float_as_uint(wt.y), __float_as_uint(wt.y));
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint64_t x = f2_pack_bits(w[q] << 16, w[q] & 0xFFFF0000u);
                    if constexpr (kWeighted) {
                        t[q] = f2_fma(x, hh, t[q]);
                        a[q] = f2_fma(x & kF2Abs, mm, a[q]);
                    } else {
                        t[q] = f2_add(t[q], x);
                        a[q] = f2_add(a[q], x & kF2Abs);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) pair2_add(s[q], c[q], t[q]);
    };
    if (k < K) {
        uint32_t j = j0 + warp;
        uint4 v[kChain];
        for (; j + 8 * (kChain - 1) < j1; j += 8 * kChain) {  // kChain rows in flight per lane, added in row order
            if ((lane & 7u) == 0) {  // the next chain's rows into L2: lanes 0, 8, 16, 24 touch the warp's 4 lines
#pragma unroll
                for (uint32_t u = kChain; u < 2 * kChain; ++u)
                    if (j + 8 * u < j1) prefetch_l2(X + (uint64_t)(j + 8 * u) * K + k);
            }
#pragma unroll
            for (uint32_t u = 0; u < kChain; ++u) v[u] = ld_stream_hint(X + (uint64_t)(j + 8 * u) * K + k, policy);
            add_rows(v, kChain, j);
        }
        if (j < j1) {  // fewer than kChain rows left
            const uint32_t n = (j1 - j + 7) / 8;
#pragma unroll
            for (uint32_t u = 0; u < kChain; ++u)
                v[u] = u < n ? ld_stream_hint(X + (uint64_t)(j + 8 * u) * K + k, policy) : make_uint4(0, 0, 0, 0);
            add_rows(v, n, j);
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float s0, s1, c0, c1, a0, a1;
        f2_unpack(s[q], s0, s1);
        f2_unpack(c[q], c0, c1);
        f2_unpack(a[q], a0, a1);
        part[warp][lane * 8 + 2 * q] = make_float4(s0, c0, a0, 0.0f);
        part[warp][lane * 8 + 2 * q + 1] = make_float4(s1, c1, a1, 0.0f);
    }
    __syncthreads();
    const uint32_t kk = bx * 256 + threadIdx.x;
    if (kk < K) {
        float4 acc = part[0][threadIdx.x];
        for (int w = 1; w < 8; ++w) {
            const float4 q = part[w][threadIdx.x];
            pair_merge(acc.x, acc.y, q.x, q.y);
            pair_merge(acc.z, acc.w, q.z, q.w);
        }
        slabs[(uint64_t)by * K + kk] = acc;
    }
    // The last slab block of this column block merges the column block's slabs (in slab order:
    // the same result whichever block is last) into split[k] = {h, m}: h the float nearest
    // sum_j X[j, k] (the merged pair's sum), m = sum_j |X[j, k]| rounded to float32.
    __syncthreads();
    // Once every block has passed its rows, the check of the other operand's rows may launch: it
    // prefetches its rows into L2 during this grid's last-block merges, then waits for the grid to
    // complete before it reads the column sums.  Without a dependent launch a no-op.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(done + bx, 1u) == n_slabs - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (kk < K) {
        float4 acc = __ldcg(slabs + kk);
        uint32_t y = 1;
        for (; y + 8 <= n_slabs; y += 8) {  // 8 slabs' loads in flight, merged in slab order
            float4 q[8];
#pragma unroll
            for (uint32_t u = 0; u < 8; ++u) q[u] = __ldcg(slabs + (uint64_t)(y + u) * K + kk);
#pragma unroll
            for (uint32_t u = 0; u < 8; ++u) {
                pair_merge(acc.x, acc.y, q[u].x, q[u].y);
                pair_merge(acc.z, acc.w, q[u].z, q[u].w);
            }
        }
        for (; y < n_slabs; ++y) {
            const float4 q = __ldcg(slabs + (uint64_t)y * K + kk);
            pair_merge(acc.x, acc.y, q.x, q.y);
            pair_merge(acc.z, acc.w, q.z, q.w);
        }
        if constexpr (kWeighted) {  // the check of column kk's accumulator checksum (contraction: the rows)
            const double ref = (double)acc.x + (double)acc.y;
            const double mag = ((double)acc.z + (double)acc.w) * (1.0 + o.delta);
            const double g = (double)rows * 0x1p-22;
            const double b = (g * (1.0 + g) + 20.0 * 0x1p-24 + (double)(o.n_sum + rows + 64) * 0x1p-44) * mag +
                             2.0 * (double)rows * (double)o.n_sum * 0x1p-126;
            const double d = o.checksum[kk] - ref;
            o.residual[kk] = d;
            o.bound[kk] = b;
            const uint8_t f = fabs(d) <= (double)o.tol_scale * b ? 0 : 1;  // NaN flags
            o.flag[kk] = f;
            if (f) atomicAdd(o.n_flagged, 1u);
        } else {
            float h = 0.0f, l = 0.0f;  // renormalise: TwoSum of the two parts
            pair_add(h, l, acc.x);
            pair_add(h, l, acc.y);
            const float2 hm = make_float2(__fadd_rn(h, l), __fadd_rn(acc.z, acc.w));
            const bool planar = second ? s1.planar : s0.planar;
            // planar: plane (kk mod 8) / 2 of vector kk / 8, half kk mod 2 (float2 units)
            split[planar ? ((kk & 7u) >> 1) * (K / 4) + (kk >> 3) * 2 + (kk & 1u) : kk] = hm;
        }
    }
    if (threadIdx.x == 0) done[bx] = 0u;  // ready for the next call
}

// Row sums of X [T][n] for the weight-gradient check: out[t] = {h, m}, h the float nearest
// sum_k X[t, k] (4-term plain chains, one per packed half of a 16-byte vector, folded into a
// float32 pair with TwoSum) and m = sum_k |X[t, k]| in plain float32 (its chain: a lane's
// 4 ceil(n / 256) terms, then 6 merges).  One warp per row, the lanes over the row's vectors in
// turn with 8 loads in flight; the lanes' sums meet in a fixed butterfly and lane 0 writes.
// blockIdx.y picks the matrix: (X0, n0, out0) or (X1, n1, out1), both with T rows.  Matrix i's
// lines are the first the L2 gives up when bit i of read_once is set (it is not read again soon).
// Block (0, 0) first sets zero[0 .. n_zero) and zero2[0 .. n_zero2) to 0 (as abft_colsum_slab_kernel).
__global__ void __launch_bounds__(256) abft_rowsum_kernel(const __nv_bfloat16 *__restrict__ X0, uint32_t n0,
                                                          float2 *__restrict__ out0, const __nv_bfloat16 *__restrict__ X1,
                                                          uint32_t n1, float2 *__restrict__ out1, uint32_t T,
                                                          uint32_t read_once, uint32_t *__restrict__ zero,
                                                          uint32_t n_zero, uint32_t *__restrict__ zero2,
                                                          uint32_t n_zero2) {
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        for (uint32_t z = threadIdx.x; z < n_zero; z += blockDim.x) zero[z] = 0u;
        for (uint32_t z = threadIdx.x; z < n_zero2; z += blockDim.x) zero2[z] = 0u;
    }
    const bool second = blockIdx.y != 0;
    const uint64_t policy = l2_policy((read_once >> (second ? 1 : 0)) & 1u);
    const __nv_bfloat16 *__restrict__ X = second ? X1 : X0;
    const uint32_t n = second ? n1 : n0;
    float2 *__restrict__ out = second ? out1 : out0;
    const uint32_t lane = threadIdx.x & 31u, t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;  // the whole warp
    const uint4 *x = (const uint4 *)(X + (uint64_t)t * n);
    const uint32_t nv = n / 8;
    uint64_t s = 0ull, c = 0ull, a = 0ull;
    auto add = [&](const uint4 &v) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint64_t tt = 0ull;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint64_t xx = f2_pack_bits(w[q] << 16, w[q] & 0xFFFF0000u);
            tt = f2_add(tt, xx);
            a = f2_add(a, xx & kF2Abs);
        }
        pair2_add(s, c, tt);
    };
    uint32_t v = lane;
    for (; v + 32 * 7 < nv; v += 32 * 8) {
        uint4 q[8];
#pragma unroll
        for (uint32_t u = 0; u < 8; ++u) q[u] = ld_stream_hint(x + v + 32 * u, policy);
#pragma unroll
        for (uint32_t u = 0; u < 8; ++u) add(q[u]);
    }
    for (; v < nv; v += 32) add(ld_stream_hint(x + v, policy));
    float s0, s1, c0, c1, a0, a1;
    f2_unpack(s, s0, s1);
    f2_unpack(c, c0, c1);
    f2_unpack(a, a0, a1);
    pair_merge(s0, c0, s1, c1);
    float m = __fadd_rn(a0, a1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        pair_merge(s0, c0, __shfl_xor_sync(0xffffffffu, s0, off), __shfl_xor_sync(0xffffffffu, c0, off));
        m = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
    if (lane == 0) {
        float h = 0.0f, l = 0.0f;  // renormalise: TwoSum of the two parts
        pair_add(h, l, s0);
        pair_add(h, l, c0);
        out[t] = make_float2(__fadd_rn(h, l), m);
    }
}

// The check of X [n_rows][K] (A for the row check, W for the column check)
// against the other operand's column sums {h, m}, one K split per block:
// part[y][i] = {s, c, m, 0} with s + c = sum_k X[i, k] h_k over split y's
// columns (8-term chains folded into a float32 pair), and
// m = sum_k |X[i, k]| m_k in plain float32.  Block = 4 warps over 32 rows; a
// warp holds its 8 rows as 4 packed row pairs in every lane, and its 32 lanes
// take the split's vectors lane, lane + 32, ...: each load of a row reads 512
// contiguous bytes, and the column sums come in the planar layout (plane q of
// vector v = {h, m} of columns 8v + 2q and 8v + 2q + 1, 16 bytes, planes
// [4][K / 8]), so that each of their loads reads 512 contiguous bytes too and
// serves 8 rows.  The lanes' sums meet in 5 butterfly steps.  The last split
// block of a row block (a counter per row block) merges the row block's
// partials in split order (the same result whichever block is last) and
// writes, per row: the reference ref = s + c, the magnitude raised by
// (1 + delta) to an upper bound, the bound over n_sum summed outputs, the
// residual against the accumulator checksum and the flag (a NaN residual
// flags).
constexpr uint32_t kChkRows = 32;  // rows per block of the check

struct CheckOut {
    const double *checksum;
    double *residual, *bound;
    uint8_t *flag;
    uint32_t *n_flagged;
    uint32_t *done;  // a counter per row block
    double delta;
    float tol_scale;
    uint32_t n_sum, n_splits;
};

// 8 columns of two rows (packed) against their column sums (the four planes
// w[q] = {h, m, h, m} of columns 2q and 2q + 1): an 8-term fused multiply-add
// chain folded into the pair (rs, rc) with TwoSum, and the magnitude's plain
// chain m.
__device__ __forceinline__ void check_vec(const uint4 &a0, const uint4 &a1, const uint4 (&w)[4], uint64_t &rs,
                                          uint64_t &rc, uint64_t &m) {
    uint64_t t = 0ull;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int q = 2 * qq + e;
            const uint32_t w0 = (&a0.x)[q >> 1], w1 = (&a1.x)[q >> 1];
            const uint64_t a2 = (q & 1) ? f2_pack_bits(w0 & 0xFFFF0000u, w1 & 0xFFFF0000u)
                                        : f2_pack_bits(w0 << 16, w1 << 16);
            const uint32_t h = e ? w[qq].z : w[qq].x, mm = e ? w[qq].w : w[qq].y;
            t = f2_fma(a2, f2_pack_bits(h, h), t);
            m = f2_fma(a2 & kF2Abs, f2_pack_bits(mm, mm), m);
        }
    }
    pair2_add(rs, rc, t);
}

// One launch serves one or two independent checks: row blocks below rb0 are side0's, the rest
// side1's; a block whose split index is past its side's split count leaves at once.
struct CheckSide {
    const __nv_bfloat16 *X;
    uint32_t n_rows, K, vec_per_split;
    const float2 *split;
    float4 *part;
    CheckOut o;
};

__global__ void __launch_bounds__(128, 7) abft_check_kernel(const CheckSide side0, const CheckSide side1, uint32_t rb0) {
    const bool second = blockIdx.x >= rb0;
    const uint32_t bx = second ? blockIdx.x - rb0 : blockIdx.x, by = blockIdx.y;
    const __nv_bfloat16 *__restrict__ X = second ? side1.X : side0.X;
    const uint32_t n_rows = second ? side1.n_rows : side0.n_rows, K = second ? side1.K : side0.K,
                   vec_per_split = second ? side1.vec_per_split : side0.vec_per_split;
    const float2 *__restrict__ split = second ? side1.split : side0.split;
    float4 *__restrict__ part = second ? side1.part : side0.part;
    const CheckOut o = second ? side1.o : side0.o;
    if (by >= o.n_splits) return;  // the whole block
    __shared__ uint32_t last;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t v0 = by * vec_per_split, v1 = min(K / 8, v0 + vec_per_split);
    const uint32_t row0 = bx * kChkRows;
    // Launched as a dependent of the column sums: their grid has completed (and its writes are
    // visible) once this returns.  Without a dependent launch a no-op.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint4 *planes = (const uint4 *)split;  // [4][K / 8]
    const uint32_t nvk = K / 8, r0 = row0 + warp * 8;  // this warp's rows r0 .. r0 + 7
    const __nv_bfloat16 *xw = X + (uint64_t)r0 * K;
    uint64_t rs[4], rc[4], m[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) rs[p] = rc[p] = m[p] = 0ull;
    for (uint32_t v = v0 + lane; v < v1; v += 32) {
        uint4 a[8], w[4];
#pragma unroll
        for (uint32_t rr = 0; rr < 8; ++rr)
            a[rr] = r0 + rr < n_rows ? ld_stream((const uint4 *)(xw + (uint64_t)rr * K) + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q) w[q] = __ldg(planes + (uint64_t)q * nvk + v);
#pragma unroll
        for (int p = 0; p < 4; ++p) check_vec(a[2 * p], a[2 * p + 1], w, rs[p], rc[p], m[p]);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float s0, s1, c0, c1, m0, m1;
        f2_unpack(rs[p], s0, s1);
        f2_unpack(rc[p], c0, c1);
        f2_unpack(m[p], m0, m1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {  // the warp's 32 lanes, a fixed butterfly
            pair_merge(s0, c0, __shfl_xor_sync(0xffffffffu, s0, off), __shfl_xor_sync(0xffffffffu, c0, off));
            pair_merge(s1, c1, __shfl_xor_sync(0xffffffffu, s1, off), __shfl_xor_sync(0xffffffffu, c1, off));
            m0 = __fadd_rn(m0, __shfl_xor_sync(0xffffffffu, m0, off));
            m1 = __fadd_rn(m1, __shfl_xor_sync(0xffffffffu, m1, off));
        }
        const uint32_t r = r0 + 2 * p;
        if (lane == (uint32_t)p) {
            float4 *dst = part + (uint64_t)by * n_rows;
            if (r < n_rows) dst[r] = make_float4(s0, c0, m0, 0.0f);
            if (r + 1 < n_rows) dst[r + 1] = make_float4(s1, c1, m1, 0.0f);
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        last = atomicAdd(o.done + bx, 1u) == o.n_splits - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const uint32_t i = row0 + tid;
    if (tid < kChkRows && i < n_rows) {
        float s = 0.0f, c = 0.0f;
        double mag = 0.0;
        uint32_t y = 0;
        for (; y + 4 <= o.n_splits; y += 4) {  // 4 splits' loads in flight, merged in split order
            float4 p[4];
#pragma unroll
            for (uint32_t u = 0; u < 4; ++u) p[u] = __ldcg(part + (uint64_t)(y + u) * n_rows + i);
#pragma unroll
            for (uint32_t u = 0; u < 4; ++u) {
                pair_merge(s, c, p[u].x, p[u].y);
                mag = __dadd_rn(mag, (double)p[u].z);
            }
        }
        for (; y < o.n_splits; ++y) {
            const float4 p = __ldcg(part + (uint64_t)y * n_rows + i);
            pair_merge(s, c, p.x, p.y);
            mag = __dadd_rn(mag, (double)p.z);
        }
        const double ref = (double)s + (double)c;
        mag *= 1.0 + o.delta;
        const double gk = (double)K * 0x1p-22;
        const double b = (gk * (1.0 + gk) + 20.0 * 0x1p-24 + (double)(o.n_sum + K + 64) * 0x1p-44) * mag +
                         2.0 * (double)K * (double)o.n_sum * 0x1p-126;
        const double d = o.checksum[i] - ref;
        o.residual[i] = d;
        o.bound[i] = b;
        const uint8_t f = fabs(d) <= (double)o.tol_scale * b ? 0 : 1;  // NaN flags
        o.flag[i] = f;
        if (f) atomicAdd(o.n_flagged, 1u);
    }
    if (tid == 0) o.done[bx] = 0u;  // ready for the next call
}

// The fused check's last pass, one launch: per row i, the accumulator checksum rowsum[i] from the
// GEMM's tile partials part[p][i] (double) in abft_sum_parts_kernel's order (eight sums over
// p = s, s + 8, ..., then added for s = 0 .. 7 in turn: the same bits), and the verdict from the
// reference partials ref[p][i] = {s, c, mh, ml} (A[i, :] (W^T 1) over tile p's K blocks and its
// magnitude, float32 pairs), merged over the same eight interleaved runs and then in run order,
// against the row's checksum: the residual, the bound (the verifier's formula, the magnitude raised
// by 1 + delta) and the flag.  Block = 32 rows x 8 threads (thread s of a row
// takes the runs' s-th); block 0's thread 0 publishes the GEMM's abort flag.
__global__ void __launch_bounds__(256) abft_fused_finalize_kernel(const double *__restrict__ part,
                                                                  const float4 *__restrict__ ref, uint32_t n_parts,
                                                                  uint32_t M, uint32_t N, uint32_t K, double delta,
                                                                  float tol_scale, double *__restrict__ rowsum,
                                                                  double *__restrict__ residual,
                                                                  double *__restrict__ bound,
                                                                  uint8_t *__restrict__ flag,
                                                                  uint32_t *__restrict__ n_flagged,
                                                                  const int *__restrict__ err,
                                                                  uint32_t *__restrict__ aborted) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *aborted = *err != 0 ? 1u : 0u;
    const uint32_t sub = threadIdx.x & 7u, i = blockIdx.x * 32 + (threadIdx.x >> 3);
    const bool in = i < M;
    double acc = 0.0;
    float s = 0.0f, c = 0.0f, a = 0.0f, e = 0.0f;
    if (in) {
        uint32_t p = sub;
        for (; p + 8 * 3 < n_parts; p += 8 * 4) {  // 4 partials of each kind in flight, merged in order
            double pd[4];
            float4 pr[4];
#pragma unroll
            for (uint32_t u = 0; u < 4; ++u) {
                pd[u] = part[(uint64_t)(p + 8 * u) * M + i];
                pr[u] = ref[(uint64_t)(p + 8 * u) * M + i];
            }
#pragma unroll
            for (uint32_t u = 0; u < 4; ++u) {
                acc = __dadd_rn(acc, pd[u]);
                pair_merge(s, c, pr[u].x, pr[u].y);
                pair_merge(a, e, pr[u].z, pr[u].w);
            }
        }
        for (; p < n_parts; p += 8) {
            acc = __dadd_rn(acc, part[(uint64_t)p * M + i]);
            const float4 r = ref[(uint64_t)p * M + i];
            pair_merge(s, c, r.x, r.y);
            pair_merge(a, e, r.z, r.w);
        }
    }
    // thread 0 of the row takes the eight runs in order (a row's threads are 8 consecutive lanes)
    const uint32_t lane0 = (threadIdx.x & 31u) & ~7u;
    double t = acc;
    float ts = s, tc = c, ta = a, te = e;
#pragma unroll
    for (uint32_t k = 1; k < 8; ++k) {
        const double ak = __shfl_sync(0xffffffffu, acc, lane0 + k);
        const float sk = __shfl_sync(0xffffffffu, s, lane0 + k), ck = __shfl_sync(0xffffffffu, c, lane0 + k);
        const float ak2 = __shfl_sync(0xffffffffu, a, lane0 + k), ek = __shfl_sync(0xffffffffu, e, lane0 + k);
        t = __dadd_rn(t, ak);
        pair_merge(ts, tc, sk, ck);
        pair_merge(ta, te, ak2, ek);
    }
    if (!in || sub != 0) return;
    rowsum[i] = t;
    const double refv = (double)ts + (double)tc;
    const double mag = ((double)ta + (double)te) * (1.0 + delta);
    const double gk = (double)K * 0x1p-22;
    const double b = (gk * (1.0 + gk) + 20.0 * 0x1p-24 + (double)(N + K + 64) * 0x1p-44) * mag +
                     2.0 * (double)K * (double)N * 0x1p-126;
    const double d = t - refv;
    residual[i] = d;
    bound[i] = b;
    const uint8_t f = fabs(d) <= (double)tol_scale * b ? 0 : 1;  // NaN flags
    flag[i] = f;
    if (f) atomicAdd(n_flagged, 1u);
}

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Row slabs of a column sum over `rows` rows of K columns: about 456 blocks in all
// (3 resident blocks on each of 152 SMs: one wave), at most kMaxSlabs, at least
// 8 rows per slab.  A function of the shapes only, so the workspace size is too.
uint32_t n_slabs_for(uint32_t rows, uint32_t K) {
    const uint32_t col_blocks = (K + 255) / 256;
    uint32_t n = 456 / col_blocks;
    if (n > kMaxSlabs) n = kMaxSlabs;
    if (n > rows / 8) n = rows / 8;
    return n < 1 ? 1 : n;
}

// K splits of the check of `rows` rows: as many as one wave of its blocks of
// kChkRows rows holds (7 resident per SM on 152 SMs: the kernel is held to 73
// registers, a few spilled, for the warps), with at least 128 vectors (4 per
// lane) per split.  A function of the shapes only, so the workspace size
// is too.
uint32_t n_splits_for(uint32_t rows, uint32_t K) {
    const uint32_t nvec = K / 8, row_blocks = (rows + kChkRows - 1) / kChkRows;
    const uint32_t n = 7u * 152u / row_blocks;
    const uint32_t most = nvec / 128 > 0 ? nvec / 128 : 1;
    return n > most ? most : (n < 1 ? 1 : n);
}

// The plain float32 chains behind the magnitude, for its raise factor: the
// longest run of rows one warp sums in a column-sum slab, and the longest run
// of columns one lane sums in a check split (8 per vector, the split's vps
// vectors dealt to 32 lanes) with the 5 butterfly steps after it.
double mag_delta(uint32_t rows_summed, uint32_t n_slabs, uint32_t vps, uint32_t n_splits) {
    const uint32_t slab_rows = (rows_summed + n_slabs - 1) / n_slabs;
    const double l1 = (double)((slab_rows + 7) / 8);
    const double l2 = 8.0 * (double)((vps + 31) / 32) + 5.0;
    return 2.0 * (l1 + l2 + (double)n_splits + 8.0) * 0x1p-24;
}

// Bytes of an operand the verifier keeps in L2 between its two launches: about half the 126 MiB L2.
constexpr uint64_t kKeepL2 = 64ull << 20;

// Workspace: row partials [ceil(N/256)][M] | column partials [ceil(M/128)][N] | W's column sums wsplit [K] |
// A's, asplit [K] | slabs [n_slabs(N, K) + n_slabs(M, K)][K] (W's, then A's) | the check's split
// partials [S(M) M + S(N) N] (A's rows, then W's) | the verifier's last-block counters: one per 256-column
// block of each side's column sums, then one per row block of each side's check (apart, so that the
// check may launch before the column sums complete; zeroed by each verify call) | abort word.
struct AbftWs {
    size_t part, cpart, wsplit, asplit, slabs, chk, done, err, total;
};
AbftWs abft_ws(uint32_t M, uint32_t N, uint32_t K) {
    AbftWs w;
    const size_t ns = (size_t)n_slabs_for(N, K) + n_slabs_for(M, K);  // both sides' slabs
    const size_t nc = (size_t)n_splits_for(M, K) * M + (size_t)n_splits_for(N, K) * N;  // both sides' partials
    w.part = 0;
    const size_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN;
    w.cpart = round_up256(tiles_n * M * sizeof(double));
    w.wsplit = w.cpart + round_up256(tiles_m * N * sizeof(double));
    w.asplit = w.wsplit + round_up256((size_t)K * sizeof(float2));
    w.slabs = w.asplit + round_up256((size_t)K * sizeof(float2));
    w.chk = w.slabs + round_up256(ns * K * sizeof(float4));
    w.done = w.chk + round_up256(nc * sizeof(float4));
    const size_t row_blocks = (M + kChkRows - 1) / kChkRows + (N + kChkRows - 1) / kChkRows,
                 col_blocks = 2 * ((K + 255) / 256);
    w.err = w.done + round_up256((col_blocks + row_blocks) * sizeof(uint32_t));
    w.total = w.err + 256;
    return w;
}

// The plain float32 chains behind a weight-gradient magnitude, for its raise factor: a row-sum
// lane's 4 ceil(n_rowsum / 256) terms and its 6 merges, then a slab warp's rows of the weighted
// column sums (their later merges run on float32 pairs).
double wgrad_mag_delta(uint32_t T, uint32_t n_rowsum, uint32_t n_slabs) {
    const uint32_t slab_rows = (T + n_slabs - 1) / n_slabs;
    const double l1 = 4.0 * (double)((n_rowsum + 255) / 256) + 6.0;
    const double l2 = (double)((slab_rows + 7) / 8);
    return 2.0 * (l1 + l2 + 8.0) * 0x1p-24;
}

// Workspace of the weight-gradient form (dW [N][K] = dY^T X over T tokens): the GEMM's row
// partials [ceil(K/256)][N] | column partials [ceil(N/128)][K] | X's row sums [T] float2 | dY's
// [T] float2 | slabs: dY's [n_slabs(T, N)][N], then X's [n_slabs(T, K)][K] float4 | the last-block
// counters (one per 256-column block of each: zeroed by each verify call) | abort word.
struct WgradWs {
    size_t part, cpart, rsplit, qsplit, slabs, done, err, total;
};
WgradWs wgrad_ws(uint32_t T, uint32_t N, uint32_t K) {
    WgradWs w;
    const size_t tiles_m = (N + kBM - 1) / kBM, tiles_n = (K + kBN - 1) / kBN;
    w.part = 0;
    w.cpart = round_up256(tiles_n * N * sizeof(double));
    w.rsplit = w.cpart + round_up256(tiles_m * K * sizeof(double));
    w.qsplit = w.rsplit + round_up256((size_t)T * sizeof(float2));
    w.slabs = w.qsplit + round_up256((size_t)T * sizeof(float2));
    w.done = w.slabs + round_up256(((size_t)n_slabs_for(T, N) * N + (size_t)n_slabs_for(T, K) * K) * sizeof(float4));
    w.err = w.done + round_up256(((N + 255) / 256 + (K + 255) / 256) * sizeof(uint32_t));
    w.total = w.err + 256;
    return w;
}

}  // namespace

}  // namespace sdc

using namespace sdc;

extern "C" {

size_t sdc_abft_workspace_size(uint32_t M, uint32_t N, uint32_t K) { return abft_ws(M, N, K).total; }

static sdc_status abft_args(const void *d_A, const void *d_W, uint32_t M, uint32_t N, uint32_t K, void *d_ws,
                            size_t ws_bytes, int *dev) {
    if (!d_A || !d_W) return fail(SDC_ERR_NULL, "NULL operand");
    if (M == 0 || N == 0 || K == 0 || N % 8 || K % 8 || K > kMaxK)
        return fail(SDC_ERR_BAD_ARG, "M must be positive, N and K positive multiples of 8, K <= 2^20");
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_device_range(d_A, (uint64_t)M * K * 2, *dev, "d_A");
    if (st == SDC_OK) st = check_device_range(d_W, (uint64_t)N * K * 2, *dev, "d_W");
    if (st != SDC_OK) return st;
    if (((uint64_t)d_A | (uint64_t)d_W) & 15u) return fail(SDC_ERR_BAD_POINTER, "A and W must be 16-byte aligned");
    if (!d_ws || ws_bytes < sdc_abft_workspace_size(M, N, K))
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    return check_device_range(d_ws, sdc_abft_workspace_size(M, N, K), *dev, "d_ws");
}

sdc_status sdc_abft_gemm(const void *d_A, const void *d_W, void *d_C, uint32_t M, uint32_t N, uint32_t K,
                         double *d_rowsum, double *d_colsum, uint32_t *d_aborted, void *d_ws, size_t ws_bytes,
                         sdc_stream_t stream) {
    int dev = -1;
    sdc_status st = abft_args(d_A, d_W, M, N, K, d_ws, ws_bytes, &dev);
    if (st != SDC_OK) return st;
    if (!d_C || !d_rowsum || !d_aborted) return fail(SDC_ERR_NULL, "NULL output");
    st = check_spans({{d_C, (uint64_t)M * N * 2, "d_C"},
                      {d_rowsum, (uint64_t)M * 8, "d_rowsum"},
                      {d_colsum, d_colsum ? (uint64_t)N * 8 : 0, "d_colsum"},
                      {d_aborted, 4, "d_aborted"}},
                     dev);
    if (st != SDC_OK) return st;
    if ((uint64_t)d_C & 15u) return fail(SDC_ERR_BAD_POINTER, "C must be 16-byte aligned");
    const uint32_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN, sms = (uint32_t)sm_count(dev);
    CUtensorMap mapA, mapW;
    st = make_map_sw128(&mapA, d_A, M, K, kBM);
    if (st == SDC_OK) st = make_map_sw128(&mapW, d_W, N, K, kBN);
    if (st != SDC_OK) return st;
    const AbftWs w = abft_ws(M, N, K);
    double *part = (double *)((char *)d_ws + w.part);
    double *cpart = (double *)((char *)d_ws + w.cpart);
    int *err = (int *)((char *)d_ws + w.err);
    cudaStream_t s = (cudaStream_t)stream;
    const bool cols = d_colsum != nullptr;
    auto kernel = cols ? abft_gemm_kernel<true, false, false> : abft_gemm_kernel<false, false, false>;
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);
    const uint32_t smem_bytes = cols ? kGemmSmemCols : kGemmSmem;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm setup");
    const uint32_t n_units = tiles_m * tiles_n;
    const uint32_t grid = n_units < sms ? n_units : sms;  // one CTA per SM
    // A band of tile rows holds about 24 MiB of A, a fraction of the 126 MiB L2.
    uint32_t band_m = (uint32_t)((24u << 20) / ((size_t)kBM * K * 2));
    band_m = band_m < 1 ? 1 : (band_m > tiles_m ? tiles_m : band_m);
    kernel<<<grid, kGemmThreads, smem_bytes, s>>>(mapA, mapW, (__nv_bfloat16 *)d_C, M, N, K, band_m, part, cpart, err,
                                                  nullptr, nullptr, nullptr, nullptr, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm launch");
    abft_sum_parts_kernel<<<(M + 31) / 32, 256, 0, s>>>(part, M, tiles_n, d_rowsum, err, d_aborted);
    if (cols) abft_sum_parts_kernel<<<(N + 31) / 32, 256, 0, s>>>(cpart, N, tiles_m, d_colsum, nullptr, nullptr);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_gemm launch");
}

sdc_status sdc_abft_verify(const void *d_A, const void *d_W, uint32_t M, uint32_t N, uint32_t K, const double *d_rowsum,
                           const double *d_colsum, float tol_scale, double *d_residual, double *d_bound,
                           uint8_t *d_flag, double *d_residual_col, double *d_bound_col, uint8_t *d_flag_col,
                           sdc_abft_summary *d_summary, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    int dev = -1;
    sdc_status st = abft_args(d_A, d_W, M, N, K, d_ws, ws_bytes, &dev);
    if (st != SDC_OK) return st;
    if (!d_rowsum || !d_residual || !d_bound || !d_flag || !d_summary) return fail(SDC_ERR_NULL, "NULL output");
    const bool cols = d_colsum != nullptr;
    if (cols && (!d_residual_col || !d_bound_col || !d_flag_col)) return fail(SDC_ERR_NULL, "NULL column output");
    if (!(tol_scale > 0.0f)) return fail(SDC_ERR_BAD_ARG, "tol_scale must be positive");
    const uint64_t nc = cols ? N : 0;
    st = check_spans({{d_rowsum, (uint64_t)M * 8, "d_rowsum"},
                      {d_residual, (uint64_t)M * 8, "d_residual"},
                      {d_bound, (uint64_t)M * 8, "d_bound"},
                      {d_flag, M, "d_flag"},
                      {d_colsum, nc * 8, "d_colsum"},
                      {d_residual_col, nc * 8, "d_residual_col"},
                      {d_bound_col, nc * 8, "d_bound_col"},
                      {d_flag_col, nc, "d_flag_col"},
                      {d_summary, sizeof(sdc_abft_summary), "d_summary"}},
                     dev);
    if (st != SDC_OK) return st;
    const AbftWs w = abft_ws(M, N, K);
    float2 *wsplit = (float2 *)((char *)d_ws + w.wsplit), *asplit = (float2 *)((char *)d_ws + w.asplit);
    float4 *slabs = (float4 *)((char *)d_ws + w.slabs), *chk = (float4 *)((char *)d_ws + w.chk);
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *done = (uint32_t *)((char *)d_ws + w.done);
    // Both sides at once, in two launches: the column sums of W (for the rows) and of A (for the
    // columns), then A's rows against W's sums and W's rows against A's.  Each side has its own
    // slabs, split partials and counters; without columns each launch serves the row side alone.
    const uint32_t cb = (K + 255) / 256, ns_w = n_slabs_for(N, K), ns_a = n_slabs_for(M, K);
    auto vps_for = [&](uint32_t n_rows) {  // vectors per split; the split count re-derived, so none is empty
        const uint32_t sp = n_splits_for(n_rows, K);
        return (K / 8 + sp - 1) / sp;
    };
    const uint32_t vps_a = vps_for(M), nsp_a = (K / 8 + vps_a - 1) / vps_a;
    const uint32_t vps_w = vps_for(N), nsp_w = (K / 8 + vps_w - 1) / vps_w;
    const uint32_t rb_a = (M + kChkRows - 1) / kChkRows, rb_w = (N + kChkRows - 1) / kChkRows;
    SlabSide sw{(const __nv_bfloat16 *)d_W, N, K, ns_w, slabs, wsplit, done, ColCheck{}};
    SlabSide sa{(const __nv_bfloat16 *)d_A, M, K, ns_a, slabs + (size_t)ns_w * K, asplit, done + cb, ColCheck{}};
    sw.planar = sa.planar = 1;  // the layout the check reads
    // L2 use: rows only, the column sums read W once (its lines leave L2 first, so that they do not
    // push out lines the check's A rows may still find).  Rows and columns: the check re-reads both
    // operands; the smaller keeps its lines if it fits in about half the L2, the other leaves first.
    const uint64_t a_bytes = (uint64_t)M * K * 2, w_bytes = (uint64_t)N * K * 2;
    sw.keep = cols && w_bytes < a_bytes && w_bytes <= kKeepL2;
    sa.keep = cols && !sw.keep && a_bytes <= kKeepL2;
    // the column sums' counters are zeroed here; the check's counters and the summary by the column
    // sums' first block (the check reads them only after that grid has completed)
    cudaError_t e = cudaMemsetAsync(done, 0, 2 * cb * sizeof(uint32_t), s);
    if (e == cudaSuccess) {
        abft_colsum_slab_kernel<false><<<dim3(cols ? 2 * cb : cb, cols && ns_a > ns_w ? ns_a : ns_w), 256, 0, s>>>(
            sw, cols ? sa : sw, cb, done + 2 * cb, rb_a + rb_w, (uint32_t *)d_summary,
            (uint32_t)(sizeof(sdc_abft_summary) / 4));
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
        // rows: A (W^T 1) over the N columns each row checksum sums; columns: W (A^T 1) over the M rows.
        // A programmatic dependent launch: its blocks start once the column sums' blocks have passed
        // their rows, prefetch their own rows into L2 and wait for that grid before they read the sums.
        uint32_t *cdone = done + 2 * cb;
        const CheckSide ca{(const __nv_bfloat16 *)d_A, M, K, vps_a, wsplit, chk,
                           CheckOut{d_rowsum, d_residual, d_bound, d_flag, &d_summary->n_flagged, cdone,
                                    mag_delta(N, ns_w, vps_a, nsp_a), tol_scale, N, nsp_a}};
        const CheckSide cw{(const __nv_bfloat16 *)d_W, N, K, vps_w, asplit, chk + (size_t)nsp_a * M,
                           CheckOut{d_colsum, d_residual_col, d_bound_col, d_flag_col, &d_summary->n_flagged_cols,
                                    cdone + rb_a, mag_delta(M, ns_a, vps_w, nsp_w), tol_scale, M, nsp_w}};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cols ? rb_a + rb_w : rb_a, cols && nsp_w > nsp_a ? nsp_w : nsp_a);
        cfg.blockDim = dim3(128);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, abft_check_kernel, ca, cols ? cw : ca, rb_a);
    }
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_verify launch");
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_verify launch");
}

size_t sdc_abft_wgrad_workspace_size(uint32_t T, uint32_t N, uint32_t K) { return wgrad_ws(T, N, K).total; }

static sdc_status wgrad_args(const void *d_dY, const void *d_X, uint32_t T, uint32_t N, uint32_t K, void *d_ws,
                             size_t ws_bytes, int *dev) {
    if (!d_dY || !d_X) return fail(SDC_ERR_NULL, "NULL operand");
    if (T == 0 || N == 0 || K == 0 || N % 8 || K % 8 || T > kMaxK)
        return fail(SDC_ERR_BAD_ARG, "T must be positive and <= 2^20, N and K positive multiples of 8");
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_device_range(d_dY, (uint64_t)T * N * 2, *dev, "d_dY");
    if (st == SDC_OK) st = check_device_range(d_X, (uint64_t)T * K * 2, *dev, "d_X");
    if (st != SDC_OK) return st;
    if (((uint64_t)d_dY | (uint64_t)d_X) & 15u) return fail(SDC_ERR_BAD_POINTER, "dY and X must be 16-byte aligned");
    if (!d_ws || ws_bytes < sdc_abft_wgrad_workspace_size(T, N, K))
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_wgrad_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    return check_device_range(d_ws, sdc_abft_wgrad_workspace_size(T, N, K), *dev, "d_ws");
}

sdc_status sdc_abft_gemm_wgrad(const void *d_dY, const void *d_X, void *d_dW, uint32_t T, uint32_t N, uint32_t K,
                               double *d_rowsum, double *d_colsum, uint32_t *d_aborted, void *d_ws, size_t ws_bytes,
                               sdc_stream_t stream) {
    int dev = -1;
    sdc_status st = wgrad_args(d_dY, d_X, T, N, K, d_ws, ws_bytes, &dev);
    if (st != SDC_OK) return st;
    if (!d_dW || !d_rowsum || !d_aborted) return fail(SDC_ERR_NULL, "NULL output");
    st = check_spans({{d_dW, (uint64_t)N * K * 2, "d_dW"},
                      {d_rowsum, (uint64_t)N * 8, "d_rowsum"},
                      {d_colsum, d_colsum ? (uint64_t)K * 8 : 0, "d_colsum"},
                      {d_aborted, 4, "d_aborted"}},
                     dev);
    if (st != SDC_OK) return st;
    if ((uint64_t)d_dW & 15u) return fail(SDC_ERR_BAD_POINTER, "dW must be 16-byte aligned");
    // the GEMM kernel on dW [N][K] = A . W^T with A = dY^T and W = X^T, both MN-major, contraction T
    const uint32_t tiles_m = (N + kBM - 1) / kBM, tiles_n = (K + kBN - 1) / kBN, sms = (uint32_t)sm_count(dev);
    CUtensorMap mapA, mapW;
    st = make_map_sw128(&mapA, d_dY, T, N, kBK);
    if (st == SDC_OK) st = make_map_sw128(&mapW, d_X, T, K, kBK);
    if (st != SDC_OK) return st;
    const WgradWs w = wgrad_ws(T, N, K);
    double *part = (double *)((char *)d_ws + w.part);
    double *cpart = (double *)((char *)d_ws + w.cpart);
    int *err = (int *)((char *)d_ws + w.err);
    cudaStream_t s = (cudaStream_t)stream;
    const bool cols = d_colsum != nullptr;
    auto kernel = cols ? abft_gemm_kernel<true, true, false> : abft_gemm_kernel<false, true, false>;
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);
    const uint32_t smem_bytes = cols ? kGemmSmemCols : kGemmSmem;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm_wgrad setup");
    const uint32_t n_units = tiles_m * tiles_n;
    const uint32_t grid = n_units < sms ? n_units : sms;  // one CTA per SM
    // a band of tile rows holds about 24 MiB of dY's columns
    uint32_t band_m = (uint32_t)((24u << 20) / ((size_t)kBM * T * 2));
    band_m = band_m < 1 ? 1 : (band_m > tiles_m ? tiles_m : band_m);
    kernel<<<grid, kGemmThreads, smem_bytes, s>>>(mapA, mapW, (__nv_bfloat16 *)d_dW, N, K, T, band_m, part, cpart, err,
                                                  nullptr, nullptr, nullptr, nullptr, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm_wgrad launch");
    abft_sum_parts_kernel<<<(N + 31) / 32, 256, 0, s>>>(part, N, tiles_n, d_rowsum, err, d_aborted);
    if (cols) abft_sum_parts_kernel<<<(K + 31) / 32, 256, 0, s>>>(cpart, K, tiles_m, d_colsum, nullptr, nullptr);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_gemm_wgrad launch");
}

sdc_status sdc_abft_verify_wgrad(const void *d_dY, const void *d_X, uint32_t T, uint32_t N, uint32_t K,
                                 const double *d_rowsum, const double *d_colsum, float tol_scale, double *d_residual,
                                 double *d_bound, uint8_t *d_flag, double *d_residual_col, double *d_bound_col,
                                 uint8_t *d_flag_col, sdc_abft_summary *d_summary, void *d_ws, size_t ws_bytes,
                                 sdc_stream_t stream) {
    int dev = -1;
    sdc_status st = wgrad_args(d_dY, d_X, T, N, K, d_ws, ws_bytes, &dev);
    if (st != SDC_OK) return st;
    if (!d_rowsum || !d_residual || !d_bound || !d_flag || !d_summary) return fail(SDC_ERR_NULL, "NULL output");
    const bool cols = d_colsum != nullptr;
    if (cols && (!d_residual_col || !d_bound_col || !d_flag_col)) return fail(SDC_ERR_NULL, "NULL column output");
    if (!(tol_scale > 0.0f)) return fail(SDC_ERR_BAD_ARG, "tol_scale must be positive");
    const uint64_t nc = cols ? K : 0;
    st = check_spans({{d_rowsum, (uint64_t)N * 8, "d_rowsum"},
                      {d_residual, (uint64_t)N * 8, "d_residual"},
                      {d_bound, (uint64_t)N * 8, "d_bound"},
                      {d_flag, N, "d_flag"},
                      {d_colsum, nc * 8, "d_colsum"},
                      {d_residual_col, nc * 8, "d_residual_col"},
                      {d_bound_col, nc * 8, "d_bound_col"},
                      {d_flag_col, nc, "d_flag_col"},
                      {d_summary, sizeof(sdc_abft_summary), "d_summary"}},
                     dev);
    if (st != SDC_OK) return st;
    const WgradWs w = wgrad_ws(T, N, K);
    float2 *rsplit = (float2 *)((char *)d_ws + w.rsplit), *qsplit = (float2 *)((char *)d_ws + w.qsplit);
    float4 *slabs = (float4 *)((char *)d_ws + w.slabs);
    uint32_t *done = (uint32_t *)((char *)d_ws + w.done);
    const size_t done_bytes = w.err - w.done;
    cudaStream_t s = (cudaStream_t)stream;
    // Both sides at once, in two launches: X's row sums (the weights of dY's column sums: the rows of
    // dW, each checksum summing K outputs) and dY's (the weights of X's: the columns, each summing N),
    // then both weighted column sums, each compared in its last blocks with its checksums.
    // L2 use: the second launch reads both operands again; X (the smaller) keeps its lines if it fits in
    // about half the L2, dY's leave first, then and in the second launch, which reads it last.
    const bool keep_x = (uint64_t)T * K * 2 <= kKeepL2;
    // its first block also zeroes the second launch's counters and the summary
    abft_rowsum_kernel<<<dim3((T + 7) / 8, cols ? 2 : 1), 256, 0, s>>>(
        (const __nv_bfloat16 *)d_X, K, rsplit, (const __nv_bfloat16 *)d_dY, N, qsplit, T, (keep_x ? 0u : 1u) | 2u, done,
        (uint32_t)(done_bytes / 4), (uint32_t *)d_summary, (uint32_t)(sizeof(sdc_abft_summary) / 4));
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        const uint32_t cb_n = (N + 255) / 256, ns_n = n_slabs_for(T, N), ns_k = n_slabs_for(T, K);
        SlabSide sr{(const __nv_bfloat16 *)d_dY, T, N, ns_n, slabs, nullptr, done,
                          ColCheck{rsplit, d_rowsum, d_residual, d_bound, d_flag, &d_summary->n_flagged,
                                   wgrad_mag_delta(T, K, ns_n), tol_scale, K}};
        const SlabSide sc{(const __nv_bfloat16 *)d_X, T, K, ns_k, slabs + (size_t)ns_n * N, nullptr, done + cb_n,
                          ColCheck{qsplit, d_colsum, d_residual_col, d_bound_col, d_flag_col,
                                   &d_summary->n_flagged_cols, wgrad_mag_delta(T, N, ns_k), tol_scale, N}};
        sr.keep = 0;
        abft_colsum_slab_kernel<true>
            <<<dim3(cols ? cb_n + (K + 255) / 256 : cb_n, cols && ns_k > ns_n ? ns_k : ns_n), 256, 0, s>>>(
                sr, cols ? sc : sr, cb_n, nullptr, 0, nullptr, 0);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_verify_wgrad launch");
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_verify_wgrad launch");
}

size_t sdc_abft_weight_sums_workspace_size(uint32_t N, uint32_t K) {
    if (N == 0 || K == 0 || N % 8 || K % 8 || K > kMaxK) return 0;
    return round_up256((size_t)n_slabs_for(N, K) * K * sizeof(float4)) + round_up256((K + 255) / 256 * sizeof(uint32_t));
}

sdc_status sdc_abft_weight_sums(const void *d_W, uint32_t N, uint32_t K, float *d_wsums, void *d_ws, size_t ws_bytes,
                                sdc_stream_t stream) {
    if (!d_W || !d_wsums || !d_ws) return fail(SDC_ERR_NULL, "NULL argument");
    if (N == 0 || K == 0 || N % 8 || K % 8 || K > kMaxK)
        return fail(SDC_ERR_BAD_ARG, "N and K positive multiples of 8, K <= 2^20");
    const size_t need = sdc_abft_weight_sums_workspace_size(N, K);
    if (ws_bytes < need) return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_weight_sums_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    if ((uint64_t)d_W & 15u) return fail(SDC_ERR_BAD_POINTER, "W must be 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    sdc_status st = check_spans({{d_W, (uint64_t)N * K * 2, "d_W"}, {d_wsums, (uint64_t)K * 8, "d_wsums"},
                                 {d_ws, need, "d_ws"}},
                                dev);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const uint32_t ns = n_slabs_for(N, K), cb = (K + 255) / 256;
    float4 *slabs = (float4 *)d_ws;
    uint32_t *done = (uint32_t *)((char *)d_ws + round_up256((size_t)ns * K * sizeof(float4)));
    e = cudaMemsetAsync(done, 0, cb * sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_weight_sums setup");
    const SlabSide sw{(const __nv_bfloat16 *)d_W, N, K, ns, slabs, (float2 *)d_wsums, done, ColCheck{}};
    abft_colsum_slab_kernel<false><<<dim3(cb, ns), 256, 0, s>>>(sw, sw, cb, nullptr, 0, nullptr, 0);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_weight_sums launch");
}

// Workspace of the fused check: the row checksums' tile partials [ceil(N/256)][M] double | the
// reference partials [ceil(N/256)][M] float4 | abort word.
size_t sdc_abft_gemm_checked_workspace_size(uint32_t M, uint32_t N, uint32_t K) {
    if (M == 0 || N == 0 || K == 0 || N % 8 || K % 8 || K > kMaxK) return 0;
    const size_t tiles_n = (N + kBN - 1) / kBN;
    return round_up256(tiles_n * M * sizeof(double)) + round_up256(tiles_n * M * sizeof(float4)) + 256;
}

sdc_status sdc_abft_gemm_checked(const void *d_A, const void *d_W, void *d_C, uint32_t M, uint32_t N, uint32_t K,
                                 const float *d_wsums, float tol_scale, double *d_rowsum, double *d_residual,
                                 double *d_bound, uint8_t *d_flag, sdc_abft_summary *d_summary, uint32_t *d_aborted,
                                 void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    if (!d_A || !d_W || !d_C || !d_wsums || !d_rowsum || !d_residual || !d_bound || !d_flag || !d_summary ||
        !d_aborted || !d_ws)
        return fail(SDC_ERR_NULL, "NULL argument");
    if (M == 0 || N == 0 || K == 0 || N % 8 || K % 8 || K > kMaxK)
        return fail(SDC_ERR_BAD_ARG, "M must be positive, N and K positive multiples of 8, K <= 2^20");
    const size_t need = sdc_abft_gemm_checked_workspace_size(M, N, K);
    if (ws_bytes < need) return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_abft_gemm_checked_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    if (((uint64_t)d_A | (uint64_t)d_W) & 15u) return fail(SDC_ERR_BAD_POINTER, "A and W must be 16-byte aligned");
    int dev = -1;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return cuda_fail(e0, "cudaGetDevice");
    sdc_status st = check_spans({{d_A, (uint64_t)M * K * 2, "d_A"}, {d_W, (uint64_t)N * K * 2, "d_W"},
                                 {d_ws, need, "d_ws"}},
                                dev);
    if (st != SDC_OK) return st;
    if (!(tol_scale > 0.0f)) return fail(SDC_ERR_BAD_ARG, "tol_scale must be positive");
    st = check_spans({{d_C, (uint64_t)M * N * 2, "d_C"},
                      {d_wsums, (uint64_t)K * 8, "d_wsums"},
                      {d_rowsum, (uint64_t)M * 8, "d_rowsum"},
                      {d_residual, (uint64_t)M * 8, "d_residual"},
                      {d_bound, (uint64_t)M * 8, "d_bound"},
                      {d_flag, M, "d_flag"},
                      {d_summary, sizeof(sdc_abft_summary), "d_summary"},
                      {d_aborted, 4, "d_aborted"}},
                     dev);
    if (st != SDC_OK) return st;
    if (((uint64_t)d_C | (uint64_t)d_wsums) & 15u) return fail(SDC_ERR_BAD_POINTER, "C and wsums must be 16-byte aligned");
    const uint32_t tiles_m = (M + kBM - 1) / kBM, tiles_n = (N + kBN - 1) / kBN, sms = (uint32_t)sm_count(dev);
    CUtensorMap mapA, mapW;
    st = make_map_sw128(&mapA, d_A, M, K, kBM);
    if (st == SDC_OK) st = make_map_sw128(&mapW, d_W, N, K, kBN);
    if (st != SDC_OK) return st;
    double *part = (double *)d_ws;
    float4 *ref = (float4 *)((char *)d_ws + round_up256((size_t)tiles_n * M * sizeof(double)));
    int *err = (int *)((char *)d_ws + need - 256);
    cudaStream_t s = (cudaStream_t)stream;
    auto kernel = abft_gemm_kernel<false, false, true>;
    cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);  // the summary is zeroed by the GEMM kernel
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmemRef);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm_checked setup");
    const uint32_t n_units = tiles_m * tiles_n;
    const uint32_t grid = n_units < sms ? n_units : sms;
    uint32_t band_m = (uint32_t)((24u << 20) / ((size_t)kBM * K * 2));
    band_m = band_m < 1 ? 1 : (band_m > tiles_m ? tiles_m : band_m);
    kernel<<<grid, kGemmThreads + kRefThreads, kGemmSmemRef, s>>>(mapA, mapW, (__nv_bfloat16 *)d_C, M, N, K, band_m,
                                                                part, nullptr, err, (const float2 *)d_wsums, ref,
                                                                (const __nv_bfloat16 *)d_A, (uint32_t *)d_summary,
                                                                (uint32_t)(sizeof(sdc_abft_summary) / 4));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sdc_abft_gemm_checked launch");
    // the magnitude's plain chains: W's column sums (a slab warp's rows), a stage's 32 terms per half
    const uint32_t ns = n_slabs_for(N, K), slab_rows = (N + ns - 1) / ns;
    const double delta = 2.0 * ((double)((slab_rows + 7) / 8) + 32.0 + 8.0) * 0x1p-24;
    abft_fused_finalize_kernel<<<(M + 31) / 32, 256, 0, s>>>(part, ref, tiles_n, M, N, K, delta, tol_scale, d_rowsum,
                                                            d_residual, d_bound, d_flag, &d_summary->n_flagged, err,
                                                            d_aborted);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_abft_gemm_checked launch");
}

}  // extern "C"
