// sdc_attn.cu -- the dV half of the attention backward on the 5th-generation
// tensor cores, with the invariant 1^T dV = 1^T dO taken from the float32
// accumulator.
//
// "Safeguarding LLM Training at Scale: Online SDC Detection and Insights from
// 35 Million GPU Hours" (review page), method section 3: in the attention
// backward dV = P^T dO, and every row of the softmax P sums to 1, so the
// column sums satisfy 1^T dV = 1^T dO.  P is rebuilt in the backward from
// Q K^T, the softmax and the log-sum-exp saved by the forward, so an error
// anywhere along that chain that breaks the row sums also breaks the
// invariant.  AEGIS takes both sides' column sums from float32 accumulators.
//
// Per head (BH heads of L tokens, head dimension 128, Q/K/dO/dV bf16
// [BH][L][128], the forward's natural-log log-sum-exp float32 [BH][L]):
//   P[i, j] = exp(scale q_i . k_j - lse_i)   (0 for j > i when causal)
//   dV[j, :] = sum_i P[i, j] dO[i, :]        (P rounded to bf16, fp32 accumulate)
//   invariant per column c: sum_j dV_acc[j, c]  vs  sum_i dO[i, c].
//
// Kernels:
//   attn_do_prep_kernel -- dO^T [BH][128][L] for the MMA (both MMA operands
//     then sit K-major in shared memory) and float32-pair column sums of dO and
//     |dO| per 128-row block;
//   attn_dv_kernel -- one CTA per (128-key block, head), 6 warps:
//     warp 0 lane 0: TMA -- the K tile once, then per 128-query step the Q
//       tile, the dO^T tile and the step's 128 log-sum-exps into one of two
//       stages;
//     warp 1 lane 0: MMA -- S^T = K Q^T (M = keys, N = queries, K = 128) into
//       one of two 128-column TMEM buffers, issued a step ahead, and
//       dV += P^T dO (M = keys, N = 128, K = queries) into a third;
//     warps 2..5: softmax -- each thread owns one key (a TMEM lane), reads its
//       128 scores, forms exp2(s scale log2(e) - lse log2(e)) (masked when
//       causal), rounds to bf16 and writes its row of P^T into one of two
//       128-byte swizzled shared-memory tiles; at the end it reads its row of
//       dV, stores it as bf16, and the 128 threads sum dV's columns (float32
//       pairs) through shared memory;
//   attn_invariant_kernel -- per (head, column): the block partials merged in
//     order, the residual, the bound, the flag.
// Every wait is bounded; a wait that gives up sets the call's abort flag and
// the block still drains its copies and MMAs (bounded) and frees its TMEM.
#include "sdc_internal.cuh"
#include "sdc_tc.cuh"

namespace sdc {

namespace {

constexpr uint32_t kHD = 128;                    // head dimension
constexpr uint32_t kBlk = 128;                   // keys per CTA, queries per step
constexpr uint32_t kTile = kBlk * kHD * 2;       // 32 KiB: a [128 x 128] bf16 tile = two 64-column swizzled blocks
constexpr uint32_t kHalf = kBlk * 128;           // 16 KiB: one 64-column block
constexpr uint32_t kStages = 2;
constexpr uint32_t kAttnThreads = 192;
// barriers: kfull, full[2], empty[2], sfull[2], sempty[2], pfull[2], pempty[2], dvfull
constexpr uint32_t kNumBars = 14;
// shared memory: K tile | stages (Q tile, dO^T tile) | P^T tiles [2] | lse [2][128] | barriers | TMEM slot
constexpr uint32_t kOffK = 0, kOffStage = kTile, kOffP = kOffStage + kStages * 2 * kTile,
                   kOffLse = kOffP + 2 * kTile, kOffBar = kOffLse + kStages * kBlk * 4, kOffSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kAttnSmem = 1024 + kOffSlot + 16;
constexpr uint32_t kScratchPitch = kHD + 1;  // float row pitch of the column-sum scratch (conflict-free both ways)
static_assert(kBlk * kScratchPitch * 4 <= kStages * 2 * kTile, "column-sum scratch must fit in the stages");
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_dv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapDoT, const float *__restrict__ lse, uint32_t L,
                   float scale_log2, uint32_t causal, __nv_bfloat16 *__restrict__ dV, float2 *__restrict__ part_dv,
                   int *__restrict__ err) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    const uint32_t kb = blockIdx.x, bh = blockIdx.y, nkb = gridDim.x;
    const uint32_t base = smem_addr(smem), pad = ((base + 1023u) & ~1023u) - base;
    unsigned char *sm = smem + pad;
    const uint32_t s0 = base + pad;
    const uint32_t sK = s0 + kOffK, sStage = s0 + kOffStage, sP = s0 + kOffP, sLse = s0 + kOffLse;
    const uint32_t bar = s0 + kOffBar;
    const uint32_t kfull = bar, full = bar + 8, empty = bar + 24, sfull = bar + 40, sempty = bar + 56,
                   pfull = bar + 72, pempty = bar + 88, dvfull = bar + 104;
    uint32_t *tmem_slot = (uint32_t *)(sm + kOffSlot);
    const uint32_t q_first = causal ? kb : 0u, nq = nkb - q_first;
    const uint32_t row0 = bh * L;  // this head's first row in the [BH * L, 128] views

    if (warp == 1) {  // S buffers at columns 0 and 128, dV at 256
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(512u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(kfull, 1);
        for (uint32_t i = 0; i < 2; ++i) {
            mbar_init(full + 8 * i, 1);
            mbar_init(empty + 8 * i, 1);
            mbar_init(sfull + 8 * i, 1);
            mbar_init(sempty + 8 * i, 4);  // one arrival per softmax warp
            mbar_init(pfull + 8 * i, 4);
            mbar_init(pempty + 8 * i, 1);
        }
        mbar_init(dvfull, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------ TMA producer
            mbar_arrive_expect_tx(kfull, kTile);
            tma_load_2d(sK, &mapK, 0, (int32_t)(row0 + kb * kBlk), kfull);
            tma_load_2d(sK + kHalf, &mapK, 64, (int32_t)(row0 + kb * kBlk), kfull);
            uint32_t t = 0;
            for (; t < nq; ++t) {
                const uint32_t st = t % kStages, qb = q_first + t;
                if (t >= kStages && !mbar_wait(empty + 8 * st, ((t / kStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t sQ = sStage + st * 2 * kTile, sDo = sQ + kTile;
                mbar_arrive_expect_tx(full + 8 * st, 2 * kTile + kBlk * 4);
                tma_load_2d(sQ, &mapQ, 0, (int32_t)(row0 + qb * kBlk), full + 8 * st);
                tma_load_2d(sQ + kHalf, &mapQ, 64, (int32_t)(row0 + qb * kBlk), full + 8 * st);
                tma_load_2d(sDo, &mapDoT, (int32_t)(qb * kBlk), (int32_t)(bh * kHD), full + 8 * st);
                tma_load_2d(sDo + kHalf, &mapDoT, (int32_t)(qb * kBlk + 64), (int32_t)(bh * kHD), full + 8 * st);
                bulk_g2s(sLse + st * kBlk * 4, lse + (uint64_t)row0 + qb * kBlk, kBlk * 4, full + 8 * st);
            }
            // Let no copy land after the block has left: wait (bounded) for the last ones issued.
            if (!mbar_wait(kfull, 0)) ok = false;
            for (uint32_t j = t > kStages ? t - kStages : 0; j < t; ++j)
                if (!mbar_wait(full + 8 * (j % kStages), (j / kStages) & 1)) ok = false;
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ------------------------------------------ MMA issuer
            constexpr uint32_t idesc = umma_idesc(kBlk, kBlk);
            auto issue_s = [&](uint32_t t) -> bool {  // S^T(t) = K Q(t)^T into buffer t & 1
                const uint32_t st = t % kStages, b = t & 1u;
                if (!mbar_wait(full + 8 * st, (t / kStages) & 1)) return false;
                if (t >= 2 && !mbar_wait(sempty + 8 * b, ((t >> 1) - 1) & 1)) return false;
                tc_fence_after();
                const uint32_t sQ = sStage + st * 2 * kTile;
#pragma unroll
                for (uint32_t ks = 0; ks < kHD / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalf + (ks & 3u) * 32;
                    tc_mma(tmem + b * kBlk, umma_desc_sw128(sK + off), umma_desc_sw128(sQ + off), idesc, ks ? 1u : 0u);
                }
                tc_commit(sfull + 8 * b);
                return true;
            };
            if (!mbar_wait(kfull, 0)) ok = false;
            if (ok && nq > 0) ok = issue_s(0);
            for (uint32_t t = 0; t < nq && ok; ++t) {
                if (t + 1 < nq && !issue_s(t + 1)) {
                    ok = false;
                    break;
                }
                const uint32_t st = t % kStages, b = t & 1u;
                if (!mbar_wait(pfull + 8 * b, (t >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sDo = sStage + st * 2 * kTile + kTile, sPb = sP + b * kTile;
#pragma unroll
                for (uint32_t ks = 0; ks < kBlk / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalf + (ks & 3u) * 32;
                    tc_mma(tmem + 2 * kBlk, umma_desc_sw128(sPb + off), umma_desc_sw128(sDo + off), idesc,
                           (t | ks) != 0 ? 1u : 0u);
                }
                tc_commit(pempty + 8 * b);   // P^T buffer b is free once these MMAs have read it
                tc_commit(empty + 8 * st);   // and so is the stage (its Q was read by the S MMA before)
            }
            tc_commit(dvfull);  // tracks every MMA issued: the epilogue and the TMEM owner wait on it
            if (!ok) atomicOr(err, 1);
        }
    } else {  // ------------------------------------------------------- softmax + epilogue
        const uint32_t quarter = warp & 3u;
        const uint32_t j = quarter * 32 + lane;  // this thread's key within the block (its TMEM lane)
        const uint32_t lane_base = (quarter * 32) << 16;
        // row j of a 128-byte swizzled [128 x 128] tile: 16-byte chunk c (c = 0..15) at
        // block c / 8, chunk position (c % 8) ^ (j % 8)
        const uint32_t prow = (j >> 3) * 1024 + (j & 7u) * 128;
        for (uint32_t t = 0; t < nq; ++t) {
            const uint32_t st = t % kStages, b = t & 1u, qb = q_first + t;
            bool got = mbar_wait(sfull + 8 * b, (t >> 1) & 1);
            if (got && t >= 2) got = mbar_wait(pempty + 8 * b, ((t >> 1) - 1) & 1);
            if (__any_sync(0xffffffffu, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *ls = (const float *)(sm + kOffLse + st * kBlk * 4);
            const bool diag = causal && qb == kb;
            const uint32_t sPb = sP + b * kTile;
#pragma unroll 1
            for (uint32_t c4 = 0; c4 < 4; ++c4) {  // 32 queries at a time
                uint32_t r[32];
                tc_ld32(tmem + lane_base + b * kBlk + c4 * 32, r);
                tc_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (uint32_t q = 0; q < 32; q += 2) {
                    const uint32_t i0 = c4 * 32 + q;
                    float p0 = ex2(__fmaf_rn(__uint_as_float(r[q]), scale_log2, -ls[i0] * kLog2e));
                    float p1 = ex2(__fmaf_rn(__uint_as_float(r[q + 1]), scale_log2, -ls[i0 + 1] * kLog2e));
                    if (diag) {  // query i attends key j only when i >= j
                        p0 = i0 >= j ? p0 : 0.0f;
                        p1 = i0 + 1 >= j ? p1 : 0.0f;
                    }
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[q / 2]) : "f"(p1), "f"(p0));
                }
#pragma unroll
                for (uint32_t cc = 0; cc < 4; ++cc) {
                    const uint32_t c = c4 * 4 + cc;  // 16-byte chunk of the row: queries 8c .. 8c + 7
                    const uint32_t addr = sPb + (c >> 3) * kHalf + prow + (((c & 7u) ^ (j & 7u)) << 4);
                    st_shared_v4(addr, w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sempty + 8 * b);
                mbar_arrive(pfull + 8 * b);
            }
        }
        // ---- epilogue: dV row j to global as bf16, then dV's column sums
        const bool got = mbar_wait(dvfull, 0);
        if (__any_sync(0xffffffffu, !got)) ok = false;
        float *scratch = (float *)(sm + kOffStage);
        if (ok) {
            tc_fence_after();
            __nv_bfloat16 *drow = dV + ((uint64_t)row0 + kb * kBlk + j) * kHD;
#pragma unroll 1
            for (uint32_t c4 = 0; c4 < 4; ++c4) {
                uint32_t r[32];
                tc_ld32(tmem + lane_base + 2 * kBlk + c4 * 32, r);
                tc_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (uint32_t q = 0; q < 32; q += 2) {
                    scratch[j * kScratchPitch + c4 * 32 + q] = __uint_as_float(r[q]);
                    scratch[j * kScratchPitch + c4 * 32 + q + 1] = __uint_as_float(r[q + 1]);
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
                        : "=r"(w[q / 2])
                        : "f"(__uint_as_float(r[q + 1])), "f"(__uint_as_float(r[q])));
                }
                uint4 *d = (uint4 *)(drow + c4 * 32);
#pragma unroll
                for (uint32_t v = 0; v < 4; ++v) d[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
        }
        named_bar_sync(1, 128);
        const uint32_t c = tid - 64;  // this thread's column of dV
        float s = 0.0f, e = 0.0f;
        if (ok) {
            for (uint32_t jj = 0; jj < kBlk; ++jj) pair_add(s, e, scratch[jj * kScratchPitch + c]);
        }
        part_dv[((uint64_t)bh * nkb + kb) * kHD + c] = make_float2(s, e);
        if (!ok && lane == 0) atomicOr(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && !mbar_wait(dvfull, 0)) atomicOr(err, 1);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
    }
}

// dO^T and the column sums of dO and |dO| over one block of 128 rows: block
// (x, y) takes rows 128x .. 128x + 127 of head y.  The tile goes through
// shared memory (row-major, read back column-wise for the transpose and the
// sums); part_do[y][x][c] = {pair of sum_i dO[i, c], pair of sum_i |dO[i, c]|}.
__global__ void __launch_bounds__(256) attn_do_prep_kernel(const __nv_bfloat16 *__restrict__ dO, uint32_t L,
                                                           __nv_bfloat16 *__restrict__ dOT,
                                                           float4 *__restrict__ part_do) {
    __shared__ __align__(16) uint16_t tile[kBlk][kHD];
    const uint32_t qb = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const uint64_t row0 = (uint64_t)bh * L + (uint64_t)qb * kBlk;
    for (uint32_t v = tid; v < kBlk * kHD / 8; v += 256) {  // 16-byte vectors, row-major
        const uint32_t r = v / (kHD / 8), c8 = v % (kHD / 8);
        *(uint4 *)&tile[r][c8 * 8] = ld_stream(dO + (row0 + r) * kHD + c8 * 8);
    }
    __syncthreads();
    for (uint32_t v = tid; v < kHD * kBlk / 8; v += 256) {  // dO^T row d, queries 8 q8 .. 8 q8 + 7
        const uint32_t d = v % kHD, q8 = v / kHD;
        uint32_t w[4];
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k)
            w[k] = (uint32_t)tile[q8 * 8 + 2 * k][d] | ((uint32_t)tile[q8 * 8 + 2 * k + 1][d] << 16);
        *(uint4 *)(dOT + ((uint64_t)bh * kHD + d) * L + (uint64_t)qb * kBlk + q8 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const uint32_t c = tid & (kHD - 1);
    float s = 0.0f, e = 0.0f;
    if (tid < kHD) {
        for (uint32_t r = 0; r < kBlk; ++r) pair_add(s, e, __uint_as_float((uint32_t)tile[r][c] << 16));
        float2 *o = (float2 *)&part_do[((uint64_t)bh * gridDim.x + qb) * kHD + c];
        o[0] = make_float2(s, e);
    } else {
        for (uint32_t r = 0; r < kBlk; ++r) pair_add(s, e, fabsf(__uint_as_float((uint32_t)tile[r][c] << 16)));
        float2 *o = (float2 *)&part_do[((uint64_t)bh * gridDim.x + qb) * kHD + c];
        o[1] = make_float2(s, e);
    }
}

// Per (head, column): dV's column sum (block partials merged in order), dO's
// column sum and |dO|'s, the residual, the bound and the flag.
__global__ void attn_invariant_kernel(const float2 *__restrict__ part_dv, const float4 *__restrict__ part_do,
                                      uint32_t BH, uint32_t nb, uint32_t L, float tol_scale,
                                      double *__restrict__ colsum_dv, double *__restrict__ colsum_do,
                                      double *__restrict__ residual, double *__restrict__ bound,
                                      uint8_t *__restrict__ flag, sdc_abft_summary *__restrict__ summary) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BH * kHD) return;
    const uint32_t bh = i / kHD, c = i % kHD;
    float vs = 0.0f, vc = 0.0f, os = 0.0f, oc = 0.0f, as = 0.0f, ac = 0.0f;
    for (uint32_t b = 0; b < nb; ++b) {
        const float2 pv = part_dv[((uint64_t)bh * nb + b) * kHD + c];
        const float4 po = part_do[((uint64_t)bh * nb + b) * kHD + c];
        pair_merge(vs, vc, pv.x, pv.y);
        pair_merge(os, oc, po.x, po.y);
        pair_merge(as, ac, po.z, po.w);
    }
    const double dv = (double)vs + (double)vc, dsum = (double)os + (double)oc, dabs = (double)as + (double)ac;
    const double g = (double)L * 0x1p-22, rho = 1.0 + 0x1p-7;
    const double b = (0x1p-8 * rho + g * (1.0 + g) * rho + 0x1p-40) * dabs + 0x1p-100;
    const double d = dv - dsum;
    colsum_dv[i] = dv;
    colsum_do[i] = dsum;
    residual[i] = d;
    bound[i] = b;
    const uint8_t f = fabs(d) <= (double)tol_scale * b ? 0 : 1;  // NaN flags
    flag[i] = f;
    if (f) atomicAdd(&summary->n_flagged, 1u);
}

__global__ void attn_abort_kernel(const int *__restrict__ err, uint32_t *__restrict__ aborted) {
    *aborted = *err != 0 ? 1u : 0u;
}

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace: dO^T [BH][128][L] bf16 | dO partials [BH][L/128][128] float4 |
// dV partials [BH][L/128][128] float2 | abort word.
struct AttnWs {
    size_t dot, pdo, pdv, err, total;
};
AttnWs attn_ws(uint32_t BH, uint32_t L) {
    AttnWs w;
    const size_t nb = L / kBlk;
    w.dot = 0;
    w.pdo = round_up256((size_t)BH * kHD * L * 2);
    w.pdv = w.pdo + round_up256((size_t)BH * nb * kHD * sizeof(float4));
    w.err = w.pdv + round_up256((size_t)BH * nb * kHD * sizeof(float2));
    w.total = w.err + 256;
    return w;
}

}  // namespace

}  // namespace sdc

using namespace sdc;

extern "C" {

size_t sdc_attn_workspace_size(uint32_t BH, uint32_t L, uint32_t D) {
    if (D != kHD) return 0;
    return attn_ws(BH, L).total;
}

sdc_status sdc_attn_dv_check(const void *d_Q, const void *d_K, const void *d_dO, const float *d_lse, uint32_t BH,
                             uint32_t L, uint32_t D, float scale, uint32_t causal, float tol_scale, void *d_dV,
                             double *d_colsum_dv, double *d_colsum_do, double *d_residual, double *d_bound,
                             uint8_t *d_flag, sdc_abft_summary *d_summary, uint32_t *d_aborted, void *d_ws,
                             size_t ws_bytes, sdc_stream_t stream) {
    if (!d_Q || !d_K || !d_dO || !d_lse) return fail(SDC_ERR_NULL, "NULL input");
    if (D != kHD) return fail(SDC_ERR_BAD_ARG, "the head dimension D must be 128");
    if (BH == 0 || L == 0 || L % kBlk || (uint64_t)BH * L >= (1ull << 31) || (uint64_t)BH * kHD >= (1ull << 31))
        return fail(SDC_ERR_BAD_ARG, "L must be a positive multiple of 128 and BH * L below 2^31");
    if (!(scale > 0.0f) || !(scale < 3.0e38f)) return fail(SDC_ERR_BAD_ARG, "scale must be positive and finite");
    if (!(tol_scale > 0.0f)) return fail(SDC_ERR_BAD_ARG, "tol_scale must be positive");
    if (causal > 1) return fail(SDC_ERR_BAD_ARG, "causal must be 0 or 1");
    if (!d_dV || !d_colsum_dv || !d_colsum_do || !d_residual || !d_bound || !d_flag || !d_summary || !d_aborted)
        return fail(SDC_ERR_NULL, "NULL output");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const uint64_t tbytes = (uint64_t)BH * L * kHD * 2;
    sdc_status st = check_device_range(d_Q, tbytes, dev, "d_Q");
    if (st == SDC_OK) st = check_device_range(d_K, tbytes, dev, "d_K");
    if (st == SDC_OK) st = check_device_range(d_dO, tbytes, dev, "d_dO");
    if (st == SDC_OK) st = check_device_range(d_dV, tbytes, dev, "d_dV");
    if (st == SDC_OK) st = check_device_range(d_lse, (uint64_t)BH * L * 4, dev, "d_lse");
    if (st != SDC_OK) return st;
    if (((uint64_t)d_Q | (uint64_t)d_K | (uint64_t)d_dO | (uint64_t)d_dV | (uint64_t)d_lse) & 15u)
        return fail(SDC_ERR_BAD_POINTER, "Q, K, dO, dV and lse must be 16-byte aligned");
    if (!d_ws || ws_bytes < sdc_attn_workspace_size(BH, L, D))
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_attn_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    const AttnWs w = attn_ws(BH, L);
    __nv_bfloat16 *dOT = (__nv_bfloat16 *)((char *)d_ws + w.dot);
    float4 *pdo = (float4 *)((char *)d_ws + w.pdo);
    float2 *pdv = (float2 *)((char *)d_ws + w.pdv);
    int *err = (int *)((char *)d_ws + w.err);
    CUtensorMap mapQ, mapK, mapDoT;
    st = make_map_sw128(&mapQ, d_Q, (uint64_t)BH * L, kHD, kBlk);
    if (st == SDC_OK) st = make_map_sw128(&mapK, d_K, (uint64_t)BH * L, kHD, kBlk);
    if (st == SDC_OK) st = make_map_sw128(&mapDoT, dOT, (uint64_t)BH * kHD, L, kHD);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    e = cudaMemsetAsync(err, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_summary, 0, sizeof(sdc_abft_summary), s);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_dv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttnSmem);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_attn_dv_check setup");
    const uint32_t nb = L / kBlk;
    attn_do_prep_kernel<<<dim3(nb, BH), 256, 0, s>>>((const __nv_bfloat16 *)d_dO, L, dOT, pdo);
    attn_dv_kernel<<<dim3(nb, BH), kAttnThreads, kAttnSmem, s>>>(mapQ, mapK, mapDoT, d_lse, L, scale * kLog2e, causal,
                                                                (__nv_bfloat16 *)d_dV, pdv, err);
    attn_invariant_kernel<<<(BH * kHD + 255) / 256, 256, 0, s>>>(pdv, pdo, BH, nb, L, tol_scale, d_colsum_dv,
                                                                 d_colsum_do, d_residual, d_bound, d_flag, d_summary);
    attn_abort_kernel<<<1, 1, 0, s>>>(err, d_aborted);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_attn_dv_check launch");
}

}  // extern "C"
