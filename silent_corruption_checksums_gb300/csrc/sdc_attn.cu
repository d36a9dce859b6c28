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
//     then sit K-major in shared memory), lse log2(e), and float32-pair column
//     sums of dO and |dO| per 128-row block;
//   attn_dv_kernel -- one CTA per (head, 128-key block), 19 warps:
//     warp 0 lane 0: TMA -- the K tile once, then per 128-query step the Q
//       tile into one of two Q stages, freed when the S MMAs have read it, and
//       the dO^T tile with the step's 128 log-sum-exps (times log2(e)) into one
//       of two dO stages, freed when the dV MMAs have read it;
//     warp 1 lane 0: S^T = K Q^T (M = keys, N = queries, K = 128) into one of
//       two 128-column TMEM buffers, as soon as a Q tile and a buffer are free;
//     warp 2 lane 0: dV += P^T dO (M = keys, N = 128, K = queries) into a
//       third.  Two issuing threads: one thread's tcgen05.mma issue rate, not
//       the tensor pipe, bounds products with N = 128, and the two products
//       share no TMEM, meeting only at barriers;
//     warps 3..18: softmax -- two groups of 8 warps take alternate steps; in
//       a group each thread owns one key (a TMEM lane) and 64 of the step's
//       queries (two warps per lane quarter), reads those 64 scores,
//       forms exp2(s scale log2(e) - lse log2(e)) (masked when causal), rounds
//       to bf16 and writes them into its row of P^T in one of two TMEM
//       buffers, from which the dV product takes its A operand; at the end it reads its 32 columns of
//       dV's row, stores them as bf16, and the threads sum dV's columns
//       (float32 pairs) through shared memory;
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
constexpr uint32_t kQStages = 2;     // Q tiles: freed by the S product
constexpr uint32_t kDStages = 3;     // dO^T tiles: freed by the dV product
constexpr uint32_t kLStages = 16;    // log-sum-exps of a step (512 bytes): freed by the softmax
// Two groups of 8 softmax warps take alternate query steps (group g: steps g, g + 2, ...; S^T and
// P^T buffer g), so one group's latency chain overlaps the other's; in a group, two warps per TMEM
// lane quarter each take 64 of the step's 128 queries.
constexpr uint32_t kSoftWarps = 16;
constexpr uint32_t kGroupWarps = kSoftWarps / 2;
constexpr uint32_t kSoftBase = 3;  // warps 0-2: TMA, S^T issuer, dV issuer
constexpr uint32_t kAttnThreads = 32 * kSoftBase + 32 * kSoftWarps;
// Barriers: kfull, qfull/qempty[kQStages], dfull/dempty[kDStages], lfull/lempty[kLStages],
// sfull/sempty[2], pfull/pempty[2], dvfull, sdone.  Each input has its own ring and is freed by its last
// reader, so every copy is issued steps before it is needed and no chain of a step waits on a copy.
constexpr uint32_t kBarK = 0, kBarQF = 1, kBarQE = kBarQF + kQStages, kBarDF = kBarQE + kQStages,
                   kBarDE = kBarDF + kDStages, kBarLF = kBarDE + kDStages, kBarLE = kBarLF + kLStages,
                   kBarSF = kBarLE + kLStages, kBarSE = kBarSF + 2, kBarPF = kBarSE + 2, kBarPE = kBarPF + 2,
                   kBarDV = kBarPE + 2, kBarSD = kBarDV + 1, kNumBars = kBarSD + 1;
// shared memory: K tile | Q stages | dO^T stages | lse stages | barriers | TMEM slot
constexpr uint32_t kOffK = 0, kOffQ = kTile, kOffD = kOffQ + kQStages * kTile, kOffLse = kOffD + kDStages * kTile,
                   kOffBar = kOffLse + kLStages * kBlk * 4, kOffSlot = kOffBar + 8 * kNumBars;
// TMEM columns: S^T buffers at 0 and 128 (fp32), dV at 256 (fp32), P^T buffers at 384 and 448
// (bf16, two per 32-bit column: the A operand of the dV product)
constexpr uint32_t kColS = 0, kColDv = 256, kColP = 384;
constexpr uint32_t kAttnSmem = 1024 + kOffSlot + 16;
constexpr uint32_t kScratchPitch = kHD + 1;  // float row pitch of the column-sum scratch (conflict-free both ways)
static_assert(kBlk * kScratchPitch * 4 <= (kQStages + kDStages) * kTile, "column-sum scratch must fit in the stages");
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_dv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapDoT, const float *__restrict__ lse2, uint32_t L,
                   float scale_log2, uint32_t causal, __nv_bfloat16 *__restrict__ dV, float2 *__restrict__ part_dv,
                   int *__restrict__ err) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    // grid (heads, key blocks): blocks start in linear order, so every head's key block 0 (the
    // most query steps when causal) starts first and the light blocks fill the tail
    const uint32_t bh = blockIdx.x, kb = blockIdx.y, nkb = gridDim.y;
    const uint32_t base = smem_addr(smem), pad = ((base + 1023u) & ~1023u) - base;
    unsigned char *sm = smem + pad;
    const uint32_t s0 = base + pad;
    const uint32_t sK = s0 + kOffK, sQ0 = s0 + kOffQ, sD0 = s0 + kOffD, sLse = s0 + kOffLse;
    const uint32_t bar = s0 + kOffBar;
    const uint32_t kfull = bar + 8 * kBarK, qfull = bar + 8 * kBarQF, qempty = bar + 8 * kBarQE,
                   dfull = bar + 8 * kBarDF, dempty = bar + 8 * kBarDE, lfull = bar + 8 * kBarLF,
                   lempty = bar + 8 * kBarLE, sfull = bar + 8 * kBarSF, sempty = bar + 8 * kBarSE,
                   pfull = bar + 8 * kBarPF, pempty = bar + 8 * kBarPE, dvfull = bar + 8 * kBarDV,
                   sdone = bar + 8 * kBarSD;
    uint32_t *tmem_slot = (uint32_t *)(sm + kOffSlot);
    const uint32_t q_first = causal ? kb : 0u, nq = nkb - q_first;
    const uint32_t row0 = bh * L;  // this head's first row in the [BH * L, 128] views

    if (warp == 1) {  // all 512 columns: S^T x 2, dV, P^T x 2
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(512u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(kfull, 1);
        for (uint32_t i = 0; i < kQStages; ++i) {
            mbar_init(qfull + 8 * i, 1);
            mbar_init(qempty + 8 * i, 1);
        }
        for (uint32_t i = 0; i < kDStages; ++i) {
            mbar_init(dfull + 8 * i, 1);
            mbar_init(dempty + 8 * i, 1);
        }
        for (uint32_t i = 0; i < kLStages; ++i) {
            mbar_init(lfull + 8 * i, 1);
            mbar_init(lempty + 8 * i, kGroupWarps);  // stage i serves steps of one parity: one group
        }
        for (uint32_t i = 0; i < 2; ++i) {
            mbar_init(sfull + 8 * i, 1);
            mbar_init(sempty + 8 * i, kGroupWarps);  // one arrival per warp of softmax group i
            mbar_init(pfull + 8 * i, kGroupWarps);
            mbar_init(pempty + 8 * i, 1);
        }
        mbar_init(dvfull, 1);
        mbar_init(sdone, 1);
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
            uint32_t tl = 0, tq = 0, td = 0;  // steps whose lse / Q / dO^T copies were issued
            for (uint32_t t = 0; t < nq && ok; ++t) {
                const uint32_t qb = q_first + t;
                const uint32_t ls = t % kLStages, qs = t % kQStages, ds = t % kDStages;
                if (t >= kLStages && !mbar_wait(lempty + 8 * ls, ((t / kLStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(lfull + 8 * ls, kBlk * 4);
                bulk_g2s(sLse + ls * kBlk * 4, lse2 + (uint64_t)row0 + qb * kBlk, kBlk * 4, lfull + 8 * ls);
                tl = t + 1;
                if (t >= kQStages && !mbar_wait(qempty + 8 * qs, ((t / kQStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t sQ = sQ0 + qs * kTile, sDo = sD0 + ds * kTile;
                mbar_arrive_expect_tx(qfull + 8 * qs, kTile);
                tma_load_2d(sQ, &mapQ, 0, (int32_t)(row0 + qb * kBlk), qfull + 8 * qs);
                tma_load_2d(sQ + kHalf, &mapQ, 64, (int32_t)(row0 + qb * kBlk), qfull + 8 * qs);
                tq = t + 1;
                if (t >= kDStages && !mbar_wait(dempty + 8 * ds, ((t / kDStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(dfull + 8 * ds, kTile);
                tma_load_2d(sDo, &mapDoT, (int32_t)(qb * kBlk), (int32_t)(bh * kHD), dfull + 8 * ds);
                tma_load_2d(sDo + kHalf, &mapDoT, (int32_t)(qb * kBlk + 64), (int32_t)(bh * kHD), dfull + 8 * ds);
                td = t + 1;
            }
            // Let no copy land after the block has left: wait (bounded) for the last ones issued.
            if (!mbar_wait(kfull, 0)) ok = false;
            for (uint32_t j = tl > kLStages ? tl - kLStages : 0; j < tl; ++j)
                if (!mbar_wait(lfull + 8 * (j % kLStages), (j / kLStages) & 1)) ok = false;
            for (uint32_t j = tq > kQStages ? tq - kQStages : 0; j < tq; ++j)
                if (!mbar_wait(qfull + 8 * (j % kQStages), (j / kQStages) & 1)) ok = false;
            for (uint32_t j = td > kDStages ? td - kDStages : 0; j < td; ++j)
                if (!mbar_wait(dfull + 8 * (j % kDStages), (j / kDStages) & 1)) ok = false;
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ------------------------------------------ S^T issuer
            constexpr uint32_t idesc = umma_idesc(kBlk, kBlk);
            if (!mbar_wait(kfull, 0)) ok = false;
            for (uint32_t t = 0; t < nq && ok; ++t) {  // S^T(t) = K Q(t)^T into buffer t & 1
                const uint32_t qs = t % kQStages, b = t & 1u;
                if (!mbar_wait(qfull + 8 * qs, (t / kQStages) & 1) ||
                    (t >= 2 && !mbar_wait(sempty + 8 * b, ((t >> 1) - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sQ = sQ0 + qs * kTile;
#pragma unroll
                for (uint32_t ks = 0; ks < kHD / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * kHalf + (ks & 3u) * 32;
                    tc_mma(tmem + kColS + b * kBlk, umma_desc_sw128(sK + off), umma_desc_sw128(sQ + off), idesc,
                           ks ? 1u : 0u);
                }
                tc_commit(sfull + 8 * b);
                tc_commit(qempty + 8 * qs);
            }
            tc_commit(sdone);  // tracks every S^T product this thread issued: the TMEM owner waits on it
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 2) {
        if (lane == 0) {  // ------------------------------------------ dV issuer
            constexpr uint32_t idesc = umma_idesc(kBlk, kBlk);
            for (uint32_t t = 0; t < nq && ok; ++t) {
                const uint32_t ds = t % kDStages, b = t & 1u;
                if (!mbar_wait(pfull + 8 * b, (t >> 1) & 1) || !mbar_wait(dfull + 8 * ds, (t / kDStages) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sDo = sD0 + ds * kTile;
#pragma unroll
                for (uint32_t ks = 0; ks < kBlk / 16; ++ks) {  // 16 queries = 8 TMEM columns of P^T
                    const uint32_t off = (ks >> 2) * kHalf + (ks & 3u) * 32;
                    tc_mma_ts(tmem + kColDv, tmem + kColP + b * 64 + ks * 8, umma_desc_sw128(sDo + off), idesc,
                              (t | ks) != 0 ? 1u : 0u);
                }
                tc_commit(pempty + 8 * b);   // P^T buffer b (TMEM) is free once these MMAs have read it
                tc_commit(dempty + 8 * ds);  // and so is the dO^T stage
            }
            tc_commit(dvfull);  // tracks every dV product: the epilogue and the TMEM owner wait on it
            if (!ok) atomicOr(err, 1);
        }
    } else {  // ------------------------------------------------------- softmax + epilogue
        const uint32_t quarter = warp & 3u;       // the TMEM lanes this warp may read
        const uint32_t part = (warp - kSoftBase) >> 2;     // which 32 of dV's columns in the epilogue
        const uint32_t grp = (warp - kSoftBase) / kGroupWarps;        // softmax group: steps grp, grp + 2, ...
        const uint32_t half = ((warp - kSoftBase) % kGroupWarps) >> 2;  // which 64 of a step's queries
        const uint32_t j = quarter * 32 + lane;  // this thread's key within the block (its TMEM lane)
        const uint32_t lane_base = (quarter * 32) << 16;
        for (uint32_t t = grp; t < nq; t += 2) {
            const uint32_t ls = t % kLStages, b = t & 1u, qb = q_first + t;
            bool got = mbar_wait(sfull + 8 * b, (t >> 1) & 1);
            if (got) got = mbar_wait(lfull + 8 * ls, (t / kLStages) & 1);  // the step's log-sum-exps
            if (got && t >= 2) got = mbar_wait(pempty + 8 * b, ((t >> 1) - 1) & 1);
            if (__any_sync(0xffffffffu, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t lsa = sLse + ls * kBlk * 4 + half * 64 * 4;  // lse log2(e) of this half's 64 queries
            const bool diag = causal && qb == kb;
            uint32_t r[64];
            tc_ld32(tmem + lane_base + kColS + b * kBlk + half * 64, *(uint32_t(*)[32]) & r[0]);
            tc_ld32(tmem + lane_base + kColS + b * kBlk + half * 64 + 32, *(uint32_t(*)[32]) & r[32]);
            tc_wait_ld();
            uint32_t w[32];  // this thread's 64 probabilities as bf16 pairs: 32 columns of its row of P^T
#pragma unroll
            for (uint32_t g = 0; g < 8; ++g) {  // 8 queries at a time
                const float4 la = ld_shared_f4(lsa + g * 32), lb = ld_shared_f4(lsa + g * 32 + 16);
                const float l8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
#pragma unroll
                for (uint32_t q = 0; q < 8; q += 2) {
                    const uint32_t i0 = half * 64 + g * 8 + q;  // query within the step
                    float p0 = ex2(__fmaf_rn(__uint_as_float(r[g * 8 + q]), scale_log2, -l8[q]));
                    float p1 = ex2(__fmaf_rn(__uint_as_float(r[g * 8 + q + 1]), scale_log2, -l8[q + 1]));
                    if (diag) {  // query i attends key j only when i >= j
                        p0 = i0 >= j ? p0 : 0.0f;
                        p1 = i0 + 1 >= j ? p1 : 0.0f;
                    }
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[g * 4 + q / 2]) : "f"(p1), "f"(p0));
                }
            }
            tc_st16(tmem + lane_base + kColP + b * 64 + half * 32, *(const uint32_t(*)[16]) & w[0]);
            tc_st16(tmem + lane_base + kColP + b * 64 + half * 32 + 16, *(const uint32_t(*)[16]) & w[16]);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(sempty + 8 * b);
                mbar_arrive(pfull + 8 * b);
                mbar_arrive(lempty + 8 * ls);
            }
        }
        // ---- epilogue: dV row j to global as bf16, then dV's column sums
        const bool got = mbar_wait(dvfull, 0);
        if (__any_sync(0xffffffffu, !got)) ok = false;
        float *scratch = (float *)(sm + kOffQ);
        if (ok) {
            tc_fence_after();
            __nv_bfloat16 *drow = dV + ((uint64_t)row0 + kb * kBlk + j) * kHD;
            uint32_t r[32];
            tc_ld32(tmem + lane_base + kColDv + part * 32, r);
            tc_wait_ld();
            float *srow = scratch + j * kScratchPitch + part * 32;
#pragma unroll
            for (uint32_t q = 0; q < 32; ++q) srow[q] = __uint_as_float(r[q]);
            uint4 *d = (uint4 *)(drow + part * 32);
#pragma unroll
            for (uint32_t v = 0; v < 4; ++v) {
                uint32_t w[4];
#pragma unroll
                for (uint32_t k = 0; k < 4; ++k)
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
                        : "=r"(w[k])
                        : "f"(__uint_as_float(r[8 * v + 2 * k + 1])), "f"(__uint_as_float(r[8 * v + 2 * k])));
                d[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        named_bar_sync(1, 32 * kSoftWarps);
        // dV's column sums: thread (column c, row quarter rq) sums rows 32 rq .. 32 rq + 31, then
        // the rq = 0 thread merges the others' pairs in order rq = 1, 2, 3
        const uint32_t c = (tid - 32 * kSoftBase) & (kHD - 1), rq = (tid - 32 * kSoftBase) >> 7;
        float s = 0.0f, e = 0.0f;
        if (ok) {
#pragma unroll 8
            for (uint32_t jj = rq * 32; jj < rq * 32 + 32; ++jj) pair_add(s, e, scratch[jj * kScratchPitch + c]);
        }
        named_bar_sync(1, 32 * kSoftWarps);  // every thread has read the scratch: reuse its first rows
        if (rq != 0) {
            scratch[(rq * kHD + c) * 2] = s;
            scratch[(rq * kHD + c) * 2 + 1] = e;
        }
        named_bar_sync(1, 32 * kSoftWarps);
        if (rq == 0) {
            for (uint32_t k = 1; k < 4; ++k) pair_merge(s, e, scratch[(k * kHD + c) * 2], scratch[(k * kHD + c) * 2 + 1]);
            part_dv[((uint64_t)bh * nkb + kb) * kHD + c] = make_float2(s, e);
        }
        if (!ok && lane == 0) atomicOr(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && (!mbar_wait(dvfull, 0) || !mbar_wait(sdone, 0))) atomicOr(err, 1);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
    }
}

// dO^T, lse log2(e), and the column sums of dO and |dO| over one block of 128 rows: block
// (x, y) takes rows 128x .. 128x + 127 of head y.  The tile goes through
// shared memory (row-major, read back column-wise for the transpose and the
// sums); part_do[y][x][c] = {pair of sum_i dO[i, c], pair of sum_i |dO[i, c]|}.
__global__ void __launch_bounds__(256) attn_do_prep_kernel(const __nv_bfloat16 *__restrict__ dO,
                                                           const float *__restrict__ lse, uint32_t L,
                                                           __nv_bfloat16 *__restrict__ dOT, float4 *__restrict__ part_do,
                                                           float *__restrict__ lse2) {
    __shared__ __align__(16) uint16_t tile[kBlk][kHD];
    const uint32_t qb = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const uint64_t row0 = (uint64_t)bh * L + (uint64_t)qb * kBlk;
    if (tid < kBlk) lse2[row0 + tid] = lse[row0 + tid] * kLog2e;  // the exponent's offset in base 2
    for (uint32_t v = tid; v < kBlk * kHD / 8; v += 256) {  // 16-byte vectors, row-major
        const uint32_t r = v / (kHD / 8), c8 = v % (kHD / 8);
        *(uint4 *)&tile[r][c8 * 8] = ld_stream(dO + (row0 + r) * kHD + c8 * 8);
    }
    __syncthreads();
    for (uint32_t v = tid; v < kHD * kBlk / 16; v += 256) {  // dO^T row d, queries 16 q16 .. 16 q16 + 15
        const uint32_t d = v % kHD, q16 = v / kHD;
        uint32_t w[8];
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k)
            w[k] = (uint32_t)tile[q16 * 16 + 2 * k][d] | ((uint32_t)tile[q16 * 16 + 2 * k + 1][d] << 16);
        uint4 *o = (uint4 *)(dOT + ((uint64_t)bh * kHD + d) * L + (uint64_t)qb * kBlk + q16 * 16);  // one 32-byte sector
        o[0] = make_uint4(w[0], w[1], w[2], w[3]);
        o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    // column sums: thread (column c, row half h) sums rows 64h .. 64h + 63 of dO and |dO|
    // (two independent chains); the half-1 pairs are merged into the half-0 ones in that order
    __shared__ float4 half1[kHD];
    const uint32_t c = tid & (kHD - 1), h = tid >> 7;
    float s = 0.0f, e = 0.0f, sa = 0.0f, ea = 0.0f;
#pragma unroll 8
    for (uint32_t r = h * 64; r < h * 64 + 64; ++r) {
        const float x = __uint_as_float((uint32_t)tile[r][c] << 16);
        pair_add(s, e, x);
        pair_add(sa, ea, fabsf(x));
    }
    if (h == 1) half1[c] = make_float4(s, e, sa, ea);
    __syncthreads();
    if (h == 0) {
        const float4 o = half1[c];
        pair_merge(s, e, o.x, o.y);
        pair_merge(sa, ea, o.z, o.w);
        part_do[((uint64_t)bh * gridDim.x + qb) * kHD + c] = make_float4(s, e, sa, ea);
    }
}

// Per (head, column): dV's column sum (block partials merged in order), dO's
// column sum and |dO|'s, the residual, the bound and the flag.
__global__ void attn_invariant_kernel(const float2 *__restrict__ part_dv, const float4 *__restrict__ part_do,
                                      uint32_t BH, uint32_t nb, uint32_t L, float tol_scale,
                                      double *__restrict__ colsum_dv, double *__restrict__ colsum_do,
                                      double *__restrict__ residual, double *__restrict__ bound,
                                      uint8_t *__restrict__ flag, sdc_abft_summary *__restrict__ summary,
                                      const int *__restrict__ err, uint32_t *__restrict__ aborted) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *aborted = *err != 0 ? 1u : 0u;
    if (i >= BH * kHD) return;
    const uint32_t bh = i / kHD, c = i % kHD;
    float vs = 0.0f, vc = 0.0f, os = 0.0f, oc = 0.0f, as = 0.0f, ac = 0.0f;
#pragma unroll 8
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

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace: dO^T [BH][128][L] bf16 | dO partials [BH][L/128][128] float4 |
// dV partials [BH][L/128][128] float2 | lse log2(e) [BH][L] float | abort word.
struct AttnWs {
    size_t dot, pdo, pdv, lse2, err, total;
};
AttnWs attn_ws(uint32_t BH, uint32_t L) {
    AttnWs w;
    const size_t nb = L / kBlk;
    w.dot = 0;
    w.pdo = round_up256((size_t)BH * kHD * L * 2);
    w.pdv = w.pdo + round_up256((size_t)BH * nb * kHD * sizeof(float4));
    w.lse2 = w.pdv + round_up256((size_t)BH * nb * kHD * sizeof(float2));
    w.err = w.lse2 + round_up256((size_t)BH * L * sizeof(float));
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
    float *lse2 = (float *)((char *)d_ws + w.lse2);
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
    attn_do_prep_kernel<<<dim3(nb, BH), 256, 0, s>>>((const __nv_bfloat16 *)d_dO, d_lse, L, dOT, pdo, lse2);
    attn_dv_kernel<<<dim3(BH, nb), kAttnThreads, kAttnSmem, s>>>(mapQ, mapK, mapDoT, lse2, L, scale * kLog2e, causal,
                                                                (__nv_bfloat16 *)d_dV, pdv, err);
    attn_invariant_kernel<<<(BH * kHD + 127) / 128, 128, 0, s>>>(pdv, pdo, BH, nb, L, tol_scale, d_colsum_dv,
                                                                 d_colsum_do, d_residual, d_bound, d_flag, d_summary,
                                                                 err, d_aborted);
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_attn_dv_check launch");
}

}  // extern "C"
