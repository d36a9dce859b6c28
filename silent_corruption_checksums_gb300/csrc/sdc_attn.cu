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
// Per head (BH query heads of L tokens, head dimension 128, Q/dO bf16
// [BH][L][128], the forward's natural-log log-sum-exp float32 [BH][L]; K/dV
// bf16 [BH / group][L][128], query head h using K/V head h / group):
//   P_h[i, j] = exp(scale q_i . k_j - lse_i)          (0 for j > i when causal)
//   dV[j, :] = sum over the group's heads h and queries i of P_h[i, j] dO_h[i, :]
//                                                      (P rounded to bf16, fp32 accumulate)
//   invariant per K/V head and column c: sum_j dV_acc[j, c]  vs  sum_h sum_i dO_h[i, c]
//   (every row of every P_h sums to 1).  group = 1 is plain multi-head attention.
//
// Kernels:
//   attn_lse2_kernel -- -lse log2(e) of every (head, token), elementwise;
//   attn_dv_kernel -- persistent, one CTA per SM; a work item is one
//     (K/V head, 128-key block), taken from a counter heaviest first (causal:
//     key block 0 of every head first), its steps running over the query
//     blocks of each of the group's query heads in turn.  24 warps:
//     warp 0 lane 0: the work queue and the K, Q and lse copies -- claims
//       the next item, hands it to the other roles through a 4-slot ring,
//       copies its K tile into one of two K stages (so the next item's K
//       arrives while this one runs), then per 128-query step the Q tile and
//       the step's 128 log-sum-exps (times -log2(e)) into their rings;
//     warp 3 lane 0: the dO copies, per step into a ring of their own (one
//       copy thread per ring: a Q copy never waits behind a dO stage);
//     warp 1 lane 0: S^T = K Q^T (M = keys, N = queries, K = 128) into one of
//       two 128-column TMEM buffers;
//     warp 2 lane 0: dV += P^T dO (M = keys, N = 128, K = queries) into one of
//       two 128-column TMEM accumulators (alternate items), its A operand P^T
//       read from TMEM.  Two issuing threads: one thread's tcgen05.mma issue
//       rate, not the tensor pipe, bounds products with N = 128;
//     warps 4..7: epilogue -- while an item's products run, they sum the
//       columns of dO and |dO| over the item's share of each of the group's
//       query heads' rows (float32 pairs; the shares cover every row once:
//       query block kb without a mask, causal a share in proportion to the
//       item's steps); when the item's dV is complete, each
//       thread stores its key's row as bf16 and the warps sum dV's columns
//       (float32 pairs) through shared memory, while the next item's
//       products run;
//     warps 8..23: softmax -- each thread owns one key (a TMEM lane) and 32
//       of the step's queries (four warps per lane quarter), reads those 32
//       scores, forms exp2(s scale log2(e) - lse log2(e)) (masked when
//       causal), rounds to bf16 and writes them as its row of P^T over the
//       first 16 of the columns it read; the S^T buffer is reused once the
//       dV product has read that P^T.
//     Every ring stage is freed by its last reader; each wait that usually
//     finds its phase complete comes before the one that blocks.
//     The item that completes a head (its last key block to finish, in
//     whichever block) merges the head's partials in order and writes the
//     invariant per column: dV's and dO's column sums, the residual, the
//     bound and the flag; the last block to finish publishes the abort word.
// Every wait is bounded; a wait that gives up sets the call's abort flag and
// the block still drains its copies and MMAs (bounded) and frees its TMEM.
#include <type_traits>

#include "sdc_internal.cuh"
#include "sdc_tc.cuh"

namespace sdc {

namespace {

constexpr uint32_t kHD = 128;                    // head dimension
constexpr uint32_t kBlk = 128;                   // keys per work item, queries per step
constexpr uint32_t kTile = kBlk * kHD * 2;       // 32 KiB: a [128 x 128] bf16 tile = two 64-column swizzled blocks
constexpr uint32_t kHalf = kBlk * 128;           // 16 KiB: one 64-column block
constexpr uint32_t kKStages = 2;     // K tiles: the next item's loads while this item's S^T products read
constexpr uint32_t kQStages = 2;     // Q tiles: freed by the S^T product
constexpr uint32_t kDStages = 2;     // dO tiles: freed by the dV product
constexpr uint32_t kLStages = 8;     // log-sum-exps of a step (512 bytes): freed by the softmax
constexpr uint32_t kItemSlots = 4;   // work items handed from the TMA thread to the other roles
constexpr uint32_t kNoItem = 0xFFFFFFFFu;
// Warps: 0 the work queue and the K, Q and lse copies, 1 S^T issuer, 2 dV issuer, 3 the dO copies
// (two copy threads, so that neither ring's copies wait behind the other's), 4-7 epilogue (one per
// TMEM lane quarter), then the softmax: kQParts warps per lane quarter, kQPer of a step's queries each.
constexpr uint32_t kQParts = 4, kQPer = kBlk / kQParts;
constexpr uint32_t kEpiBase = 4, kEpiWarps = 4, kSoftBase = kEpiBase + kEpiWarps, kSoftWarps = 4 * kQParts;
// TMEM: kSBufs S^T buffers, then kDvBufs dV accumulators, 128 columns each.  More S^T buffers let the
// S^T product run further ahead of the chain S^T -> softmax -> dV that frees a buffer.
constexpr uint32_t kSBufs = 2, kDvBufs = 2;
static_assert((kSBufs + kDvBufs) * kBlk <= 512, "TMEM has 512 columns");
static_assert(kQPer % 32 == 0, "the softmax reads its scores 32 columns at a time");
constexpr uint32_t kAttnThreads = 32 * (kSoftBase + kSoftWarps);
constexpr uint32_t kItemReaders = 3 + kEpiWarps + kSoftWarps;  // issuers, dO copier, one per other warp
// Barriers (each ring indexed by a counter that runs across work items):
constexpr uint32_t kBarKF = 0, kBarKE = kBarKF + kKStages, kBarQF = kBarKE + kKStages, kBarQE = kBarQF + kQStages,
                   kBarDF = kBarQE + kQStages, kBarDE = kBarDF + kDStages, kBarLF = kBarDE + kDStages,
                   kBarLE = kBarLF + kLStages, kBarSF = kBarLE + kLStages, kBarPF = kBarSF + kSBufs,
                   kBarPE = kBarPF + kSBufs, kBarVF = kBarPE + kSBufs, kBarVE = kBarVF + kDvBufs, kBarIF = kBarVE + kDvBufs, kBarIE = kBarIF + kItemSlots,
                   kBarSD = kBarIE + kItemSlots, kBarMD = kBarSD + 1, kNumBars = kBarMD + 1;
// shared memory: K stages | Q stages | dO stages | lse stages | epilogue scratch (a padded 32 x 32
// float tile per epilogue warp) | column partials [4][128] float2 | item slots | barriers | TMEM slot
constexpr uint32_t kScrPitch = 33;
constexpr uint32_t kOffK = 0, kOffQ = kOffK + kKStages * kTile, kOffD = kOffQ + kQStages * kTile,
                   kOffLse = kOffD + kDStages * kTile, kOffScr = kOffLse + kLStages * kBlk * 4,
                   kOffCp = kOffScr + kEpiWarps * 32 * kScrPitch * 4, kOffItems = kOffCp + 4 * kHD * 8,
                   kOffFlag = kOffItems + 4 * kItemSlots, kOffBar = kOffFlag + 8, kOffSlot = kOffBar + 8 * kNumBars;
// TMEM columns: S^T buffers at 0 and 128 (fp32; the softmax overwrites the first 32 columns of each
// half with its P^T, bf16 pairs: the dV product's A operand), dV accumulators at 256 and 384
constexpr uint32_t kColS = 0, kColDv = kSBufs * kBlk;
constexpr uint32_t kAttnSmem = 1024 + kOffSlot + 16;
static_assert(kAttnSmem <= 232448, "shared memory per block");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kDoChain = 8;  // rows of dO's plain float32 chains before each is folded into a pair

// Programmatic dependent launch: the lse2 kernel lets the dV kernel launch at once, and the dV
// kernel's thread that copies -lse log2(e) waits for that grid to complete first; its other work
// (TMEM, barriers, the K and Q copies) overlaps the lse2 kernel.
// Without a dependent launch the wait returns at once.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// The invariant of K/V head kvh, column c, once every key block's partials are in part_dv and
// part_do: dV's column sum and dO's and |dO|'s (the blocks' partials merged in order), the
// residual, the bound and the flag.
struct AttnOut {
    double *colsum_dv, *colsum_do, *residual, *bound;
    uint8_t *flag;
    sdc_abft_summary *summary;
    uint32_t *aborted;
    float tol_scale;
};
__device__ void head_invariant(const float2 *part_dv, const float4 *part_do, uint32_t kvh, uint32_t c, uint32_t nb,
                               uint32_t group, uint32_t L, const AttnOut &o) {
    float vs = 0.0f, vc = 0.0f, os = 0.0f, oc = 0.0f, as = 0.0f, ac = 0.0f;
    // L2 reads: other blocks wrote these partials; block b's dO partial covers query block b of every
    // query head of the group
#pragma unroll 8
    for (uint32_t b = 0; b < nb; ++b) {
        const float2 pv = __ldcg(part_dv + ((uint64_t)kvh * nb + b) * kHD + c);
        const float4 po = __ldcg(part_do + ((uint64_t)kvh * nb + b) * kHD + c);
        pair_merge(vs, vc, pv.x, pv.y);
        pair_merge(os, oc, po.x, po.y);
        pair_merge(as, ac, po.z, po.w);
    }
    const double dv = (double)vs + (double)vc, dsum = (double)os + (double)oc, dabs = (double)as + (double)ac;
    // dV's accumulation runs over the group's group * L query rows.  Beyond the method's terms the
    // bound carries this kernel's own: the float32 pairs of both column sums (2^-40) and dO's plain
    // chains of at most 8 rows (below 8 2^-24 each, twice over: 16 2^-24), and it takes sum |dO| raised
    // by 8 2^-24, above the exact sum whatever the chains lost.
    const double g = (double)group * (double)L * 0x1p-22, rho = 1.0 + 0x1p-7;
    const double own = 0x1p-40 + 16.0 * 0x1p-24;
    const double bnd = (0x1p-8 * rho + g * (1.0 + g) * rho + own) * dabs * (1.0 + 8.0 * 0x1p-24) + 0x1p-100;
    const double d = dv - dsum;
    const uint32_t i = kvh * kHD + c;
    o.colsum_dv[i] = dv;
    o.colsum_do[i] = dsum;
    o.residual[i] = d;
    o.bound[i] = bnd;
    const uint8_t f = fabs(d) <= (double)o.tol_scale * bnd ? 0 : 1;  // NaN flags
    o.flag[i] = f;
    if (f) atomicAdd(&o.summary->n_flagged, 1u);
}

// Persistent: one CTA per SM takes (K/V head, key block) items from a counter, heaviest first (item
// w: key block w / n_kv of K/V head w % n_kv; when causal, key block kb meets nkb - kb query blocks
// of each of the group's query heads kvh * group .. kvh * group + group - 1, taken head by head).
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_dv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapDo, const float *__restrict__ lse2, uint32_t L,
                   uint32_t n_kv, uint32_t group, float scale_log2, uint32_t causal, __nv_bfloat16 *__restrict__ dV,
                   float2 *__restrict__ part_dv, float4 *__restrict__ part_do, const AttnOut out,
                   int *__restrict__ err, uint32_t *__restrict__ ctr, const __nv_bfloat16 *__restrict__ dO) {
    // ctr: [0] the work counter, [1] blocks finished, [3 + h] key blocks of head h finished
    uint32_t *next_item = ctr;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
    const uint32_t nkb = (L + kBlk - 1) / kBlk, n_items = n_kv * nkb;  // the last block may be partial
    const uint32_t base = smem_addr(smem), pad = ((base + 1023u) & ~1023u) - base;
    unsigned char *sm = smem + pad;
    const uint32_t s0 = base + pad;
    const uint32_t bar = s0 + kOffBar;
#define BAR(i) (bar + 8u * (i))
    volatile uint32_t *items = (volatile uint32_t *)(sm + kOffItems);
    uint32_t *tmem_slot = (uint32_t *)(sm + kOffSlot);

    if (warp == 1) {  // all 512 columns: S^T x 2, dV x 2
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(512u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (uint32_t i = 0; i < kKStages; ++i) {
            mbar_init(BAR(kBarKF + i), 1);
            mbar_init(BAR(kBarKE + i), 1);
        }
        for (uint32_t i = 0; i < kQStages; ++i) {
            mbar_init(BAR(kBarQF + i), 1);
            mbar_init(BAR(kBarQE + i), 1);
        }
        for (uint32_t i = 0; i < kDStages; ++i) {
            mbar_init(BAR(kBarDF + i), 1);
            mbar_init(BAR(kBarDE + i), 1);
        }
        for (uint32_t i = 0; i < kLStages; ++i) {
            mbar_init(BAR(kBarLF + i), 1);
            mbar_init(BAR(kBarLE + i), kSoftWarps);
        }
        for (uint32_t i = 0; i < kSBufs; ++i) {
            mbar_init(BAR(kBarSF + i), 1);
            mbar_init(BAR(kBarPF + i), kSoftWarps);
            mbar_init(BAR(kBarPE + i), 1);
        }
        for (uint32_t i = 0; i < kDvBufs; ++i) {
            mbar_init(BAR(kBarVF + i), 1);
            mbar_init(BAR(kBarVE + i), kEpiWarps);
        }
        for (uint32_t i = 0; i < kItemSlots; ++i) {
            mbar_init(BAR(kBarIF + i), 1);
            mbar_init(BAR(kBarIE + i), kItemReaders);
        }
        mbar_init(BAR(kBarSD), 1);
        mbar_init(BAR(kBarMD), 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------ work queue + TMA
            uint32_t nk = 0, tl = 0, tq = 0;  // K tiles and steps whose copies were issued
            bool lse2_done = false;           // the lse2 grid's -lse log2(e) is complete
            for (uint32_t i = 0; ok; ++i) {
                const uint32_t slot = i % kItemSlots;
                if (i >= kItemSlots && !mbar_wait(BAR(kBarIE + slot), ((i / kItemSlots) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint32_t w = atomicAdd(next_item, 1u);
                if (w >= n_items) w = kNoItem;
                items[slot] = w;
                mbar_arrive(BAR(kBarIF + slot));  // release: the readers see the slot after their wait
                if (w == kNoItem) break;
                const uint32_t kb = w / n_kv, kvh = w % n_kv, q_first = causal ? kb : 0u, nq = nkb - q_first;
                const uint32_t ks = i % kKStages, sK = s0 + kOffK + ks * kTile;
                if (i >= kKStages && !mbar_wait(BAR(kBarKE + ks), ((i / kKStages) - 1) & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(BAR(kBarKF + ks), kTile);
                tma_load_3d(sK, &mapK, 0, (int32_t)(kb * kBlk), (int32_t)kvh, BAR(kBarKF + ks));
                tma_load_3d(sK + kHalf, &mapK, 64, (int32_t)(kb * kBlk), (int32_t)kvh, BAR(kBarKF + ks));
                nk = i + 1;
                uint32_t qb = q_first, qh = kvh * group;  // the step's query block and query head
                for (uint32_t t = 0; t < group * nq; ++t, ++qb) {
                    if (qb == nkb) {  // the next query head of the group
                        qb = q_first;
                        ++qh;
                    }
                    const uint32_t g = tl;
                    const uint32_t ls = g % kLStages, qs = g % kQStages;
                    if (g >= kLStages && !mbar_wait(BAR(kBarLE + ls), ((g / kLStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (!lse2_done) {
                        grid_dep_wait();
                        lse2_done = true;
                    }
                    // the block's queries inside the sequence (a multiple of 4: 16-byte copies)
                    const uint32_t lbytes = (L - qb * kBlk < kBlk ? L - qb * kBlk : kBlk) * 4;
                    mbar_arrive_expect_tx(BAR(kBarLF + ls), lbytes);
                    bulk_g2s(s0 + kOffLse + ls * kBlk * 4, lse2 + (uint64_t)qh * L + qb * kBlk, lbytes,
                             BAR(kBarLF + ls));
                    tl = g + 1;
                    if (g >= kQStages && !mbar_wait(BAR(kBarQE + qs), ((g / kQStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sQ = s0 + kOffQ + qs * kTile;
                    mbar_arrive_expect_tx(BAR(kBarQF + qs), kTile);
                    tma_load_3d(sQ, &mapQ, 0, (int32_t)(qb * kBlk), (int32_t)qh, BAR(kBarQF + qs));
                    tma_load_3d(sQ + kHalf, &mapQ, 64, (int32_t)(qb * kBlk), (int32_t)qh, BAR(kBarQF + qs));
                    tq = g + 1;
                }
            }
            // Let no copy land after the block has left: wait (bounded) for the last ones issued.
            for (uint32_t j = nk > kKStages ? nk - kKStages : 0; j < nk; ++j)
                if (!mbar_wait(BAR(kBarKF + j % kKStages), (j / kKStages) & 1)) ok = false;
            for (uint32_t j = tl > kLStages ? tl - kLStages : 0; j < tl; ++j)
                if (!mbar_wait(BAR(kBarLF + j % kLStages), (j / kLStages) & 1)) ok = false;
            for (uint32_t j = tq > kQStages ? tq - kQStages : 0; j < tq; ++j)
                if (!mbar_wait(BAR(kBarQF + j % kQStages), (j / kQStages) & 1)) ok = false;
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 3) {
        if (lane == 0) {  // ------------------------------------------ dO copies
            uint32_t td = 0;  // steps whose dO copies were issued
            for (uint32_t i = 0; ok; ++i) {
                const uint32_t slot = i % kItemSlots;
                if (!mbar_wait(BAR(kBarIF + slot), (i / kItemSlots) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t w = items[slot];
                mbar_arrive(BAR(kBarIE + slot));
                if (w == kNoItem) break;
                const uint32_t kb = w / n_kv, kvh = w % n_kv, q_first = causal ? kb : 0u, nq = nkb - q_first;
                uint32_t qb = q_first, qh = kvh * group;
                for (uint32_t t = 0; t < group * nq; ++t, ++qb) {
                    if (qb == nkb) {
                        qb = q_first;
                        ++qh;
                    }
                    const uint32_t g = td, ds = g % kDStages, sDo = s0 + kOffD + ds * kTile;
                    if (g >= kDStages && !mbar_wait(BAR(kBarDE + ds), ((g / kDStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(BAR(kBarDF + ds), kTile);
                    // the step's 128 rows of dO, head dimensions 0-63 then 64-127: K rows of the
                    // MN-major B operand
                    tma_load_3d(sDo, &mapDo, 0, (int32_t)(qb * kBlk), (int32_t)qh, BAR(kBarDF + ds));
                    tma_load_3d(sDo + kHalf, &mapDo, 64, (int32_t)(qb * kBlk), (int32_t)qh, BAR(kBarDF + ds));
                    td = g + 1;
                }
            }
            for (uint32_t j = td > kDStages ? td - kDStages : 0; j < td; ++j)
                if (!mbar_wait(BAR(kBarDF + j % kDStages), (j / kDStages) & 1)) ok = false;
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ------------------------------------------ S^T issuer
            constexpr uint32_t idesc = umma_idesc(kBlk, kBlk);
            uint32_t g = 0;
            for (uint32_t i = 0; ok; ++i) {
                const uint32_t slot = i % kItemSlots;
                if (!mbar_wait(BAR(kBarIF + slot), (i / kItemSlots) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t w = items[slot];
                mbar_arrive(BAR(kBarIE + slot));
                if (w == kNoItem) break;
                const uint32_t kb = w / n_kv, nq = group * (nkb - (causal ? kb : 0u));
                const uint32_t ks = i % kKStages, sK = s0 + kOffK + ks * kTile;
                if (!mbar_wait(BAR(kBarKF + ks), (i / kKStages) & 1)) {
                    ok = false;
                    break;
                }
                for (uint32_t t = 0; t < nq; ++t, ++g) {  // S^T(g) = K Q(g)^T into buffer g % kSBufs
                    const uint32_t qs = g % kQStages, b = g % kSBufs;
                    // buffer b is free once dV(g - kSBufs) has read the P^T the softmax wrote over it
                    if (!mbar_wait(BAR(kBarQF + qs), (g / kQStages) & 1) ||
                        (g >= kSBufs && !mbar_wait(BAR(kBarPE + b), ((g / kSBufs) - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sQ = s0 + kOffQ + qs * kTile;
#pragma unroll
                    for (uint32_t k = 0; k < kHD / 16; ++k) {
                        const uint32_t off = (k >> 2) * kHalf + (k & 3u) * 32;
                        tc_mma(tmem + kColS + b * kBlk, umma_desc_sw128(sK + off), umma_desc_sw128(sQ + off), idesc,
                               k ? 1u : 0u);
                    }
                    tc_commit(BAR(kBarSF + b));
                    tc_commit(BAR(kBarQE + qs));
                }
                if (!ok) break;
                tc_commit(BAR(kBarKE + ks));  // the K stage is free once this item's products have read it
            }
            tc_commit(BAR(kBarSD));  // tracks every product this thread issued: the TMEM owner waits on it
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp == 2) {
        if (lane == 0) {  // ------------------------------------------ dV issuer
            constexpr uint32_t idesc = umma_idesc_bmn(kBlk, kHD);  // B = dO, MN-major
            uint32_t g = 0;
            for (uint32_t i = 0; ok; ++i) {
                const uint32_t slot = i % kItemSlots;
                if (!mbar_wait(BAR(kBarIF + slot), (i / kItemSlots) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t w = items[slot];
                mbar_arrive(BAR(kBarIE + slot));
                if (w == kNoItem) break;
                const uint32_t kb = w / n_kv, nq = group * (nkb - (causal ? kb : 0u)), db = i % kDvBufs;
                if (i >= kDvBufs && !mbar_wait(BAR(kBarVE + db), ((i / kDvBufs) - 1) & 1)) {  // its last reader
                    ok = false;
                    break;
                }
                for (uint32_t t = 0; t < nq; ++t, ++g) {
                    const uint32_t ds = g % kDStages, b = g % kSBufs;
                    if (!mbar_wait(BAR(kBarDF + ds), (g / kDStages) & 1) ||  // copied steps ahead: first
                        !mbar_wait(BAR(kBarPF + b), (g / kSBufs) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sDo = s0 + kOffD + ds * kTile;
#pragma unroll
                    for (uint32_t k = 0; k < kBlk / 16; ++k) {  // 16 queries = 8 TMEM columns of P^T
                        // queries 16k .. 16k + 15: softmax part 16k / kQPer wrote them at its first columns;
                        // their rows of dO start 16k rows (2 KB) into each 64-column half
                        const uint32_t pa = kColS + b * kBlk + (16 * k / kQPer) * kQPer + (16 * k % kQPer) / 2;
                        tc_mma_ts(tmem + kColDv + db * kBlk, tmem + pa, umma_desc_sw128_mn(sDo + k * 2048, kHalf),
                                  idesc, (t | k) != 0 ? 1u : 0u);
                    }
                    tc_commit(BAR(kBarPE + b));   // S^T buffer b free once these products have read its P^T
                    tc_commit(BAR(kBarDE + ds));  // and so is the dO stage
                }
                if (!ok) break;
                tc_commit(BAR(kBarVF + db));  // the item's dV is complete
            }
            tc_commit(BAR(kBarMD));
            if (!ok) atomicOr(err, 1);
        }
    } else if (warp < kSoftBase) {  // ------------------------------ epilogue
        const uint32_t quarter = warp & 3u, j = quarter * 32 + lane, lane_base = (quarter * 32) << 16;
        float *scr = (float *)(sm + kOffScr) + (warp - kEpiBase) * 32 * kScrPitch;
        float2 *cpart = (float2 *)(sm + kOffCp);  // [lane quarter][column]
        volatile uint32_t *last = (volatile uint32_t *)(sm + kOffFlag);
        const uint32_t et = tid - kEpiBase * 32, cp = et & (kHD / 2 - 1), half = et / (kHD / 2);
        static_assert(kEpiWarps * 32 == kHD, "the dO sums: one thread per column pair and half of the share");
        for (uint32_t i = 0;; ++i) {
            const uint32_t slot = i % kItemSlots;
            bool got = mbar_wait(BAR(kBarIF + slot), (i / kItemSlots) & 1);
            if (bar_any(2, 32 * kEpiWarps, !got)) {
                ok = false;
                break;
            }
            const uint32_t w = items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(kBarIE + slot));
            if (w == kNoItem) break;
            const uint32_t kb = w / n_kv, kvh = w % n_kv, db = i % kDvBufs;
            {  // dO's column sums over this item's share of the rows of each of the group's query heads,
               // while the item's products run.  The shares cover every row of a head once: without a
               // mask the item on the diagonal takes query block kb; causal, item kb takes rows in
               // proportion to its steps (nkb - kb), in units of whole chains, so that the short items
               // at the end of the schedule carry only a few rows.  Thread (column pair cp, half) sums
               // columns 2cp, 2cp + 1 over its half of the share: plain float32 chains of kDoChain rows
               // folded into packed float32 pairs; the halves meet through the scratch (free until the
               // dV epilogue below).
                uint32_t lo, hi;
                if (causal) {
                    const uint32_t steps = nkb * (nkb + 1) / 2;
                    const uint32_t unit = kDoChain * ((L + kDoChain * steps - 1) / (kDoChain * steps));
                    const uint32_t before = kb * nkb - kb * (kb - 1) / 2;  // steps of the items kb' < kb
                    lo = min(L, unit * before);
                    hi = min(L, unit * (before + nkb - kb));
                } else {
                    lo = kb * kBlk;
                    hi = min(L, lo + kBlk);
                }
                const uint32_t mid = lo + (hi - lo + 2 * kDoChain - 1) / (2 * kDoChain) * kDoChain;
                const uint32_t r0 = half ? min(mid, hi) : lo, r1 = half ? hi : min(mid, hi);
                uint64_t ds = 0ull, dc = 0ull, das = 0ull, dac = 0ull;
                for (uint32_t h = 0; h < group; ++h) {
                    const uint32_t *src = (const uint32_t *)(dO + (uint64_t)(kvh * group + h) * L * kHD) + cp;
                    for (uint32_t rc = r0; rc < r1; rc += kDoChain) {
                        uint32_t wv[kDoChain];
#pragma unroll
                        for (uint32_t u = 0; u < kDoChain; ++u) wv[u] = rc + u < r1 ? __ldg(src + (rc + u) * (kHD / 2)) : 0u;
                        uint64_t t = 0ull, ta = 0ull;
#pragma unroll
                        for (uint32_t u = 0; u < kDoChain; ++u) {
                            const uint32_t wa = wv[u] & 0x7FFF7FFFu;
                            t = f2_add(t, f2_pack_bits(wv[u] << 16, wv[u] & 0xFFFF0000u));
                            ta = f2_add(ta, f2_pack_bits(wa << 16, wa & 0xFFFF0000u));
                        }
                        pair2_add(ds, dc, t);
                        pair2_add(das, dac, ta);
                    }
                }
                ulonglong2 *xs = (ulonglong2 *)(sm + kOffScr);  // [column pair][2]
                if (half == 1) {
                    xs[cp * 2] = make_ulonglong2(ds, dc);
                    xs[cp * 2 + 1] = make_ulonglong2(das, dac);
                }
                named_bar_sync(2, 32 * kEpiWarps);
                if (half == 0) {
                    const ulonglong2 o = xs[cp * 2], oa = xs[cp * 2 + 1];
                    pair2_add(ds, dc, o.x);
                    dc = f2_add(dc, o.y);
                    pair2_add(das, dac, oa.x);
                    dac = f2_add(dac, oa.y);
                    float s0, s1, c0, c1, a0, a1, e0, e1;
                    f2_unpack(ds, s0, s1);
                    f2_unpack(dc, c0, c1);
                    f2_unpack(das, a0, a1);
                    f2_unpack(dac, e0, e1);
                    float4 *o4 = part_do + ((uint64_t)kvh * nkb + kb) * kHD + 2 * cp;
                    o4[0] = make_float4(s0, c0, a0, e0);
                    o4[1] = make_float4(s1, c1, a1, e1);
                }
                named_bar_sync(2, 32 * kEpiWarps);  // the scratch is read before the dV epilogue writes it
            }
            got = mbar_wait(BAR(kBarVF + db), (i / kDvBufs) & 1);
            if (bar_any(2, 32 * kEpiWarps, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            __nv_bfloat16 *drow = dV + ((uint64_t)kvh * L + kb * kBlk + j) * kHD;
#pragma unroll 1
            for (uint32_t cc = 0; cc < kHD / 32; ++cc) {
                uint32_t r[32];
                tc_ld32(tmem + lane_base + kColDv + db * kBlk + cc * 32, r);
                tc_wait_ld();
                uint4 *d = (uint4 *)(drow + cc * 32);
#pragma unroll
                for (uint32_t v = 0; v < 4; ++v) {
                    uint32_t p[4];
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)
                        asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
                            : "=r"(p[k])
                            : "f"(__uint_as_float(r[8 * v + 2 * k + 1])), "f"(__uint_as_float(r[8 * v + 2 * k])));
                    if (kb * kBlk + j < L) d[v] = make_uint4(p[0], p[1], p[2], p[3]);  // keys inside the sequence
                }
                // this warp's 32 rows of the chunk's 32 columns, summed in row order (float32 pair)
#pragma unroll
                for (uint32_t q = 0; q < 32; ++q) scr[lane * kScrPitch + q] = __uint_as_float(r[q]);
                __syncwarp();
                float s = 0.0f, e = 0.0f;
#pragma unroll 8
                for (uint32_t rr = 0; rr < 32; ++rr) pair_add(s, e, scr[rr * kScrPitch + lane]);
                cpart[quarter * kHD + cc * 32 + lane] = make_float2(s, e);
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(kBarVE + db));  // the accumulator may take its next item
            named_bar_sync(2, 32 * kEpiWarps);
            const uint32_t c = (warp - kEpiBase) * 32 + lane;  // one column per epilogue thread
            {  // the lane quarters' partials merged in order: the item's column sums of dV
                float2 a = cpart[c];
#pragma unroll
                for (uint32_t q = 1; q < 4; ++q) pair_merge(a.x, a.y, cpart[q * kHD + c].x, cpart[q * kHD + c].y);
                part_dv[((uint64_t)kvh * nkb + kb) * kHD + c] = a;
            }
            // the item that completes its head (the head's last key block to finish, in any block)
            // finishes the head's invariant
            __threadfence();
            named_bar_sync(2, 32 * kEpiWarps);
            if (c == 0) *last = atomicAdd(ctr + 3 + kvh, 1u) == nkb - 1 ? 1u : 0u;
            named_bar_sync(2, 32 * kEpiWarps);
            if (*last) {
                __threadfence();
                head_invariant(part_dv, part_do, kvh, c, nkb, group, L, out);
            }
        }
        if (!ok && lane == 0) atomicOr(err, 1);
    } else {  // ------------------------------------------------------- softmax
        const uint32_t quarter = warp & 3u;               // the TMEM lanes this warp may access
        const uint32_t qpart = (warp - kSoftBase) >> 2;   // which kQPer of a step's queries
        const uint32_t j = quarter * 32 + lane;           // this thread's key within the item (its TMEM lane)
        const uint32_t lane_base = (quarter * 32) << 16;
        const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
        uint32_t g = 0;
        for (uint32_t i = 0; ok; ++i) {
            const uint32_t slot = i % kItemSlots;
            const bool got_item = mbar_wait(BAR(kBarIF + slot), (i / kItemSlots) & 1);
            if (__any_sync(0xffffffffu, !got_item)) {
                ok = false;
                break;
            }
            const uint32_t w = items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(kBarIE + slot));
            if (w == kNoItem) break;
            const uint32_t kb = w / n_kv, q_first = causal ? kb : 0u, nq = nkb - q_first;
            const bool key_ok = kb * kBlk + j < L;  // this thread's key is inside the sequence
            uint32_t qb = q_first;
            for (uint32_t t = 0; t < group * nq; ++t, ++g, ++qb) {
                if (qb == nkb) qb = q_first;  // the next query head of the group
                const uint32_t ls = g % kLStages, b = g % kSBufs;
                // the step's log-sum-exps (copied steps ahead) first, then the scores: the wait that
                // blocks comes last, so nothing stands between the scores' arrival and their use
                bool got = mbar_wait(BAR(kBarLF + ls), (g / kLStages) & 1);
                if (got) got = mbar_wait(BAR(kBarSF + b), (g / kSBufs) & 1);
                if (__any_sync(0xffffffffu, !got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t lsa = s0 + kOffLse + ls * kBlk * 4 + qpart * kQPer * 4;  // -lse log2(e) of its queries
                // steps that need a mask: the causal diagonal block, a partial last query block, a key
                // past L (a partial last key block)
                const bool diag = causal && qb == kb;
                const bool edge = diag || qb * kBlk + kBlk > L || !key_ok;
                const uint32_t col = tmem + lane_base + kColS + b * kBlk + qpart * kQPer;
                uint32_t r[kQPer];
#pragma unroll
                for (uint32_t c = 0; c < kQPer / 32; ++c) tc_ld32(col + 32 * c, *(uint32_t(*)[32]) & r[32 * c]);
                tc_wait_ld();
                uint32_t pw[kQPer / 2];  // this thread's probabilities as bf16 pairs
                uint32_t mbits = ~0u;    // with a mask: bit q for query qpart * kQPer + q
                // two copies of the loop, the masked one only for the steps that need it (a mask tested
                // inside a single loop costs every step)
                auto probs = [&](auto masked) {
#pragma unroll
                    for (uint32_t q8 = 0; q8 < kQPer / 8; ++q8) {  // 8 queries at a time
                        const float4 la = ld_shared_f4(lsa + q8 * 32), lb = ld_shared_f4(lsa + q8 * 32 + 16);
                        const float l8[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
#pragma unroll
                        for (uint32_t q = 0; q < 8; q += 2) {
                            // both exponents in one packed FMA (each lane rounded as a scalar fma.rn)
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack_bits(r[q8 * 8 + q], r[q8 * 8 + q + 1]), scale2,
                                             f2_pack(l8[q], l8[q + 1])),
                                      x0, x1);
                            float p0 = ex2(x0);
                            float p1 = ex2(x1);
                            if constexpr (decltype(masked)::value) {  // selected, not multiplied: a masked
                                p0 = (mbits >> (q8 * 8 + q)) & 1u ? p0 : 0.0f;       // score may be anything
                                p1 = (mbits >> (q8 * 8 + q + 1)) & 1u ? p1 : 0.0f;
                            }
                            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pw[q8 * 4 + q / 2]) : "f"(p1), "f"(p0));
                        }
                    }
                };
                if (edge) {
                    // bit q: this thread's query qpart * kQPer + q attends its key (on the diagonal, query
                    // i >= key j; queries past L, and a key past L, take no probability)
                    const uint32_t qbase = qpart * kQPer;
                    mbits = ~0u;
                    if (diag && j > qbase) mbits = j - qbase >= 32 ? 0u : ~0u << (j - qbase);
                    const uint32_t q_lim = key_ok ? (L - qb * kBlk < kBlk ? L - qb * kBlk : kBlk) : 0u;
                    if (q_lim < qbase + 32) mbits &= (1u << (q_lim > qbase ? q_lim - qbase : 0u)) - 1u;
                    probs(std::true_type{});
                } else {
                    probs(std::false_type{});
                }
                // P^T over the first kQPer / 2 of the columns just read (this thread's own lane and columns)
#pragma unroll
                for (uint32_t c = 0; c < kQPer / 32; ++c) tc_st16(col + 16 * c, *(const uint32_t(*)[16]) & pw[16 * c]);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(BAR(kBarPF + b));
                    mbar_arrive(BAR(kBarLE + ls));
                }
            }
        }
        if (!ok && lane == 0) atomicOr(err, 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && (!mbar_wait(BAR(kBarMD), 0) || !mbar_wait(BAR(kBarSD), 0))) atomicOr(err, 1);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
    }
    __syncthreads();
    if (tid == 0) {  // the last block to finish publishes whether any wait gave up
        __threadfence();
        if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
            __threadfence();
            *out.aborted = atomicOr(err, 0) != 0 ? 1u : 0u;
        }
    }
#undef BAR
}

// -lse log2(e) of every (head, token): the exponent's offset in base 2, negated, which the softmax
// adds (one float32 product per value, four values per thread and step).  The dV kernel is launched as
// its programmatic dependent: its set-up and its K and Q copies overlap this grid.  Block 0 also zeroes
// the call's summary, which the dV kernel touches only after it has waited for this grid.
__global__ void __launch_bounds__(256) attn_lse2_kernel(const float4 *__restrict__ lse, uint32_t n4,
                                                        float4 *__restrict__ lse2, uint32_t *__restrict__ zero,
                                                        uint32_t n_zero) {
    if (blockIdx.x == 0)
        for (uint32_t z = threadIdx.x; z < n_zero; z += blockDim.x) zero[z] = 0u;
    grid_dep_launch();  // the dV kernel may start its set-up now
    for (uint32_t i = blockIdx.x * 256 + threadIdx.x; i < n4; i += gridDim.x * 256) {
        const float4 v = lse[i];
        lse2[i] = make_float4(v.x * -kLog2e, v.y * -kLog2e, v.z * -kLog2e, v.w * -kLog2e);
    }
}

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace: dO partials [BH][L/128][128] float4 |
// dV partials [BH][L/128][128] float2 | -lse log2(e) [BH][L] float | the abort word, the dV
// kernel's work counter, its count of finished blocks (one word of padding) and of finished
// key blocks per head [BH].
struct AttnWs {
    size_t pdo, pdv, lse2, err, total;
};
AttnWs attn_ws(uint32_t BH, uint32_t L) {
    AttnWs w;
    const size_t nb = (L + kBlk - 1) / kBlk;
    w.pdo = 0;
    w.pdv = w.pdo + round_up256((size_t)BH * nb * kHD * sizeof(float4));
    w.lse2 = w.pdv + round_up256((size_t)BH * nb * kHD * sizeof(float2));
    w.err = w.lse2 + round_up256((size_t)BH * L * sizeof(float));
    w.total = w.err + round_up256(16 + (size_t)BH * 4);
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

sdc_status sdc_attn_dv_check_grouped(const void *d_Q, const void *d_K, const void *d_dO, const float *d_lse,
                                     uint32_t BH, uint32_t group, uint32_t L, uint32_t D, float scale, uint32_t causal,
                                     float tol_scale, void *d_dV, double *d_colsum_dv, double *d_colsum_do,
                                     double *d_residual, double *d_bound, uint8_t *d_flag, sdc_abft_summary *d_summary,
                                     uint32_t *d_aborted, void *d_ws, size_t ws_bytes, sdc_stream_t stream) {
    if (!d_Q || !d_K || !d_dO || !d_lse) return fail(SDC_ERR_NULL, "NULL input");
    if (D != kHD) return fail(SDC_ERR_BAD_ARG, "the head dimension D must be 128");
    if (BH == 0 || L == 0 || L % 4 || (uint64_t)BH * L >= (1ull << 31) || (uint64_t)BH * kHD >= (1ull << 31))
        return fail(SDC_ERR_BAD_ARG, "L must be a positive multiple of 4 and BH * L below 2^31");
    if (group == 0 || BH % group) return fail(SDC_ERR_BAD_ARG, "group must divide BH");
    const uint32_t n_kv = BH / group;  // K/V heads
    // one work item's steps (group x key blocks) stay well inside a bounded wait (the epilogue waits
    // for a whole item): 2^19 steps take under a second even on a throttled GPU
    if ((uint64_t)group * ((L + kBlk - 1) / kBlk) > (1ull << 19))
        return fail(SDC_ERR_BAD_ARG, "group * ceil(L / 128) must not exceed 2^19");
    if (!(scale > 0.0f) || !(scale < 3.0e38f)) return fail(SDC_ERR_BAD_ARG, "scale must be positive and finite");
    if (!(tol_scale > 0.0f)) return fail(SDC_ERR_BAD_ARG, "tol_scale must be positive");
    if (causal > 1) return fail(SDC_ERR_BAD_ARG, "causal must be 0 or 1");
    if (!d_dV || !d_colsum_dv || !d_colsum_do || !d_residual || !d_bound || !d_flag || !d_summary || !d_aborted)
        return fail(SDC_ERR_NULL, "NULL output");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const uint64_t tbytes = (uint64_t)BH * L * kHD * 2, kvbytes = (uint64_t)n_kv * L * kHD * 2;
    sdc_status st = check_device_range(d_Q, tbytes, dev, "d_Q");
    if (st == SDC_OK) st = check_device_range(d_K, kvbytes, dev, "d_K");
    if (st == SDC_OK) st = check_device_range(d_dO, tbytes, dev, "d_dO");
    if (st == SDC_OK) st = check_device_range(d_dV, kvbytes, dev, "d_dV");
    if (st == SDC_OK) st = check_device_range(d_lse, (uint64_t)BH * L * 4, dev, "d_lse");
    if (st == SDC_OK)
        st = check_spans({{d_colsum_dv, (uint64_t)n_kv * kHD * 8, "d_colsum_dv"},
                          {d_colsum_do, (uint64_t)n_kv * kHD * 8, "d_colsum_do"},
                          {d_residual, (uint64_t)n_kv * kHD * 8, "d_residual"},
                          {d_bound, (uint64_t)n_kv * kHD * 8, "d_bound"},
                          {d_flag, (uint64_t)n_kv * kHD, "d_flag"},
                          {d_summary, sizeof(sdc_abft_summary), "d_summary"},
                          {d_aborted, 4, "d_aborted"}},
                         dev);
    if (st != SDC_OK) return st;
    if (((uint64_t)d_Q | (uint64_t)d_K | (uint64_t)d_dO | (uint64_t)d_dV | (uint64_t)d_lse) & 15u)
        return fail(SDC_ERR_BAD_POINTER, "Q, K, dO, dV and lse must be 16-byte aligned");
    if (!d_ws || ws_bytes < sdc_attn_workspace_size(BH, L, D))
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_attn_workspace_size");
    if ((uint64_t)d_ws & 255u) return fail(SDC_ERR_BAD_POINTER, "workspace is not 256-byte aligned");
    st = check_device_range(d_ws, sdc_attn_workspace_size(BH, L, D), dev, "d_ws");
    if (st != SDC_OK) return st;
    const AttnWs w = attn_ws(BH, L);
    float4 *pdo = (float4 *)((char *)d_ws + w.pdo);
    float2 *pdv = (float2 *)((char *)d_ws + w.pdv);
    float *lse2 = (float *)((char *)d_ws + w.lse2);
    int *err = (int *)((char *)d_ws + w.err);
    CUtensorMap mapQ, mapK, mapDo;
    // one plane per head: a partial last block reads zeros past L, never the next head's rows
    st = make_map_sw128_3d(&mapQ, d_Q, BH, L, kHD, kBlk);
    if (st == SDC_OK) st = make_map_sw128_3d(&mapK, d_K, n_kv, L, kHD, kBlk);
    if (st == SDC_OK) st = make_map_sw128_3d(&mapDo, d_dO, BH, L, kHD, kBlk);
    if (st != SDC_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t *ctr = (uint32_t *)(err + 1);  // the counters after the abort word
    int n_sm = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    const uint32_t n_items = n_kv * ((L + kBlk - 1) / kBlk);
    const uint32_t grid = n_items < (uint32_t)n_sm ? n_items : (uint32_t)n_sm;
    // the abort word and the counters (the work counter is taken before the dV kernel waits for the
    // lse2 grid); the summary is zeroed by the lse2 grid
    e = cudaMemsetAsync(err, 0, 16 + (size_t)BH * 4, s);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_dv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttnSmem);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_attn_dv_check setup");
    const AttnOut out{d_colsum_dv, d_colsum_do, d_residual, d_bound, d_flag, d_summary, d_aborted, tol_scale};
    const uint32_t n4 = BH * L / 4;  // L is a multiple of 4
    const uint32_t lse_grid = (n4 + 255) / 256 < 4u * (uint32_t)n_sm ? (n4 + 255) / 256 : 4u * (uint32_t)n_sm;
    attn_lse2_kernel<<<lse_grid, 256, 0, s>>>((const float4 *)d_lse, n4, (float4 *)lse2, (uint32_t *)d_summary,
                                              (uint32_t)(sizeof(sdc_abft_summary) / 4));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = kAttnSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before lse2 is complete
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_dv_kernel, mapQ, mapK, mapDo, (const float *)lse2, L, n_kv, group,
                           scale * kLog2e, causal, (__nv_bfloat16 *)d_dV, pdv, pdo, out, err, ctr,
                           (const __nv_bfloat16 *)d_dO);
    if (e != cudaSuccess) return cuda_fail(e, "sdc_attn_dv_check launch");
    e = cudaGetLastError();
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_attn_dv_check launch");
}

sdc_status sdc_attn_dv_check(const void *d_Q, const void *d_K, const void *d_dO, const float *d_lse, uint32_t BH,
                             uint32_t L, uint32_t D, float scale, uint32_t causal, float tol_scale, void *d_dV,
                             double *d_colsum_dv, double *d_colsum_do, double *d_residual, double *d_bound,
                             uint8_t *d_flag, sdc_abft_summary *d_summary, uint32_t *d_aborted, void *d_ws,
                             size_t ws_bytes, sdc_stream_t stream) {
    return sdc_attn_dv_check_grouped(d_Q, d_K, d_dO, d_lse, BH, 1, L, D, scale, causal, tol_scale, d_dV, d_colsum_dv,
                                     d_colsum_do, d_residual, d_bound, d_flag, d_summary, d_aborted, d_ws, ws_bytes,
                                     stream);
}

}  // extern "C"
