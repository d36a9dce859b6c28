// sdc_grad.cu -- non-finite gradient scan with the squared L2 norm, and the
// fused average-and-scan pass.
//
// Method: "Detecting and recovering from silent data corruption on Amazon
// SageMaker HyperPod", "Check 1: NaN/Inf gradients, before and after the
// all-reduce" (a rank is flagged when its local gradient norm is NaN or Inf,
// and the reduced gradient is checked before the update) and "Decide what the
// alarm means" (a float32 norm above about 1.8e19 counts as non-finite).
//
// Per element: NaN / Inf / finite; a finite x is "big" when x^2 > FLT_MAX.
// The squared norm sums x^2 over finite elements in float64 precision.
//
// Why not a float64 add per element: this part's FP64 rate is a small
// fraction of its FP32 rate, far below what a bf16 stream at HBM speed needs.
// Every lane instead adds squares in float32 and captures each add's rounding
// error exactly, on packed f32x2 pairs:
//  - bf16 and f16 (the "offset runs" below): each square is a float32, added
//    with one fused multiply-add whose rounding error a second one recovers,
//    the run's sum started at a power-of-two offset so that Sterbenz's lemma
//    makes every step exact (checked after the run; a run that fails the
//    check is redone).  Error below 3.8e-11 of each run's sum.
//  - f32: x^2 = p + e exactly with p = fl(x*x), e = fma(x, x, -p), provided
//    the biased exponent of x is >= 76 (or x == 0; smaller values are caught
//    by a running minimum of the lane's magnitudes); p is added with Dekker's
//    Fast2Sum on the ordered pair.  The error of such a sum of n terms is
//    below gamma_{n-1}^2 * sum, gamma_k = k u / (1 - k u), u = 2^-24 (Ogita,
//    Rump and Oishi, "Accurate sum and dot product", 2005); with n = 64 terms
//    per lane half between flushes that is 1.4e-11 relative.
// Each run is added into the lane's own float32 pair (h, l) with TwoSum, and
// a warp's lanes are added in a fixed xor tree of TwoSums; float64 is used
// only for the warp's total, or for each lane's pair if the float32 tree
// overflows.
// A run whose float32 sum is not finite (NaN, Inf, big, an overflowing sum)
// or that holds a tiny f32 value is redone exactly: each element classified
// and its square added in float64 (exact squares).
// All reductions have a fixed shape, so results are identical on every run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sdc_internal.cuh"

namespace sdc {

namespace {

constexpr int kRunVec = 16;           // vectors per lane between flushes
constexpr double kFltMax = 3.4028234663852886e38;
constexpr uint32_t kF32TinyLimit = (76u << 24) - 2u;  // (bits << 1) - 2 below this: tiny, non-zero

// ---------------------------------------------------------------- exact element path
__device__ __forceinline__ float to_float(uint32_t bits, uint32_t dt) {
    if (dt == SDC_DTYPE_F32) return __uint_as_float(bits);
    if (dt == SDC_DTYPE_BF16) return __uint_as_float(bits << 16);
    return __half2float(__ushort_as_half((unsigned short)bits));
}

struct Counts {
    uint32_t nan = 0, inf = 0, big = 0;
};

__device__ __forceinline__ void exact_elem(uint32_t bits, uint32_t dt, double &acc, Counts &n) {
    const float f = to_float(bits, dt);
    if (isnan(f)) {
        n.nan++;
    } else if (isinf(f)) {
        n.inf++;
    } else {
        const double x = f;
        const double x2 = __dmul_rn(x, x);  // exact: <= 48 significant bits
        if (x2 > kFltMax) n.big++;
        acc = __dadd_rn(acc, x2);
    }
}

template <int DT>
__device__ __forceinline__ void exact_vec(const uint4 &v, double &acc, Counts &n) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (DT == SDC_DTYPE_F32) {
            exact_elem(w[k], DT, acc, n);
        } else {
            exact_elem(w[k] & 0xFFFFu, DT, acc, n);
            exact_elem(w[k] >> 16, DT, acc, n);
        }
    }
}

// ---------------------------------------------------------------- fast path
struct FastAcc {
    uint64_t s = 0, c = 0;  // packed f32x2 sum and compensation
    uint32_t tmin = 0xFFFFFFFFu;
};

// The f32 fast path (bf16 and f16 take the offset runs below).
__device__ __forceinline__ void fast_vec_f32(const uint4 &v, FastAcc &a) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
        const uint64_t p = f2_pack_bits(w[j], w[j + 1]);
        const uint64_t sq = f2_mul(p, p);
        const uint64_t e = f2_fma(p, p, sq ^ 0x8000000080000000ull);  // x*x - fl(x*x), exact
        f2_two_sum_acc(a.s, a.c, sq);
        a.c = f2_add(a.c, e);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) a.tmin = min(a.tmin, w[j] * 2u - 2u);
}

// A lane's runs summed as a float32 pair h + l.
struct FF {
    float h = 0.0f, l = 0.0f;
};

// Adds a finished run into f: the two packed halves merged error-free, then
// TwoSum with f.h.  Returns false, leaving f unchanged, when the run must be
// redone exactly: a half not finite, a tiny f32 value, or a sum that overflows.
template <int DT>
__device__ __forceinline__ bool fast_flush_ff(FastAcc &a, FF &f) {
    float sx, sy, cx, cy;
    f2_unpack(a.s, sx, sy);
    f2_unpack(a.c, cx, cy);
    bool ok = isfinite(sx) && isfinite(sy);
    if (DT == SDC_DTYPE_F32) ok = ok && a.tmin >= kF32TinyLimit;
    if (ok) {
        const float t = sx + sy;
        const float bb = t - sx;
        const float e = (sx - (t - bb)) + (sy - bb);
        const float h2 = f.h + t;  // Inf when t or the new sum overflows
        const float b2 = h2 - f.h;
        const float e2 = (f.h - (h2 - b2)) + (t - b2);
        ok = isfinite(h2);
        if (ok) {
            f.h = h2;
            f.l = __fadd_rn(f.l, __fadd_rn(__fadd_rn(__fadd_rn(cx, cy), e), e2));
        }
    }
    a.s = 0;
    a.c = 0;
    a.tmin = 0xFFFFFFFFu;
    return ok;
}

// The warp's total: the lanes' pairs added in a fixed xor tree (TwoSum's
// error term is exact whichever operand comes first, so every lane ends with
// the same bits); if that overflows float32, each lane's pair in float64
// instead.  Then plus the exactly summed elements (acc_e).
template <int DT>
__device__ __forceinline__ double warp_total(const FF &f, double acc_e) {
    float h = f.h, l = f.l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ho = __shfl_xor_sync(0xffffffffu, h, o), lo = __shfl_xor_sync(0xffffffffu, l, o);
        const float t = __fadd_rn(h, ho);
        const float bb = __fsub_rn(t, h);
        const float e = __fadd_rn(__fsub_rn(h, __fsub_rn(t, bb)), __fsub_rn(ho, bb));
        h = t;
        l = __fadd_rn(__fadd_rn(l, lo), e);
    }
    double tot;
    if (isfinite(h))  // the same on every lane
        tot = __dadd_rn((double)h, (double)l);
    else
        tot = warp_sum_f64(__dadd_rn((double)f.h, (double)f.l));
    if (__any_sync(0xffffffffu, acc_e != 0.0)) tot = __dadd_rn(tot, warp_sum_f64(acc_e));
    return tot;
}

// ---------------------------------------------------------------- 16-bit path: offset runs
// For bf16 and f16 each square x^2 is a float32 (8- and 11-bit significands
// square to at most 22 bits) unless it leaves the float32 range, so a lane can
// add it with one fused multiply-add and recover the rounding error of that
// add exactly, without ordering the operands:
//   s' = fl(s + x^2) = fma(x, x, s),   d = s - s',   e = fma(x, x, d) = s + x^2 - s'.
// d is exact by Sterbenz's lemma whenever s <= s' <= 2s, which holds when
// x^2 <= s; then d + x^2 is the exact rounding error, a float32, so the second
// fma returns it exactly.  To make x^2 <= s hold for every term, a run of
// kRun16 vectors per lane (64 terms per packed half) starts its sum at an
// offset sigma, the power of two at or above 2.5 times the previous run's sum;
// the run is accepted only when, afterwards,
//   (1) s_final <= 1.96875 sigma: then the run's true sum is below sigma (the
//       rounding errors of s are below 2^-24 s each), so every term was below
//       the running sum, every d and e above were exact, and s_final - sigma is
//       exact (Sterbenz again);
//   (2) sigma <= 16 (s_final - sigma): the errors e are at most 2^-24 sigma
//       each (s stays inside one binade), and each vector's four are added
//       pairwise before their sum joins c, so c is off by at most
//       16 * 8 + 4 * 135 = 668 units of 2^-48 sigma: below 3.8e-11 of the run's sum;
//   (3) sigma >= 2^-100: a bf16 square below 2^-126 is not a float32, and
//       the second fma then rounds e by at most 2^-150, negligible against a
//       run sum of at least 2^-104.
// A packed half with sigma == 0 is accepted only when a pass over the run has
// seen every one of its elements be +-0 (a square below 2^-149 rounds to 0,
// so s == 0 alone does not show that the sum is 0).
// A run that fails is redone from its vectors with sigma from its own sum
// estimate (which then satisfies (1) and (2)), and if that fails too (NaN,
// Inf, a square or sum past FLT_MAX, a tiny sum) element by element exactly.
// Accepted runs are added into the lane's float32 pair (h, l) with TwoSum.
constexpr int kRun16 = 16;

struct SAcc {
    uint64_t s, c;  // packed running sum (starting at sigma) and error sum
};

// A lane's accepted runs, packed halves: h + l.
struct FF2 {
    uint64_t h = 0, l = 0;
};

template <int DT>
__device__ __forceinline__ uint64_t widen16(uint32_t w) {
    if constexpr (DT == SDC_DTYPE_BF16) {
        return f2_pack_bits(w << 16, w & 0xFFFF0000u);
    } else {
        return f2_pack(__half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))),
                       __half2float(__ushort_as_half((unsigned short)(w >> 16))));
    }
}

template <int DT>
__device__ __forceinline__ void sacc_vec(const uint4 &v, SAcc &a) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint64_t e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t x = widen16<DT>(w[j]);
        const uint64_t s1 = f2_fma(x, x, a.s);  // fl(s + x^2)
        const uint64_t d = f2_sub(a.s, s1);     // exact while x^2 <= s
        e[j] = f2_fma(x, x, d);                 // s + x^2 - s1, exact
        a.s = s1;
    }
    a.c = f2_add(a.c, f2_add(f2_add(e[0], e[1]), f2_add(e[2], e[3])));
}

// The offset for the run after one whose sum is about est: the power of two
// at or above 2.5 est (0 when est is not a positive finite value).
__device__ __forceinline__ float sigma_from(float est) {
    const float y = 2.5f * est;
    if (!(y > 0.0f) || !isfinite(y)) return 0.0f;
    return __uint_as_float((__float_as_uint(y) + 0x007FFFFFu) & 0xFF800000u);
}
__device__ __forceinline__ uint64_t sigma_next(uint64_t est) {
    float e0, e1;
    f2_unpack(est, e0, e1);
    return f2_pack(sigma_from(e0), sigma_from(e1));
}

// zero: every element of the half is known to be +-0 (then sigma is 0 too).
__device__ __forceinline__ bool sigma_half_ok(float s, float g, float q, bool zero) {
    return (g >= 0x1p-100f && s <= 1.96875f * g && g <= 16.0f * q) || (zero && g == 0.0f);
}

// Checks conditions (1)-(3) on both halves and, when they hold, adds the run
// into f.  est receives the run's sum estimate (s - sigma + c) either way.
// zero0 / zero1: the low / high half's elements are all known to be +-0.
__device__ __forceinline__ bool sacc_accept(const SAcc &a, uint64_t sig, FF2 &f, uint64_t &est, bool zero0 = false,
                                            bool zero1 = false) {
    const uint64_t q = f2_sub(a.s, sig);  // exact when (1) holds
    est = f2_add(q, a.c);
    float s0, s1, g0, g1, q0, q1;
    f2_unpack(a.s, s0, s1);
    f2_unpack(sig, g0, g1);
    f2_unpack(q, q0, q1);
    if (!(sigma_half_ok(s0, g0, q0, zero0) && sigma_half_ok(s1, g1, q1, zero1))) return false;
    const uint64_t t = f2_add(f.h, q);  // TwoSum(h, q)
    const uint64_t bb = f2_sub(t, f.h);
    const uint64_t err = f2_add(f2_sub(f.h, f2_sub(t, bb)), f2_sub(q, bb));
    float t0, t1;
    f2_unpack(t, t0, t1);
    if (!(isfinite(t0) && isfinite(t1))) return false;
    f.h = t;
    f.l = f2_add(f.l, f2_add(a.c, err));
    return true;
}

// A failed run again from its vectors (lane + 32 i for i in [r0, r1), below
// nvec) with the offset sig.
template <int DT>
__device__ __forceinline__ bool sacc_redo(const uint4 *src, uint32_t lane, uint32_t r0, uint32_t r1, uint32_t nvec,
                                          uint64_t sig, FF2 &f) {
    SAcc b{sig, 0ull};
    uint32_t mag = 0;  // OR of the magnitude bits of both halves' elements
    for (uint32_t i = r0; i < r1; ++i) {
        const uint32_t vi = lane + (i << 5);
        if (vi < nvec) {
            const uint4 v = src[vi];
            sacc_vec<DT>(v, b);
            mag |= v.x | v.y | v.z | v.w;
        }
    }
    mag &= 0x7FFF7FFFu;
    uint64_t est;
    return sacc_accept(b, sig, f, est, (mag & 0xFFFFu) == 0, (mag >> 16) == 0);
}

// A run that the offset check refused, out of line (rare; keeping it out of
// the scan loops keeps their code small): redone with the offset sig, else
// element by element exactly into acc / cnt (the nan, inf and big counts at
// cnt[0], cnt[stride], cnt[2 stride]).  Returns the lane's updated pair.
template <int DT>
__device__ __noinline__ FF2 run_fallback(const uint4 *src, uint32_t lane, uint32_t r0, uint32_t r1, uint32_t nvec,
                                         uint64_t sig, FF2 f, double *acc, uint32_t *cnt, uint32_t stride) {
    if (sacc_redo<DT>(src, lane, r0, r1, nvec, sig, f)) return f;
    double a = *acc;
    Counts n;
    n.nan = cnt[0];
    n.inf = cnt[stride];
    n.big = cnt[2 * stride];
    for (uint32_t i = r0; i < r1; ++i) {
        const uint32_t vi = lane + (i << 5);
        if (vi < nvec) exact_vec<DT>(src[vi], a, n);
    }
    *acc = a;
    cnt[0] = n.nan;
    cnt[stride] = n.inf;
    cnt[2 * stride] = n.big;
    return f;
}

// The warp's total from the lanes' packed pairs: each lane's halves merged
// with TwoSum, then the same fixed xor tree as warp_total (float64 per lane if
// the float32 sums overflow), plus the exactly summed elements acc_e.
__device__ __forceinline__ double warp_total2(const FF2 &f, double acc_e) {
    float h0, h1, l0, l1;
    f2_unpack(f.h, h0, h1);
    f2_unpack(f.l, l0, l1);
    const float t = __fadd_rn(h0, h1);
    const float bb = __fsub_rn(t, h0);
    const float e = __fadd_rn(__fsub_rn(h0, __fsub_rn(t, bb)), __fsub_rn(h1, bb));
    float h = t, l = __fadd_rn(__fadd_rn(l0, l1), e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ho = __shfl_xor_sync(0xffffffffu, h, o), lo = __shfl_xor_sync(0xffffffffu, l, o);
        const float t2 = __fadd_rn(h, ho);
        const float b2 = __fsub_rn(t2, h);
        const float e2 = __fadd_rn(__fsub_rn(h, __fsub_rn(t2, b2)), __fsub_rn(ho, b2));
        h = t2;
        l = __fadd_rn(__fadd_rn(l, lo), e2);
    }
    double tot;
    if (isfinite(h))  // the same on every lane
        tot = __dadd_rn((double)h, (double)l);
    else
        tot = warp_sum_f64(__dadd_rn(__dadd_rn((double)h0, (double)h1), __dadd_rn((double)l0, (double)l1)));
    if (__any_sync(0xffffffffu, acc_e != 0.0)) tot = __dadd_rn(tot, warp_sum_f64(acc_e));
    return tot;
}

// ---------------------------------------------------------------- plan-based scan
// Chunk geometry (mirrors the fingerprint pass).
struct GGeom {
    uint64_t addr;
    uint32_t head, nvec, tail, l2;
};
__device__ __forceinline__ GGeom ggeom(const Chunk &ch) {
    GGeom g;
    g.addr = ch.addr;
    g.l2 = chunk_log2es(ch.tag);
    uint32_t head = (uint32_t)((16u - (uint32_t)(ch.addr & 15u)) & 15u);
    if (head > ch.nbytes) head = ch.nbytes;
    g.head = head;
    g.nvec = (ch.nbytes - head) >> 4;
    g.tail = ch.nbytes - head - (g.nvec << 4);
    return g;
}

// A chunk's head and tail elements (fewer than 8 of each, outside its
// 16-byte vectors), exactly: lanes 0..7 the head, lanes 16..23 the tail.
template <int DT>
__device__ __forceinline__ void grad_head_tail(const GGeom &g, uint32_t lane, double &acc_exact, Counts &n) {
    const uint32_t he = g.head >> g.l2, te = g.tail >> g.l2;
    if (lane < he) {
        const uint64_t a = g.addr + ((uint64_t)lane << g.l2);
        const uint32_t bits = g.l2 == 2 ? *(const uint32_t *)a : (uint32_t)(*(const uint16_t *)a);
        exact_elem(bits, DT, acc_exact, n);
    } else if (lane >= 16 && lane - 16 < te) {
        const uint64_t a = g.addr + g.head + ((uint64_t)g.nvec << 4) + ((uint64_t)(lane - 16) << g.l2);
        const uint32_t bits = g.l2 == 2 ? *(const uint32_t *)a : (uint32_t)(*(const uint16_t *)a);
        exact_elem(bits, DT, acc_exact, n);
    }
}

template <int DT, int U>
__device__ __forceinline__ double grad_chunk(const GGeom &g, uint32_t lane, Counts &n) {
    static_assert(DT == SDC_DTYPE_F32, "bf16 and f16 take grad_chunk16");
    const uint4 *vb = (const uint4 *)(g.addr + g.head);
    const uint32_t niter = (g.nvec + 31) >> 5;
    FF ff;
    double acc_exact = 0.0;
    // one bulk L2 prefetch of the chunk's aligned body: the later runs of the
    // chunk then load from L2 while this run computes
    if (lane == 0 && g.nvec) prefetch_l2_bulk(vb, g.nvec * 16u);
    for (uint32_t r0 = 0; r0 < niter; r0 += kRunVec) {
        const uint32_t r1 = min(r0 + (uint32_t)kRunVec, niter);
        FastAcc a;
        for (uint32_t i0 = r0; i0 < r1; i0 += U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t vi = lane + ((i0 + u) << 5);
                v[u] = (i0 + u < r1 && vi < g.nvec) ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) fast_vec_f32(v[u], a);
        }
        if (!fast_flush_ff<DT>(a, ff)) {
            for (uint32_t i = r0; i < r1; ++i) {
                const uint32_t vi = lane + (i << 5);
                if (vi < g.nvec) exact_vec<DT>(vb[vi], acc_exact, n);
            }
        }
    }
    grad_head_tail<DT>(g, lane, acc_exact, n);
    return warp_total<DT>(ff, acc_exact);  // the warp's total, on every lane
}

// The 16-bit form: U vectors per lane in flight, taken as runs of kRun16 that
// start at the lane's offset sig, which carries over from chunk to chunk.
template <int DT, int U>
__device__ __forceinline__ double grad_chunk16(const GGeom &g, uint32_t lane, Counts &n, uint64_t &sig) {
    static_assert(U % kRun16 == 0, "whole runs per batch");
    const uint4 *vb = (const uint4 *)(g.addr + g.head);
    const uint32_t niter = (g.nvec + 31) >> 5;
    FF2 ff;
    double acc_exact = 0.0;
    if (lane == 0 && g.nvec) prefetch_l2_bulk(vb, g.nvec * 16u);
    for (uint32_t b0 = 0; b0 < niter; b0 += U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t vi = lane + ((b0 + u) << 5);
            v[u] = (b0 + u < niter && vi < g.nvec) ? ld_stream(vb + vi) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < U; r += kRun16) {
            const uint32_t r0 = b0 + r;
            if (r0 < niter) {  // the same on every lane
                const uint32_t r1 = min(r0 + (uint32_t)kRun16, niter);
                SAcc a{sig, 0ull};
#pragma unroll
                for (int u = r; u < r + kRun16; ++u) sacc_vec<DT>(v[u], a);  // zeros past the end add nothing
                uint64_t est;
                const bool ok = sacc_accept(a, sig, ff, est);
                const uint64_t sn = sigma_next(est);
                if (!ok) {
                    uint32_t cnt[3] = {n.nan, n.inf, n.big};
                    ff = run_fallback<DT>(vb, lane, r0, r1, g.nvec, sn, ff, &acc_exact, cnt, 1);
                    n.nan = cnt[0];
                    n.inf = cnt[1];
                    n.big = cnt[2];
                }
                sig = sn;
            }
        }
    }
    grad_head_tail<DT>(g, lane, acc_exact, n);
    return warp_total2(ff, acc_exact);
}

template <int U>
__global__ void __launch_bounds__(kScanBlock) grad_scan_kernel(const Chunk *__restrict__ chunks, uint64_t n_chunks,
                                                               StatPartial *__restrict__ partials) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    uint64_t sig = 0ull;  // the 16-bit path's run offset, carried across the warp's chunks
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const Chunk ch = chunks[c];
        const GGeom g = ggeom(ch);
        Counts n;
        double acc;
        switch (chunk_dtype(ch.tag)) {
            case SDC_DTYPE_F32: acc = grad_chunk<SDC_DTYPE_F32, U>(g, lane, n); break;
            case SDC_DTYPE_BF16: acc = grad_chunk16<SDC_DTYPE_BF16, U>(g, lane, n, sig); break;
            default: acc = grad_chunk16<SDC_DTYPE_F16, U>(g, lane, n, sig); break;
        }
        const uint32_t nn = warp_sum_u32(n.nan), ni = warp_sum_u32(n.inf), nb = warp_sum_u32(n.big);
        if (lane == 0) partials[c] = StatPartial{acc, nn, ni, nb, 0u};
    }
}

// ---------------------------------------------------------------- fused average + scan
struct BufPtrs {
    const void *p[8];
};

// Average of NB words (one per input) holding 2 bf16/f16 or 1 f32 element(s)
// in each half-word/word lane; returns the output word.
template <int DT, int NB>
__device__ __forceinline__ uint32_t avg_word_pair16(const uint32_t (&w)[NB], float inv) {
    float lo, hi;
    if (DT == SDC_DTYPE_BF16) {
        uint64_t a = f2_pack_bits(w[0] << 16, w[0] & 0xFFFF0000u);
#pragma unroll
        for (int b = 1; b < NB; ++b) a = f2_add(a, f2_pack_bits(w[b] << 16, w[b] & 0xFFFF0000u));
        f2_unpack(a, lo, hi);
    } else {
        lo = __half2float(__ushort_as_half((unsigned short)(w[0] & 0xFFFFu)));
        hi = __half2float(__ushort_as_half((unsigned short)(w[0] >> 16)));
        uint64_t a = f2_pack(lo, hi);
#pragma unroll
        for (int b = 1; b < NB; ++b) {
            const float l2 = __half2float(__ushort_as_half((unsigned short)(w[b] & 0xFFFFu)));
            const float h2 = __half2float(__ushort_as_half((unsigned short)(w[b] >> 16)));
            a = f2_add(a, f2_pack(l2, h2));
        }
        f2_unpack(a, lo, hi);
    }
    if ((NB & (NB - 1)) == 0) {  // power of two: multiplying by 1/NB is exact and equals the division
        lo = __fmul_rn(lo, inv);
        hi = __fmul_rn(hi, inv);
    } else {
        lo = __fdiv_rn(lo, (float)NB);
        hi = __fdiv_rn(hi, (float)NB);
    }
    uint32_t r;
    if (DT == SDC_DTYPE_BF16) {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        const uint32_t t = r & 0x7FFF7FFFu;
        if ((t + 0x007F007Fu) & 0x80008000u) {  // some half is NaN: canonical quiet NaN
            if ((t & 0xFFFFu) > 0x7F80u) r = (r & 0xFFFF0000u) | 0x7FC0u;
            if ((t >> 16) > 0x7F80u) r = (r & 0x0000FFFFu) | 0x7FC00000u;
        }
    } else {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        const uint32_t t = r & 0x7FFF7FFFu;
        if ((t + 0x03FF03FFu) & 0x80008000u) {
            if ((t & 0xFFFFu) > 0x7C00u) r = (r & 0xFFFF0000u) | 0x7E00u;
            if ((t >> 16) > 0x7C00u) r = (r & 0x0000FFFFu) | 0x7E000000u;
        }
    }
    return r;
}

template <int NB>
__device__ __forceinline__ uint32_t avg_word_f32(const uint32_t (&w)[NB], float inv) {
    float a = __uint_as_float(w[0]);
#pragma unroll
    for (int b = 1; b < NB; ++b) a = __fadd_rn(a, __uint_as_float(w[b]));
    a = ((NB & (NB - 1)) == 0) ? __fmul_rn(a, inv) : __fdiv_rn(a, (float)NB);
    uint32_t r = __float_as_uint(a);
    if ((r & 0x7FFFFFFFu) > 0x7F800000u) r = 0x7FC00000u;
    return r;
}

template <int DT, int NB>
__device__ __forceinline__ uint4 avg_vec(const uint4 (&v)[NB], float inv) {
    uint4 o;
    uint32_t wx[NB], wy[NB], wz[NB], ww[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        wx[b] = v[b].x;
        wy[b] = v[b].y;
        wz[b] = v[b].z;
        ww[b] = v[b].w;
    }
    if (DT == SDC_DTYPE_F32) {
        o.x = avg_word_f32<NB>(wx, inv);
        o.y = avg_word_f32<NB>(wy, inv);
        o.z = avg_word_f32<NB>(wz, inv);
        o.w = avg_word_f32<NB>(ww, inv);
    } else {
        o.x = avg_word_pair16<DT, NB>(wx, inv);
        o.y = avg_word_pair16<DT, NB>(wy, inv);
        o.z = avg_word_pair16<DT, NB>(wz, inv);
        o.w = avg_word_pair16<DT, NB>(ww, inv);
    }
    return o;
}

// One element of the average, for tails and the element path.
template <int DT>
__device__ __forceinline__ uint32_t avg_elem(const BufPtrs &bp, int nb, uint64_t i) {
    float a = 0.0f;
    for (int b = 0; b < nb; ++b) {
        uint32_t bits = DT == SDC_DTYPE_F32 ? ((const uint32_t *)bp.p[b])[i] : ((const uint16_t *)bp.p[b])[i];
        const float x = to_float(bits, DT);
        a = b == 0 ? x : __fadd_rn(a, x);
    }
    a = __fdiv_rn(a, (float)nb);  // equals the multiply by 1/nb when nb is a power of two
    if (DT == SDC_DTYPE_F32) {
        uint32_t r = __float_as_uint(a);
        return (r & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : r;
    } else if (DT == SDC_DTYPE_BF16) {
        if (isnan(a)) return 0x7FC0u;
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a));
    } else {
        if (isnan(a)) return 0x7E00u;
        return (uint32_t)__half_as_ushort(__float2half_rn(a));
    }
}

template <int DT>
__device__ __forceinline__ uint32_t load_bits(const void *p, uint64_t i) {
    return DT == SDC_DTYPE_F32 ? ((const uint32_t *)p)[i] : ((const uint16_t *)p)[i];
}
template <int DT>
__device__ __forceinline__ void store_bits(void *p, uint64_t i, uint32_t v) {
    if (DT == SDC_DTYPE_F32) ((uint32_t *)p)[i] = v;
    else ((uint16_t *)p)[i] = (uint16_t)v;
}

// Vector path: every pointer 16-byte aligned.  Warp task c covers elements
// [c * CE, min((c + 1) * CE, numel)), CE = kAvgChunkBytes / elem size.
// Partials: [s][c] for streams s = 0..NB-1 (inputs) and s = NB (average).
template <int DT, int NB, int U>
__global__ void __launch_bounds__(kScanBlock) avg_scan_kernel(BufPtrs bp, void *__restrict__ outp, uint64_t numel,
                                                              uint64_t n_chunks, StatPartial *__restrict__ partials) {
    static_assert(DT == SDC_DTYPE_F32, "bf16 and f16 take avg_scan16_kernel");
    constexpr int NS = NB + 1;
    constexpr uint32_t ES = 4u;
    constexpr uint64_t CE = kAvgChunkBytes / ES;
    const float inv = 1.0f / (float)NB;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const uint64_t e0 = c * CE;
        const uint64_t ne = min(CE, numel - e0);
        const uint32_t nvec = (uint32_t)((ne * ES) >> 4);
        const uint32_t niter = (nvec + 31) >> 5;
        const uint4 *in[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) in[b] = (const uint4 *)((const char *)bp.p[b] + e0 * ES);
        uint4 *out = (uint4 *)((char *)outp + e0 * ES);
        FF ff[NS];
        double acc_e[NS];
        Counts n[NS];
#pragma unroll
        for (int s = 0; s < NS; ++s) acc_e[s] = 0.0;
        for (uint32_t r0 = 0; r0 < niter; r0 += kRunVec) {
            const uint32_t r1 = min(r0 + (uint32_t)kRunVec, niter);
            FastAcc a[NS];
            for (uint32_t i0 = r0; i0 < r1; i0 += U) {
                // L2 prefetch of the batch after next: lanes 0, 8, 16, 24 touch the
                // four 128-byte lines of each input's 512-byte warp slice
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t vi = lane + ((i0 + 2 * U + u) << 5);
                    if ((lane & 7u) == 0 && vi < nvec)
#pragma unroll
                        for (int b = 0; b < NB; ++b) prefetch_l2(in[b] + vi);
                }
                uint4 v[U][NB];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t vi = lane + ((i0 + u) << 5);
                    const bool ok = i0 + u < r1 && vi < nvec;
#pragma unroll
                    for (int b = 0; b < NB; ++b) v[u][b] = ok ? ld_stream(in[b] + vi) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t vi = lane + ((i0 + u) << 5);
                    const bool ok = i0 + u < r1 && vi < nvec;
#pragma unroll
                    for (int b = 0; b < NB; ++b) fast_vec_f32(v[u][b], a[b]);
                    uint4 o = avg_vec<DT, NB>(v[u], inv);
                    if (ok) {
                        __stcs(out + vi, o);
                    } else {
                        o = make_uint4(0, 0, 0, 0);
                    }
                    fast_vec_f32(o, a[NB]);
                }
            }
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                if (!fast_flush_ff<DT>(a[s], ff[s])) {
                    const uint4 *src = s < NB ? in[s] : (const uint4 *)out;
                    for (uint32_t i = r0; i < r1; ++i) {
                        const uint32_t vi = lane + (i << 5);
                        if (vi < nvec) exact_vec<DT>(src[vi], acc_e[s], n[s]);
                    }
                }
            }
        }
        // tail elements of the last chunk (fewer than one vector)
        const uint64_t done = (uint64_t)nvec * (16u / ES);
        if (lane < ne - done) {
            const uint64_t i = e0 + done + lane;
            const uint32_t r = avg_elem<DT>(bp, NB, i);
            store_bits<DT>(outp, i, r);
#pragma unroll
            for (int b = 0; b < NB; ++b) exact_elem(load_bits<DT>(bp.p[b], i), DT, acc_e[b], n[b]);
            exact_elem(r, DT, acc_e[NB], n[NB]);
        }
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const double acc = warp_total<DT>(ff[s], acc_e[s]);
            const uint32_t nn = warp_sum_u32(n[s].nan), ni = warp_sum_u32(n[s].inf), nbg = warp_sum_u32(n[s].big);
            if (lane == 0) partials[(uint64_t)s * n_chunks + c] = StatPartial{acc, nn, ni, nbg, 0u};
        }
    }
}

// The 16-bit form of avg_scan_kernel (bf16, f16): every stream accumulated in
// offset runs of kRun16 vectors per lane, each stream's offset carried across
// the warp's tasks.  The exact path's sums and counts, touched only by runs
// that fail and by the tail, live in shared memory ([stream][thread]) so that
// two blocks of 256 threads fit on an SM.
template <int DT, int NB, int U>
__global__ void __launch_bounds__(kScanBlock) avg_scan16_kernel(BufPtrs bp, void *__restrict__ outp, uint64_t numel,
                                                                uint64_t n_chunks, StatPartial *__restrict__ partials) {
    static_assert(kRun16 % U == 0, "whole batches per run");
    constexpr int NS = NB + 1;
    constexpr uint64_t CE = kAvgChunkBytes / 2;
    __shared__ double sh_acc[NS][kScanBlock];
    __shared__ uint32_t sh_cnt[NS][3][kScanBlock];
    const float inv = 1.0f / (float)NB;
    const uint32_t tid = threadIdx.x, lane = tid & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + tid) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    uint64_t sig[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) sig[s] = 0ull;
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const uint64_t e0 = c * CE;
        const uint64_t ne = min(CE, numel - e0);
        const uint32_t nvec = (uint32_t)((ne * 2u) >> 4);
        const uint32_t niter = (nvec + 31) >> 5;
        const uint4 *in[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) in[b] = (const uint4 *)((const char *)bp.p[b] + e0 * 2u);
        uint4 *out = (uint4 *)((char *)outp + e0 * 2u);
        FF2 ff[NS];
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            sh_acc[s][tid] = 0.0;
            sh_cnt[s][0][tid] = sh_cnt[s][1][tid] = sh_cnt[s][2][tid] = 0u;
        }
        for (uint32_t r0 = 0; r0 < niter; r0 += kRun16) {
            const uint32_t r1 = min(r0 + (uint32_t)kRun16, niter);
            SAcc a[NS];
#pragma unroll
            for (int s = 0; s < NS; ++s) a[s] = SAcc{sig[s], 0ull};
            for (uint32_t i0 = r0; i0 < r1; i0 += U) {  // not unrolled: the body stays in the instruction cache
                // L2 prefetch of the batch after next: lanes 0, 8, 16, 24 touch the
                // four 128-byte lines of each input's 512-byte warp slice
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t vi = lane + ((i0 + 2 * U + u) << 5);
                    if ((lane & 7u) == 0 && vi < nvec)
#pragma unroll
                        for (int b = 0; b < NB; ++b) prefetch_l2(in[b] + vi);
                }
                uint4 v[U][NB];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t vi = lane + ((i0 + u) << 5);
                    const bool ok = i0 + u < r1 && vi < nvec;
#pragma unroll
                    for (int b = 0; b < NB; ++b) v[u][b] = ok ? ld_stream(in[b] + vi) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t vi = lane + ((i0 + u) << 5);
                    const bool ok = i0 + u < r1 && vi < nvec;
#pragma unroll
                    for (int b = 0; b < NB; ++b) sacc_vec<DT>(v[u][b], a[b]);
                    uint4 o = avg_vec<DT, NB>(v[u], inv);
                    if (ok) {
                        __stcs(out + vi, o);
                    } else {
                        o = make_uint4(0, 0, 0, 0);
                    }
                    sacc_vec<DT>(o, a[NB]);
                }
            }
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                uint64_t est;
                const bool ok = sacc_accept(a[s], sig[s], ff[s], est);
                const uint64_t sn = sigma_next(est);
                if (!ok)
                    ff[s] = run_fallback<DT>(s < NB ? in[s] : (const uint4 *)out, lane, r0, r1, nvec, sn, ff[s],
                                             &sh_acc[s][tid], &sh_cnt[s][0][tid], kScanBlock);
                sig[s] = sn;
            }
        }
        // tail elements of the last chunk (fewer than one vector)
        const uint64_t done = (uint64_t)nvec * 8u;
        if (lane < ne - done) {
            const uint64_t i = e0 + done + lane;
            const uint32_t r = avg_elem<DT>(bp, NB, i);
            store_bits<DT>(outp, i, r);
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                double acc = sh_acc[s][tid];
                Counts cn;
                cn.nan = sh_cnt[s][0][tid];
                cn.inf = sh_cnt[s][1][tid];
                cn.big = sh_cnt[s][2][tid];
                exact_elem(s < NB ? load_bits<DT>(bp.p[s], i) : r, DT, acc, cn);
                sh_acc[s][tid] = acc;
                sh_cnt[s][0][tid] = cn.nan;
                sh_cnt[s][1][tid] = cn.inf;
                sh_cnt[s][2][tid] = cn.big;
            }
        }
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const double acc = warp_total2(ff[s], sh_acc[s][tid]);
            const uint32_t nn = warp_sum_u32(sh_cnt[s][0][tid]), ni = warp_sum_u32(sh_cnt[s][1][tid]),
                           nbg = warp_sum_u32(sh_cnt[s][2][tid]);
            if (lane == 0) partials[(uint64_t)s * n_chunks + c] = StatPartial{acc, nn, ni, nbg, 0u};
        }
    }
}

// Element path (some pointer not 16-byte aligned): same task layout, every
// element exact.
template <int DT>
__global__ void __launch_bounds__(kScanBlock) avg_scan_elem_kernel(BufPtrs bp, int nb, void *__restrict__ outp,
                                                                   uint64_t numel, uint64_t n_chunks,
                                                                   StatPartial *__restrict__ partials) {
    constexpr uint32_t ES = DT == SDC_DTYPE_F32 ? 4u : 2u;
    constexpr uint64_t CE = kAvgChunkBytes / ES;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const int ns = nb + 1;
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const uint64_t e0 = c * CE;
        const uint64_t ne = min(CE, numel - e0);
        for (int s = 0; s < ns; ++s) {
            double acc = 0.0;
            Counts n;
            for (uint64_t j = lane; j < ne; j += 32) {
                const uint64_t i = e0 + j;
                uint32_t bits;
                if (s < nb) {
                    bits = load_bits<DT>(bp.p[s], i);
                } else {
                    bits = avg_elem<DT>(bp, nb, i);
                    store_bits<DT>(outp, i, bits);
                }
                exact_elem(bits, DT, acc, n);
            }
            acc = warp_sum_f64(acc);
            const uint32_t nn = warp_sum_u32(n.nan), ni = warp_sum_u32(n.inf), nbg = warp_sum_u32(n.big);
            if (lane == 0) partials[(uint64_t)s * n_chunks + c] = StatPartial{acc, nn, ni, nbg, 0u};
        }
    }
}

// ---------------------------------------------------------------- combine
// Two fixed-shape passes per stream, so the float64 sum has the same
// association on every run whatever the grid: pass 1 splits a stream's
// partials into kGroups contiguous ranges (range bounds depend only on the
// count), one CTA per (stream, group) summing its range in a fixed order
// (thread t takes t, t + B, ...; then a fixed tree); pass 2 sums the kGroups
// group results of each stream in a fixed tree and writes the derived fields.
constexpr int kCombineBlock = 256;

struct StreamSel {
    const uint64_t *first;  // plan mode: R + 1 chunk offsets; null in buffer mode
    const uint64_t *numel_arr;
    uint64_t n_chunks;      // buffer mode: chunks per stream (partials are stream-major)
    uint64_t numel;         // buffer mode: elements per stream
    uint32_t n_streams;
    uint32_t n_pre;         // buffer mode: streams written to out_pre (the rest to out_post)
};

__device__ __forceinline__ void stream_range(const StreamSel &sel, uint32_t s, uint64_t &base, uint64_t &count) {
    if (sel.first) {
        base = sel.first[s];
        count = sel.first[s + 1] - base;
    } else {
        base = (uint64_t)s * sel.n_chunks;
        count = sel.n_chunks;
    }
}

struct Acc {
    double sum;
    unsigned long long nan, inf, big;
};

// Fixed-shape block reduction of one Acc per thread; result valid in thread 0.
__device__ __forceinline__ Acc block_reduce(Acc a) {
    __shared__ double sa[kCombineBlock];
    __shared__ unsigned long long sn[3][kCombineBlock];
    sa[threadIdx.x] = a.sum;
    sn[0][threadIdx.x] = a.nan;
    sn[1][threadIdx.x] = a.inf;
    sn[2][threadIdx.x] = a.big;
    __syncthreads();
    for (int h = kCombineBlock / 2; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) {
            sa[threadIdx.x] = __dadd_rn(sa[threadIdx.x], sa[threadIdx.x + h]);
            sn[0][threadIdx.x] += sn[0][threadIdx.x + h];
            sn[1][threadIdx.x] += sn[1][threadIdx.x + h];
            sn[2][threadIdx.x] += sn[2][threadIdx.x + h];
        }
        __syncthreads();
    }
    return Acc{sa[0], sn[0][0], sn[1][0], sn[2][0]};
}

__global__ void __launch_bounds__(kCombineBlock) stats_combine1_kernel(const StatPartial *__restrict__ partials,
                                                                       StreamSel sel, StatGroup *__restrict__ groups) {
    const uint32_t s = blockIdx.y, g = blockIdx.x;
    uint64_t base, count;
    stream_range(sel, s, base, count);
    const uint64_t lo = base + count * g / kStatGroups, hi = base + count * (g + 1) / kStatGroups;
    Acc a{0.0, 0, 0, 0};
    for (uint64_t i = lo + threadIdx.x; i < hi; i += kCombineBlock) {
        const StatPartial p = partials[i];
        a.sum = __dadd_rn(a.sum, p.sumsq);
        a.nan += p.n_nan;
        a.inf += p.n_inf;
        a.big += p.n_big;
    }
    a = block_reduce(a);
    if (threadIdx.x == 0)
        groups[(uint64_t)s * kStatGroups + g] = StatGroup{a.sum, a.nan, a.inf, a.big};
}

__global__ void __launch_bounds__(kCombineBlock) stats_combine2_kernel(const StatGroup *__restrict__ groups,
                                                                       StreamSel sel, sdc_grad_stats *out_pre,
                                                                       sdc_grad_stats *out_post) {
    const uint32_t s = blockIdx.x;
    Acc a{0.0, 0, 0, 0};
    for (uint32_t g = threadIdx.x; g < kStatGroups; g += kCombineBlock) {
        const StatGroup p = groups[(uint64_t)s * kStatGroups + g];
        a.sum = __dadd_rn(a.sum, p.sumsq);
        a.nan += p.n_nan;
        a.inf += p.n_inf;
        a.big += p.n_big;
    }
    a = block_reduce(a);
    if (threadIdx.x == 0) {
        sdc_grad_stats r;
        r.n_nan = a.nan;
        r.n_inf = a.inf;
        r.n_big = a.big;
        r.n_elems = sel.first ? sel.numel_arr[s] : sel.numel;
        r.sumsq_finite = a.sum;
        if (r.n_nan) r.norm = __longlong_as_double(0x7FF8000000000000ll);
        else if (r.n_inf) r.norm = __longlong_as_double(0x7FF0000000000000ll);
        else r.norm = __dsqrt_rn(a.sum);
        r.nonfinite_fp32 = (r.n_nan || r.n_inf || a.sum > kFltMax) ? 1u : 0u;
        r.reserved = 0;
        sdc_grad_stats *dst = sel.first ? out_pre + s : (s < sel.n_pre ? out_pre + s : out_post);
        *dst = r;
    }
}

cudaError_t launch_combine(const StatPartial *partials, StatGroup *groups, const StreamSel &sel,
                           sdc_grad_stats *out_pre, sdc_grad_stats *out_post, cudaStream_t st) {
    stats_combine1_kernel<<<dim3(kStatGroups, sel.n_streams), kCombineBlock, 0, st>>>(partials, sel, groups);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    stats_combine2_kernel<<<sel.n_streams, kCombineBlock, 0, st>>>(groups, sel, out_pre, out_post);
    return cudaGetLastError();
}

constexpr int kGradUnroll = 16;  // a whole run (kRunVec vectors per lane) in flight
constexpr int kAvgUnroll = 2;
constexpr int kAvg16Unroll = 2;

template <int DT, int NB>
cudaError_t launch_avg_t(const BufPtrs &bp, void *avg, uint64_t numel, StatPartial *partials, uint64_t n_chunks,
                         int device, cudaStream_t st) {
    void (*kernel)(BufPtrs, void *, uint64_t, uint64_t, StatPartial *);
    if constexpr (DT == SDC_DTYPE_F32) kernel = avg_scan_kernel<DT, NB, kAvgUnroll>;
    else kernel = avg_scan16_kernel<DT, NB, kAvg16Unroll>;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kScanBlock, 0);
    if (per_sm < 1) per_sm = 1;
    uint64_t grid = (uint64_t)sm_count(device) * per_sm;
    const uint64_t need = (n_chunks * 32 + kScanBlock - 1) / kScanBlock;
    if (need < grid) grid = need;
    kernel<<<(unsigned)grid, kScanBlock, 0, st>>>(bp, avg, numel, n_chunks, partials);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_avg_dt(const BufPtrs &bp, uint32_t nb, void *avg, uint64_t numel, StatPartial *partials,
                          uint64_t n_chunks, int device, cudaStream_t st) {
    switch (nb) {
        case 1: return launch_avg_t<DT, 1>(bp, avg, numel, partials, n_chunks, device, st);
        case 2: return launch_avg_t<DT, 2>(bp, avg, numel, partials, n_chunks, device, st);
        case 3: return launch_avg_t<DT, 3>(bp, avg, numel, partials, n_chunks, device, st);
        case 4: return launch_avg_t<DT, 4>(bp, avg, numel, partials, n_chunks, device, st);
        case 5: return launch_avg_t<DT, 5>(bp, avg, numel, partials, n_chunks, device, st);
        case 6: return launch_avg_t<DT, 6>(bp, avg, numel, partials, n_chunks, device, st);
        case 7: return launch_avg_t<DT, 7>(bp, avg, numel, partials, n_chunks, device, st);
        default: return launch_avg_t<DT, 8>(bp, avg, numel, partials, n_chunks, device, st);
    }
}

}  // namespace

int grad_scan_blocks_per_sm() {
    int n = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, grad_scan_kernel<kGradUnroll>, kScanBlock, 0);
    return n > 0 ? n : 1;
}

cudaError_t launch_grad_scan(const sdc_plan *plan, StatPartial *partials, cudaStream_t st) {
    if (plan->n_chunks == 0) return cudaSuccess;
    uint64_t grid = (uint64_t)sm_count(plan->device) * grad_scan_blocks_per_sm();
    const uint64_t need = (plan->n_chunks * 32 + kScanBlock - 1) / kScanBlock;
    if (need < grid) grid = need;
    grad_scan_kernel<kGradUnroll><<<(unsigned)grid, kScanBlock, 0, st>>>(plan->d_chunks, plan->n_chunks, partials);
    return cudaGetLastError();
}

cudaError_t launch_stats_combine_plan(const sdc_plan *plan, const StatPartial *partials, StatGroup *groups,
                                      sdc_grad_stats *out, cudaStream_t st) {
    StreamSel sel{plan->d_replica_first_chunk, plan->d_replica_numel, 0, 0, plan->R, plan->R};
    return launch_combine(partials, groups, sel, out, out, st);
}

cudaError_t launch_avg_scan(const void *const *bufs, uint32_t n_bufs, void *avg, uint64_t numel, uint32_t dtype,
                            StatPartial *partials, uint64_t n_chunks, bool vector_path, int device,
                            cudaStream_t st) {
    if (n_chunks == 0) return cudaSuccess;
    BufPtrs bp{};
    for (uint32_t b = 0; b < n_bufs; ++b) bp.p[b] = bufs[b];
    if (vector_path) {
        switch (dtype) {
            case SDC_DTYPE_F32: return launch_avg_dt<SDC_DTYPE_F32>(bp, n_bufs, avg, numel, partials, n_chunks, device, st);
            case SDC_DTYPE_BF16: return launch_avg_dt<SDC_DTYPE_BF16>(bp, n_bufs, avg, numel, partials, n_chunks, device, st);
            default: return launch_avg_dt<SDC_DTYPE_F16>(bp, n_bufs, avg, numel, partials, n_chunks, device, st);
        }
    }
    uint64_t grid = (uint64_t)sm_count(device) * 4;
    const uint64_t need = (n_chunks * 32 + kScanBlock - 1) / kScanBlock;
    if (need < grid) grid = need;
    switch (dtype) {
        case SDC_DTYPE_F32:
            avg_scan_elem_kernel<SDC_DTYPE_F32><<<(unsigned)grid, kScanBlock, 0, st>>>(bp, (int)n_bufs, avg, numel, n_chunks, partials);
            break;
        case SDC_DTYPE_BF16:
            avg_scan_elem_kernel<SDC_DTYPE_BF16><<<(unsigned)grid, kScanBlock, 0, st>>>(bp, (int)n_bufs, avg, numel, n_chunks, partials);
            break;
        default:
            avg_scan_elem_kernel<SDC_DTYPE_F16><<<(unsigned)grid, kScanBlock, 0, st>>>(bp, (int)n_bufs, avg, numel, n_chunks, partials);
            break;
    }
    return cudaGetLastError();
}

cudaError_t launch_stats_combine_streams(const StatPartial *partials, StatGroup *groups, uint32_t n_streams,
                                         uint64_t n_chunks, uint64_t numel, sdc_grad_stats *out_pre,
                                         sdc_grad_stats *out_post, cudaStream_t st) {
    StreamSel sel{nullptr, nullptr, n_chunks, numel, n_streams, n_streams - 1};
    return launch_combine(partials, groups, sel, out_pre, out_post, st);
}

}  // namespace sdc
