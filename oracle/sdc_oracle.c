/*
 * sdc_oracle.c -- the plain, slow, obviously-correct CPU statement of what the
 * replica-integrity scan computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline load it (through oracle/__init__.py).  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * Sources (web pages on silent data corruption):
 *   [AWS]   "Detecting and recovering from silent data corruption on Amazon
 *            SageMaker HyperPod" (AWS Machine Learning Blog)
 *   [AEGIS] "Safeguarding LLM Training at Scale: Online SDC Detection and
 *            Insights from 35 Million GPU Hours" (review page)
 *
 * Every loop below walks the elements one at a time, in flat row-major order,
 * with no blocking, chunking or reordering.  Integer results wrap mod 2^64.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Raw bit pattern of element i, widened to 64 bits.                          */
/*                                                                            */
/* [AWS] "Compare by fingerprint": a tensor is viewed through an integer type */
/* of its element width -- unsigned 8-bit for 1-byte elements, signed 16/32/64 */
/* for wider ones -- and then widened to int64.  So 1-byte elements are        */
/* zero-extended and wider ones sign-extended.  Bytes are little-endian.       */
/* ------------------------------------------------------------------------ */
static uint64_t element_bits_widened(const unsigned char *p, uint64_t i, uint32_t esize)
{
    if (esize == 1) {
        return (uint64_t)p[i];
    } else if (esize == 2) {
        int16_t v;
        memcpy(&v, p + 2 * i, 2);
        return (uint64_t)(int64_t)v;
    } else if (esize == 4) {
        int32_t v;
        memcpy(&v, p + 4 * i, 4);
        return (uint64_t)(int64_t)v;
    } else {
        int64_t v;
        memcpy(&v, p + 8 * i, 8);
        return (uint64_t)v;
    }
}

/* Same element, zero-extended (the xorsum reading: raw bits, no sign). */
static uint64_t element_bits_zero_extended(const unsigned char *p, uint64_t i, uint32_t esize)
{
    uint64_t v = 0;
    memcpy(&v, p + (uint64_t)esize * i, esize); /* little-endian host */
    return v;
}

/* ------------------------------------------------------------------------ */
/* Fingerprint of one tensor.  [AWS] "Compare by fingerprint":               */
/*   S = sum_i b_i            (mod 2^64)                                      */
/*   W = sum_i (i + 1) * b_i  (mod 2^64), i = 0-based flat index              */
/* The page's position vector starts at 1 and runs across its chunks, so the */
/* weight is the global 1-based index.  `first_index` is the global index of  */
/* data[0]: a caller may walk one tensor in consecutive slices, exactly as    */
/* the page's chunk loop does, and add the slices' (S, W) mod 2^64.           */
/* Returns 0, or -1 on a bad esize.                                           */
/* ------------------------------------------------------------------------ */
int oracle_fingerprint(const void *data, uint64_t numel, uint32_t esize, uint64_t first_index,
                       uint64_t out[2])
{
    const unsigned char *p = (const unsigned char *)data;
    uint64_t s = 0, w = 0;
    if (esize != 1 && esize != 2 && esize != 4 && esize != 8) return -1;
    for (uint64_t i = 0; i < numel; ++i) {
        uint64_t b = element_bits_widened(p, i, esize);
        s += b;
        w += (first_index + i + 1) * b;
    }
    out[0] = s;
    out[1] = w;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Xorsum of one tensor.  [AEGIS] section 4 ("reusing deterministic          */
/* recomputation"): the original and recomputed results are each reduced to  */
/* an xorsum fingerprint and any differing bit is a confirmed anomaly.  The   */
/* page gives no width; read here as the XOR of every element's raw bits,     */
/* zero-extended to 64 bits.                                                 */
/* ------------------------------------------------------------------------ */
int oracle_xorsum(const void *data, uint64_t numel, uint32_t esize, uint64_t *out)
{
    const unsigned char *p = (const unsigned char *)data;
    uint64_t x = 0;
    if (esize != 1 && esize != 2 && esize != 4 && esize != 8) return -1;
    for (uint64_t i = 0; i < numel; ++i) x ^= element_bits_zero_extended(p, i, esize);
    *out = x;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Floating-point element decoding, from the IEEE-754 layouts:               */
/*   kind 0 = finite (value = (-1)^sign * m * 2^q, m >= 0 an integer)         */
/*   kind 1 = NaN, kind 2 = +-Inf                                             */
/* dtype codes of this file: 1 = float32, 2 = bfloat16, 3 = float16.         */
/* ------------------------------------------------------------------------ */
#define ORACLE_F32 1
#define ORACLE_BF16 2
#define ORACLE_F16 3

static int decode(const unsigned char *p, uint64_t i, uint32_t dtype, uint64_t *m, int *q)
{
    if (dtype == ORACLE_F32) {
        uint32_t u;
        memcpy(&u, p + 4 * i, 4);
        uint32_t e = (u >> 23) & 0xFFu, f = u & 0x7FFFFFu;
        if (e == 0xFFu) return f ? 1 : 2;
        if (e == 0) { *m = f; *q = 1 - 127 - 23; }
        else { *m = f | 0x800000u; *q = (int)e - 127 - 23; }
        return 0;
    } else if (dtype == ORACLE_BF16) {
        uint16_t h;
        memcpy(&h, p + 2 * i, 2);
        uint32_t e = (h >> 7) & 0xFFu, f = h & 0x7Fu;
        if (e == 0xFFu) return f ? 1 : 2;
        if (e == 0) { *m = f; *q = 1 - 127 - 7; }
        else { *m = f | 0x80u; *q = (int)e - 127 - 7; }
        return 0;
    } else { /* ORACLE_F16 */
        uint16_t h;
        memcpy(&h, p + 2 * i, 2);
        uint32_t e = (h >> 10) & 0x1Fu, f = h & 0x3FFu;
        if (e == 0x1Fu) return f ? 1 : 2;
        if (e == 0) { *m = f; *q = 1 - 15 - 10; }
        else { *m = f | 0x400u; *q = (int)e - 15 - 10; }
        return 0;
    }
}

/* Lowest exponent q any of the three formats produces (float32 subnormals). */
#define ORACLE_QMIN (-149)
/* Number of exponent bins: q runs from -149 (f32 subnormal) to 120 (bf16 max). */
#define ORACLE_NBINS 270

/* ------------------------------------------------------------------------ */
/* Gradient statistics of one buffer.                                        */
/* [AWS] "Check 1: NaN/Inf gradients, before and after the all-reduce": the  */
/* hook keeps the squared norm of the local gradient, and a rank is flagged   */
/* when that norm is NaN or Inf -- which, in float32, includes a norm above   */
/* about 1.8e19 ("Decide what the alarm means" table).                        */
/*                                                                            */
/* Per element: NaN, Inf, or finite.  A finite element is "big" when its      */
/* exact square exceeds FLT_MAX (its square alone overflows float32).         */
/* The sum of squares over finite elements is accumulated EXACTLY: each       */
/* finite x = m * 2^q has x^2 = m^2 * 4^q, and m^2 is added, as a 128-bit     */
/* integer, to the bin of its exponent q.  The caller turns the bins into one */
/* correctly rounded double.                                                  */
/*                                                                            */
/* counts[0..2] = n_nan, n_inf, n_big.  bins = ORACLE_NBINS pairs (lo, hi)    */
/* of 64-bit words, bin b holding the sum of m^2 for q = b + ORACLE_QMIN.      */
/* The bins are ADDED to (callers zero them first), so one buffer may be      */
/* processed in several calls.                                                */
/* ------------------------------------------------------------------------ */
int oracle_grad_stats(const void *data, uint64_t numel, uint32_t dtype, uint64_t counts[3],
                      uint64_t *bins)
{
    const unsigned char *p = (const unsigned char *)data;
    const double flt_max = 3.4028234663852886e38; /* (2 - 2^-23) * 2^127 */
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    for (uint64_t i = 0; i < numel; ++i) {
        uint64_t m = 0;
        int q = 0;
        int kind = decode(p, i, dtype, &m, &q);
        if (kind == 1) { counts[0]++; continue; }
        if (kind == 2) { counts[1]++; continue; }
        /* m < 2^24, so m^2 < 2^48 is exact in a double; ldexp scales exactly */
        double x2 = ldexp((double)(m * m), 2 * q);
        if (x2 > flt_max) counts[2]++;
        unsigned __int128 acc;
        int b = q - ORACLE_QMIN;
        memcpy(&acc, bins + 2 * b, 16);
        acc += (unsigned __int128)(m * m);
        memcpy(bins + 2 * b, &acc, 16);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Round a float32 value to a narrower binary format, ties to even, from the  */
/* IEEE-754 definition: keep `mant` fraction bits, exponent range down to     */
/* 2^emin for normals (subnormals below, spaced 2^(emin - mant)), and values  */
/* whose rounded magnitude reaches 2^(emax+1) become Inf.  NaN is handled by  */
/* the caller.  Returns the encoded bits (sign | exponent | fraction).        */
/* ------------------------------------------------------------------------ */
static uint32_t round_to_format(float xf, int mant, int ebits, int emin, int emax)
{
    uint32_t sign_bit = 1u << (mant + ebits);
    uint32_t sign = signbit(xf) ? sign_bit : 0u;
    double a = fabs((double)xf); /* exact */
    int bias = (1 << (ebits - 1)) - 1;
    if (isinf(a)) return sign | ((uint32_t)((1 << ebits) - 1) << mant);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): the leading bit has weight 2^(e-1) */
    int lead = e - 1;
    if (lead < emin) lead = emin;          /* subnormal spacing below 2^emin */
    double ulp = ldexp(1.0, lead - mant);  /* spacing of representable values */
    double k = a / ulp;                    /* exact: a has 24 bits */
    double r = nearbyint(k);               /* default mode: round half to even */
    double v = r * ulp;                    /* exact */
    if (v >= ldexp(1.0, emax + 1)) return sign | ((uint32_t)((1 << ebits) - 1) << mant);
    if (v == 0.0) return sign; /* rounded down to zero */
    /* encode v */
    int ve;
    frexp(v, &ve);
    int vlead = ve - 1;
    if (vlead < emin) { /* subnormal: fraction = v / 2^(emin - mant) */
        uint32_t frac = (uint32_t)(v / ldexp(1.0, emin - mant));
        return sign | frac;
    }
    uint32_t bexp = (uint32_t)(vlead + bias);
    uint32_t frac = (uint32_t)(v / ldexp(1.0, vlead - mant) - ldexp(1.0, mant));
    return sign | (bexp << mant) | frac;
}

/* ------------------------------------------------------------------------ */
/* Average of n local gradient buffers, the one-device stand-in for the      */
/* all-reduce.  [AWS] "Step 1: Detect": after backward, an all-reduce         */
/* averages the replicas' gradients and every replica applies that average.   */
/* The pages fix no arithmetic; the reading used here is:                     */
/*   acc = float32 sum of the n inputs in buffer order (each add rounded)     */
/*   avg = acc / n in float32 (correctly rounded)                             */
/*   out = avg rounded to the buffers' dtype, ties to even;                   */
/*         any NaN becomes the canonical quiet NaN of that dtype.             */
/* ------------------------------------------------------------------------ */
static float load_as_float(const unsigned char *p, uint64_t i, uint32_t dtype)
{
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, p + 4 * i, 4);
        return f;
    }
    uint64_t m = 0;
    int q = 0;
    uint16_t h;
    memcpy(&h, p + 2 * i, 2);
    int neg = (h >> 15) & 1;
    int kind = decode(p, i, dtype, &m, &q);
    if (kind == 1) return NAN;
    if (kind == 2) return neg ? -INFINITY : INFINITY;
    float v = (float)ldexp((double)m, q); /* exact: 8 or 11 bits in float32 range */
    return neg ? -v : v;
}

int oracle_average(const void *const *bufs, uint32_t n_bufs, uint64_t numel, uint32_t dtype, void *out)
{
    unsigned char *o = (unsigned char *)out;
    if (n_bufs == 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    for (uint64_t i = 0; i < numel; ++i) {
        volatile float acc = load_as_float((const unsigned char *)bufs[0], i, dtype);
        for (uint32_t b = 1; b < n_bufs; ++b) {
            volatile float x = load_as_float((const unsigned char *)bufs[b], i, dtype);
            acc = acc + x;
        }
        volatile float avg = acc / (float)n_bufs;
        if (dtype == ORACLE_F32) {
            uint32_t u;
            float a = avg;
            memcpy(&u, &a, 4);
            if (isnan(a)) u = 0x7FC00000u;
            memcpy(o + 4 * i, &u, 4);
        } else {
            uint16_t h;
            if (isnan(avg)) h = (dtype == ORACLE_BF16) ? 0x7FC0u : 0x7E00u;
            else if (dtype == ORACLE_BF16) h = (uint16_t)round_to_format(avg, 7, 8, -126, 127);
            else h = (uint16_t)round_to_format(avg, 10, 5, -14, 15);
            memcpy(o + 2 * i, &h, 2);
        }
    }
    return 0;
}

/* Exposed for the oracle's own pins: float32 -> bf16 / f16 bits. */
uint32_t oracle_round_f32(float x, uint32_t dtype)
{
    if (isnan(x)) return dtype == ORACLE_BF16 ? 0x7FC0u : 0x7E00u;
    if (dtype == ORACLE_BF16) return round_to_format(x, 7, 8, -126, 127);
    return round_to_format(x, 10, 5, -14, 15);
}

/* ------------------------------------------------------------------------ */
/* One AdamW step with gradient clipping, in place.                          */
/* [AWS] "Use case: Testing the checks on SageMaker HyperPod": AdamW with     */
/* betas (0.9, 0.95), weight decay 0.1, gradient clipping at 1.0; `train()`   */
/* clips (clip_grad_norm_), skips the step when the reduced gradient is not   */
/* finite, else steps.  The pages fix no float arithmetic; the reading here   */
/* is this sequence of separately rounded float32 operations (decoupled       */
/* weight decay, bias-corrected moments), with the scalars already rounded    */
/* to float32 by the caller:                                                  */
/*   g  = grad * coef                       (coef == 1: g = grad)            */
/*   p  = p * decay                         decay = 1 - lr * wd               */
/*   m  = m + omb1 * (g - m)                omb1 = 1 - beta1                  */
/*   v  = v * beta2 + (g * g) * omb2        omb2 = 1 - beta2                  */
/*   d  = sqrt(v) / bc2s + eps              bc2s = sqrt(1 - beta2^t)          */
/*   p  = p - step_size * (m / d)           step_size = lr / (1 - beta1^t)    */
/* grad dtype: 1 = float32, 2 = bfloat16, 3 = float16 (this file's codes).    */
/* ------------------------------------------------------------------------ */
int oracle_adamw(float *p, const void *grad, uint32_t gdtype, float *m, float *v, uint64_t n, float coef,
                 int use_coef, float decay, float omb1, float beta2, float omb2, float bc2s, float eps,
                 float step_size)
{
    const unsigned char *g8 = (const unsigned char *)grad;
    if (gdtype != ORACLE_F32 && gdtype != ORACLE_BF16 && gdtype != ORACLE_F16) return -1;
    for (uint64_t i = 0; i < n; ++i) {
        volatile float g = load_as_float(g8, i, gdtype);
        if (use_coef) g = g * coef;
        volatile float pp = p[i] * decay;
        volatile float diff = g - m[i];
        volatile float mm = m[i] + omb1 * diff;
        volatile float g2 = g * g;
        volatile float t2 = g2 * omb2;
        volatile float vv = v[i] * beta2 + t2;
        volatile float r = sqrtf(vv);
        volatile float den = r / bc2s + eps;
        volatile float q = mm / den;
        volatile float upd = step_size * q;
        p[i] = pp - upd;
        m[i] = mm;
        v[i] = vv;
    }
    return 0;
}
