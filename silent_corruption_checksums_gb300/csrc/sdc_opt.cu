// sdc_opt.cu -- one pass that clips, takes an AdamW step and fingerprints the
// weights it writes.
//
// "Detecting and recovering from silent data corruption on Amazon SageMaker
// HyperPod": `train()` clips the reduced gradient (clip_grad_norm_), skips
// the step when that gradient is NaN/Inf, steps the optimizer, and then the
// weight check fingerprints every replica's weights ("Check 3").  The use
// case trains with AdamW (betas 0.9/0.95, weight decay 0.1, clipping at 1.0).
// Fused here: each element is read once (weight, averaged gradient, both
// moments), updated, written, and its new bits enter the fingerprint, so the
// check's separate re-read of the weights is saved.  It fingerprints the
// values as written; a re-read of stored weights (sdc_fingerprint) remains the
// check for corruption that happens after the write.
//
// The clip coefficient and the skip decision come from the reduced
// gradient's sdc_grad_stats in device memory (written by the post-average
// scan), so the step needs no host round trip.
//
// Float32 arithmetic per element, every operation separately rounded (no
// contraction), with the scalars rounded to float32 on the host:
//   g = grad * coef; p = p * decay; m = m + omb1 * (g - m);
//   v = v * beta2 + (g * g) * omb2; d = sqrt(v) / bc2s + eps;
//   p = p - step_size * (m / d)
#include <cuda_fp16.h>

#include <cmath>
#include <new>

#include "sdc_internal.cuh"

struct sdc_opt_state {
    int device = -1;
    const sdc_plan *plan = nullptr;
    uint32_t grad_dtype = 0;
    struct Ptrs {
        uint64_t g, m, v;
    };
    Ptrs *d_ptrs = nullptr;  // one per plan descriptor
};

namespace sdc {

namespace {

struct AdamK {
    float decay, omb1, beta2, omb2, bc2s, eps, step_size, max_norm;
    uint32_t use_clip;
};

__device__ __forceinline__ void adam_elem(float &p, float g, float &m, float &v, const AdamK &k, float coef,
                                          bool use_coef) {
    if (use_coef) g = __fmul_rn(g, coef);
    const float pp = __fmul_rn(p, k.decay);
    const float mm = __fadd_rn(m, __fmul_rn(k.omb1, __fsub_rn(g, m)));
    const float vv = __fadd_rn(__fmul_rn(v, k.beta2), __fmul_rn(__fmul_rn(g, g), k.omb2));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(vv), k.bc2s), k.eps);
    p = __fsub_rn(pp, __fmul_rn(k.step_size, __fdiv_rn(mm, den)));
    m = mm;
    v = vv;
}

template <int GDT>
__device__ __forceinline__ float grad_at(uint64_t g, uint64_t i) {
    if (GDT == SDC_DTYPE_F32) return ((const float *)g)[i];
    const unsigned short h = ((const unsigned short *)g)[i];
    if (GDT == SDC_DTYPE_BF16) return __uint_as_float((uint32_t)h << 16);
    return __half2float(__ushort_as_half(h));
}

// Four gradients of a vector: 16 bytes (f32) or 8 bytes (bf16/f16).
template <int GDT>
__device__ __forceinline__ float4 grad4(uint64_t gaddr) {
    if (GDT == SDC_DTYPE_F32) return *(const float4 *)gaddr;
    const uint2 w = *(const uint2 *)gaddr;
    float4 r;
    if (GDT == SDC_DTYPE_BF16) {
        r.x = __uint_as_float(w.x << 16);
        r.y = __uint_as_float(w.x & 0xFFFF0000u);
        r.z = __uint_as_float(w.y << 16);
        r.w = __uint_as_float(w.y & 0xFFFF0000u);
    } else {
        r.x = __half2float(__ushort_as_half((unsigned short)(w.x & 0xFFFFu)));
        r.y = __half2float(__ushort_as_half((unsigned short)(w.x >> 16)));
        r.z = __half2float(__ushort_as_half((unsigned short)(w.y & 0xFFFFu)));
        r.w = __half2float(__ushort_as_half((unsigned short)(w.y >> 16)));
    }
    return r;
}

// Scalar element j of a chunk (element index o0 + j of its tensor): update
// (when `apply`) and fingerprint contribution of the resulting weight bits.
template <int GDT>
__device__ __forceinline__ void adam_scalar(uint64_t pbase, const sdc_opt_state::Ptrs &op, uint64_t idx, uint64_t j,
                                            const AdamK &k, float coef, bool use_coef, bool apply, uint64_t &S,
                                            uint64_t &W) {
    float *pp = (float *)pbase + idx;
    float p = *pp;
    if (apply) {
        float *mp = (float *)op.m + idx;
        float *vp = (float *)op.v + idx;
        float m = *mp, v = *vp;
        adam_elem(p, grad_at<GDT>(op.g, idx), m, v, k, coef, use_coef);
        *pp = p;
        *mp = m;
        *vp = v;
    }
    const uint64_t b = (uint64_t)(int64_t)__float_as_int(p);
    S += b;
    W += (j + 1) * b;
}

template <int GDT>
__device__ __forceinline__ void adam_chunk(const Chunk &ch, const DescDev &dd, const sdc_opt_state::Ptrs &op,
                                           uint32_t lane, const AdamK &k, float coef, bool use_coef, bool apply,
                                           uint64_t &S, uint64_t &W) {
    constexpr uint32_t GS = GDT == SDC_DTYPE_F32 ? 4u : 2u;
    const uint64_t o0 = (ch.addr - dd.ptr) >> 2;
    const uint32_t nel = ch.nbytes >> 2;
    uint32_t hel = (uint32_t)(((16u - (uint32_t)(ch.addr & 15u)) & 15u) >> 2);
    if (hel > nel) hel = nel;
    const uint64_t ob = o0 + hel;  // first element of the aligned body
    const bool vec_ok = ((op.m + 4 * ob) & 15u) == 0 && ((op.v + 4 * ob) & 15u) == 0 &&
                        ((op.g + GS * ob) & (GS == 4 ? 15u : 7u)) == 0;
    S = 0;
    W = 0;
    if (!vec_ok) {  // moments or gradient not co-aligned with the weights: element by element
        for (uint32_t j = lane; j < nel; j += 32)
            adam_scalar<GDT>(dd.ptr, op, o0 + j, j, k, coef, use_coef, apply, S, W);
        return;
    }
    const uint32_t nvec = (nel - hel) >> 2;
    const uint32_t tail = nel - hel - (nvec << 2);
    if (lane < hel) adam_scalar<GDT>(dd.ptr, op, o0 + lane, lane, k, coef, use_coef, apply, S, W);
    if (lane >= 16 && lane - 16 < tail) {
        const uint32_t j = hel + (nvec << 2) + (lane - 16);
        adam_scalar<GDT>(dd.ptr, op, o0 + j, j, k, coef, use_coef, apply, S, W);
    }
    float4 *pv = (float4 *)(dd.ptr + 4 * ob);
    float4 *mv = (float4 *)(op.m + 4 * ob);
    float4 *vv = (float4 *)(op.v + 4 * ob);
    const uint64_t gb = op.g + GS * ob;
    for (uint32_t vi = lane; vi < nvec; vi += 32) {
        float4 p = pv[vi];
        if (apply) {
            float4 m = mv[vi], v = vv[vi];
            const float4 g = grad4<GDT>(gb + (uint64_t)vi * 4 * GS);
            adam_elem(p.x, g.x, m.x, v.x, k, coef, use_coef);
            adam_elem(p.y, g.y, m.y, v.y, k, coef, use_coef);
            adam_elem(p.z, g.z, m.z, v.z, k, coef, use_coef);
            adam_elem(p.w, g.w, m.w, v.w, k, coef, use_coef);
            pv[vi] = p;
            mv[vi] = m;
            vv[vi] = v;
        }
        const int64_t a = __float_as_int(p.x), b = __float_as_int(p.y), c = __float_as_int(p.z),
                      d = __float_as_int(p.w);
        const uint64_t s = (uint64_t)(a + b + c + d);
        const uint64_t j0 = hel + 4ull * vi;  // chunk-local index of the vector's first element
        S += s;
        W += (j0 + 1) * s + (uint64_t)(b + 2 * c + 3 * d);
    }
}

__global__ void __launch_bounds__(kScanBlock) adamw_fp_kernel(const Chunk *__restrict__ chunks, uint64_t n_chunks,
                                                              const DescDev *__restrict__ descs,
                                                              const sdc_opt_state::Ptrs *__restrict__ ptrs, AdamK k,
                                                              uint32_t gdt, const sdc_grad_stats *__restrict__ post,
                                                              FpPartial *__restrict__ partials) {
    // the page's gate and clip: skip the step on the reduced-gradient alarm,
    // else scale the gradient by min(1, max_norm / (norm + 1e-6)) in float32
    bool apply = true, use_coef = false;
    float coef = 1.0f;
    if (post) {
        apply = post->nonfinite_fp32 == 0;
        if (k.use_clip && apply) {
            use_coef = true;
            coef = fminf(__fdiv_rn(k.max_norm, __fadd_rn(__double2float_rn(post->norm), 1e-6f)), 1.0f);
        }
    }
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t c = warp; c < n_chunks; c += nwarps) {
        const Chunk ch = chunks[c];
        const uint32_t d = chunk_desc(ch.tag);
        const DescDev dd = descs[d];
        const sdc_opt_state::Ptrs op = ptrs[d];
        uint64_t S, W;
        switch (gdt) {
            case SDC_DTYPE_F32: adam_chunk<SDC_DTYPE_F32>(ch, dd, op, lane, k, coef, use_coef, apply, S, W); break;
            case SDC_DTYPE_BF16: adam_chunk<SDC_DTYPE_BF16>(ch, dd, op, lane, k, coef, use_coef, apply, S, W); break;
            default: adam_chunk<SDC_DTYPE_F16>(ch, dd, op, lane, k, coef, use_coef, apply, S, W); break;
        }
        S = warp_sum_u64(S);
        W = warp_sum_u64(W);
        if (lane == 0) partials[c] = FpPartial{S, W};
    }
}

}  // namespace

}  // namespace sdc

using namespace sdc;

extern "C" {

sdc_status sdc_opt_state_create(const sdc_plan *plan, const void *const *host_grads, uint32_t grad_dtype,
                                void *const *host_exp_avg, void *const *host_exp_avg_sq, sdc_opt_state **out) {
    if (!out) return fail(SDC_ERR_NULL, "out is NULL");
    *out = nullptr;
    if (!plan) return fail(SDC_ERR_NULL, "plan is NULL");
    if (grad_dtype != SDC_DTYPE_F32 && grad_dtype != SDC_DTYPE_BF16 && grad_dtype != SDC_DTYPE_F16)
        return fail(SDC_ERR_BAD_DTYPE, "grad_dtype must be F32, BF16 or F16");
    if (plan->n_desc && (!host_grads || !host_exp_avg || !host_exp_avg_sq))
        return fail(SDC_ERR_NULL, "NULL pointer table");
    sdc_status st = check_plan_device(plan);
    if (st != SDC_OK) return st;
    const uint32_t gs = grad_dtype == SDC_DTYPE_F32 ? 4 : 2;
    std::vector<sdc_opt_state::Ptrs> ptrs(plan->n_desc);
    for (uint64_t d = 0; d < plan->n_desc; ++d) {
        const sdc_tensor_desc &x = plan->descs[d];
        if (x.dtype != SDC_DTYPE_F32) return fail(SDC_ERR_BAD_DTYPE, "the plan's weights must be F32");
        const uint64_t k = d % plan->T;
        const void *g = host_grads[k];
        const void *m = host_exp_avg[d];
        const void *v = host_exp_avg_sq[d];
        const std::string w = "descriptor " + std::to_string(d);
        if (x.numel) {
            if ((uint64_t)g % gs || (uint64_t)m % 4 || (uint64_t)v % 4)
                return fail(SDC_ERR_BAD_POINTER, w + ": gradient or moment not aligned to its element size");
            st = check_device_range(g, x.numel * gs, plan->device, (w + " gradient").c_str());
            if (st == SDC_OK) st = check_device_range(m, x.numel * 4, plan->device, (w + " exp_avg").c_str());
            if (st == SDC_OK) st = check_device_range(v, x.numel * 4, plan->device, (w + " exp_avg_sq").c_str());
            if (st != SDC_OK) return st;
        }
        ptrs[d] = sdc_opt_state::Ptrs{(uint64_t)g, (uint64_t)m, (uint64_t)v};
    }
    sdc_opt_state *s = new (std::nothrow) sdc_opt_state();
    if (!s) return fail(SDC_ERR_BAD_ARG, "out of host memory");
    s->device = plan->device;
    s->plan = plan;
    s->grad_dtype = grad_dtype;
    if (!ptrs.empty()) {
        cudaError_t e = cudaMalloc((void **)&s->d_ptrs, ptrs.size() * sizeof(sdc_opt_state::Ptrs));
        if (e == cudaSuccess)
            e = cudaMemcpy(s->d_ptrs, ptrs.data(), ptrs.size() * sizeof(sdc_opt_state::Ptrs), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            if (s->d_ptrs) cudaFree(s->d_ptrs);
            delete s;
            return cuda_fail(e, "optimizer pointer table");
        }
    }
    *out = s;
    return SDC_OK;
}

sdc_status sdc_opt_state_destroy(sdc_opt_state *state) {
    if (!state) return SDC_OK;
    if (state->d_ptrs) cudaFree(state->d_ptrs);
    delete state;
    return SDC_OK;
}

sdc_status sdc_adamw_fingerprint(const sdc_plan *plan, const sdc_opt_state *state, const sdc_adamw_hparams *hp,
                                 const sdc_grad_stats *d_post, uint64_t *d_fp_out, void *d_ws, size_t ws_bytes,
                                 sdc_stream_t stream) {
    if (!plan || !state || !hp) return fail(SDC_ERR_NULL, "NULL plan, state or hyperparameters");
    if (state->plan != plan) return fail(SDC_ERR_BAD_ARG, "the optimizer state belongs to another plan");
    sdc_status st = check_plan_device(plan);
    if (st != SDC_OK) return st;
    if (plan->n_desc && !d_fp_out) return fail(SDC_ERR_NULL, "d_fp_out is NULL");
    if (hp->step == 0) return fail(SDC_ERR_BAD_ARG, "step counts from 1");
    if (hp->clip && !d_post) return fail(SDC_ERR_NULL, "clipping needs the reduced gradient's stats");
    if (d_post) {
        st = check_device_range(d_post, sizeof(sdc_grad_stats), plan->device, "d_post");
        if (st != SDC_OK) return st;
    }
    if (plan->n_chunks && (!d_ws || ws_bytes < plan->n_chunks * sizeof(FpPartial)))
        return fail(SDC_ERR_WS_TOO_SMALL, "workspace smaller than sdc_workspace_size(plan)");
    st = check_spans({{d_fp_out, plan->n_desc * 16, "d_fp_out"},
                      {d_ws, plan->n_chunks * sizeof(FpPartial), "d_ws"}},
                     plan->device);
    if (st != SDC_OK) return st;
    // float32 scalars, each formed in double from the float32 inputs and rounded once
    const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, t = (double)hp->step;
    AdamK k;
    k.decay = (float)(1.0 - lr * (double)hp->weight_decay);
    k.omb1 = (float)(1.0 - b1);
    k.beta2 = hp->beta2;
    k.omb2 = (float)(1.0 - b2);
    k.bc2s = (float)std::sqrt(1.0 - std::pow(b2, t));
    k.eps = hp->eps;
    k.step_size = (float)(lr / (1.0 - std::pow(b1, t)));
    k.max_norm = hp->max_grad_norm;
    k.use_clip = hp->clip ? 1u : 0u;
    cudaStream_t s = (cudaStream_t)stream;
    FpPartial *part = (FpPartial *)d_ws;
    cudaError_t e = cudaSuccess;
    if (plan->n_chunks) {
        uint64_t grid = (uint64_t)sm_count(plan->device) * 4;
        const uint64_t need = (plan->n_chunks * 32 + kScanBlock - 1) / kScanBlock;
        if (need < grid) grid = need;
        adamw_fp_kernel<<<(unsigned)grid, kScanBlock, 0, s>>>(plan->d_chunks, plan->n_chunks, plan->d_descs,
                                                             state->d_ptrs, k, state->grad_dtype, d_post, part);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_fp_combine(plan, part, d_fp_out, s);
    return e == cudaSuccess ? SDC_OK : cuda_fail(e, "sdc_adamw_fingerprint launch");
}

}  // extern "C"
