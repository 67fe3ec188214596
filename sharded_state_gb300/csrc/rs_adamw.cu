// rs_adamw.cu -- reduce-scatter of N virtual ranks' gradients fused with
// mixed-precision AdamW on every rank's shard, and optimizer-state init.
//
// "Scaling data parallel", sections 9.1-9.3: the reduce-scatter leaves rank s
// the sum over ranks of its 1/N of the gradient; divided by N it is the
// data-parallel mean.  Each rank then updates the fp32 master copy and the
// Adam moments of its own shard and casts the result to bf16 ("FSDP1 vs
// FSDP2", mixed precision: the optimizer updates the original dtype, the cast
// happens at the all-gather boundary).
//
// With all N ranks in one HBM, every packed buffer (N gradient buffers,
// master / exp_avg / exp_avg_sq, parameter shards) is indexed by the same
// element index f, so the whole step is one streaming pass: per element it
// reads N gradient values and three fp32 state values and writes three fp32
// state values and one parameter value -- 2N + 26 bytes for bf16.  Nothing is
// reused, so the kernel is bound by HBM bandwidth: it moves 128-bit vectors
// (8 bf16 / 4 fp32 elements) and keeps N + 6 independent loads in flight per
// thread.  The grid has one thread per vector: short-lived CTAs retire in
// address order, so all SMs stream through a narrow, advancing window of HBM,
// which measured 7-8 % faster on GB300 than a persistent grid-stride loop over
// the same vectors.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "device_utils.cuh"
#include "internal.h"

namespace {

struct RankPtrs {
    const void* p[SS_MAX_WORLD];
};

// AdamW coefficients, computed once per call on the host in double and
// rounded to fp32.
struct AdamCoef {
    float decay;         // 1 - lr * wd
    float b1, omb1;      // beta1, 1 - beta1
    float b2, omb2;      // beta2, 1 - beta2
    float step_size;     // lr / (1 - beta1^t)
    float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
    float eps;
};

constexpr int kThreads = 256;

// AdamW update of one element, in fp32.
__device__ __forceinline__ void adamw_elem(float g, float& theta, float& m, float& v,
                                           const AdamCoef& c) {
    theta = __fmul_rn(theta, c.decay);
    m = __fmaf_rn(c.b1, m, __fmul_rn(c.omb1, g));
    v = __fmaf_rn(c.b2, v, __fmul_rn(c.omb2, __fmul_rn(g, g)));
    float denom = __fmaf_rn(__fsqrt_rn(v), c.inv_sqrt_bc2, c.eps);
    theta = __fmaf_rn(-c.step_size, __fdiv_rn(m, denom), theta);
}

// ---------------------------------------------------------------------------
// bf16 gradients / shards: 8 elements per 128-bit vector
// ---------------------------------------------------------------------------

// MASTER == false: no fp32 master copy; theta is the bf16 shard itself, widened,
// updated in fp32 and rounded back (the optimizer-state recipe without master
// weights, "FSDP1 vs FSDP2" ledger: 2 B params + 2 B grads + 8 B moments).
// ACC_IN: last micro-batch of gradient accumulation: the gradient AdamW uses is
// (accum + reduce-scatter) / kdiv.
template <int NR, bool ADAM, bool WRITE_G, bool MASTER = true, bool ACC_IN = false>
__global__ void __launch_bounds__(kThreads, 3)
rs_adamw_bf16_kernel(RankPtrs grads, int N, int64_t vbeg, int64_t nvec, float* __restrict__ master,
                     float* __restrict__ exp_avg, float* __restrict__ exp_avg_sq,
                     uint16_t* __restrict__ shards, float* __restrict__ gout, AdamCoef c,
                     const float* __restrict__ accum, float kdiv) {
    const int n = NR > 0 ? NR : N;
    const float fN = (float)n;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nvec; q += stride) {
        const int64_t f = vbeg + q * 8;  // first element of this vector
        // issue every load of this vector before any arithmetic: N gradient
        // vectors and the six state vectors are all in flight together
        constexpr int kW = NR > 0 ? NR : 8;
        uint4 w[kW];
        const int nfirst = NR > 0 ? NR : (n < 8 ? n : 8);
#pragma unroll
        for (int r = 0; r < kW; ++r)
            if (NR > 0 || r < nfirst)
                w[r] = ss::ld_stream_u4(static_cast<const uint16_t*>(grads.p[r]) + f);
        float4 t0, t1, m0, m1, v0, v1;
        if (ADAM) {
            if (MASTER) {
                t0 = ss::ld_rw_f4(master + f);
                t1 = ss::ld_rw_f4(master + f + 4);
            } else {
                uint4 pw;
                asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(pw.x), "=r"(pw.y), "=r"(pw.z), "=r"(pw.w)
                             : "l"(shards + f));
                t0 = make_float4(ss::bf16_lo(pw.x), ss::bf16_hi(pw.x), ss::bf16_lo(pw.y), ss::bf16_hi(pw.y));
                t1 = make_float4(ss::bf16_lo(pw.z), ss::bf16_hi(pw.z), ss::bf16_lo(pw.w), ss::bf16_hi(pw.w));
            }
            m0 = ss::ld_rw_f4(exp_avg + f);
            m1 = ss::ld_rw_f4(exp_avg + f + 4);
            v0 = ss::ld_rw_f4(exp_avg_sq + f);
            v1 = ss::ld_rw_f4(exp_avg_sq + f + 4);
        }
        float4 a0, a1;
        if (ACC_IN) {
            a0 = ss::ld_rw_f4(accum + f);
            a1 = ss::ld_rw_f4(accum + f + 4);
        }
        // rank-order fp32 sum, starting from rank 0's value
        float s[8] = {ss::bf16_lo(w[0].x), ss::bf16_hi(w[0].x), ss::bf16_lo(w[0].y),
                      ss::bf16_hi(w[0].y), ss::bf16_lo(w[0].z), ss::bf16_hi(w[0].z),
                      ss::bf16_lo(w[0].w), ss::bf16_hi(w[0].w)};
#pragma unroll
        for (int r = 1; r < kW; ++r) {
            if (NR > 0 || r < nfirst) {
                s[0] = __fadd_rn(s[0], ss::bf16_lo(w[r].x));
                s[1] = __fadd_rn(s[1], ss::bf16_hi(w[r].x));
                s[2] = __fadd_rn(s[2], ss::bf16_lo(w[r].y));
                s[3] = __fadd_rn(s[3], ss::bf16_hi(w[r].y));
                s[4] = __fadd_rn(s[4], ss::bf16_lo(w[r].z));
                s[5] = __fadd_rn(s[5], ss::bf16_hi(w[r].z));
                s[6] = __fadd_rn(s[6], ss::bf16_lo(w[r].w));
                s[7] = __fadd_rn(s[7], ss::bf16_hi(w[r].w));
            }
        }
        if (NR == 0) {
            // ranks beyond the first 8 (N > 8), 8 at a time: each batch's
            // loads go out together into the first batch's registers, then
            // add in rank order
            for (int r0 = 8; r0 < n; r0 += 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (r0 + j < n)
                        w[j] = ss::ld_stream_u4(static_cast<const uint16_t*>(grads.p[r0 + j]) + f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (r0 + j < n) {
                        s[0] = __fadd_rn(s[0], ss::bf16_lo(w[j].x));
                        s[1] = __fadd_rn(s[1], ss::bf16_hi(w[j].x));
                        s[2] = __fadd_rn(s[2], ss::bf16_lo(w[j].y));
                        s[3] = __fadd_rn(s[3], ss::bf16_hi(w[j].y));
                        s[4] = __fadd_rn(s[4], ss::bf16_lo(w[j].z));
                        s[5] = __fadd_rn(s[5], ss::bf16_hi(w[j].z));
                        s[6] = __fadd_rn(s[6], ss::bf16_lo(w[j].w));
                        s[7] = __fadd_rn(s[7], ss::bf16_hi(w[j].w));
                    }
                }
            }
        }
        float g[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) g[k] = __fdiv_rn(s[k], fN);
        if (ACC_IN) {
            const float acc[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) g[k] = __fdiv_rn(__fadd_rn(acc[k], g[k]), kdiv);
        }
        if (WRITE_G) {
            ss::st_stream_f4(gout + f, make_float4(g[0], g[1], g[2], g[3]));
            ss::st_stream_f4(gout + f + 4, make_float4(g[4], g[5], g[6], g[7]));
        }
        if (ADAM) {
            float th[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
            float mm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
            float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) adamw_elem(g[k], th[k], mm[k], vv[k], c);
            if (MASTER) {
                ss::st_stream_f4(master + f, make_float4(th[0], th[1], th[2], th[3]));
                ss::st_stream_f4(master + f + 4, make_float4(th[4], th[5], th[6], th[7]));
            }
            ss::st_stream_f4(exp_avg + f, make_float4(mm[0], mm[1], mm[2], mm[3]));
            ss::st_stream_f4(exp_avg + f + 4, make_float4(mm[4], mm[5], mm[6], mm[7]));
            ss::st_stream_f4(exp_avg_sq + f, make_float4(vv[0], vv[1], vv[2], vv[3]));
            ss::st_stream_f4(exp_avg_sq + f + 4, make_float4(vv[4], vv[5], vv[6], vv[7]));
            uint4 p;
            p.x = ss::pack_bf16x2(th[0], th[1]);
            p.y = ss::pack_bf16x2(th[2], th[3]);
            p.z = ss::pack_bf16x2(th[4], th[5]);
            p.w = ss::pack_bf16x2(th[6], th[7]);
            ss::st_stream_u4(shards + f, p);
        }
    }
}

// ---------------------------------------------------------------------------
// fp32 gradients / shards: 4 elements per 128-bit vector
// ---------------------------------------------------------------------------

template <int NR, bool ADAM, bool WRITE_G, bool MASTER = true>
__global__ void __launch_bounds__(kThreads, 3)
rs_adamw_f32_kernel(RankPtrs grads, int N, int64_t vbeg, int64_t nvec, float* __restrict__ master,
                    float* __restrict__ exp_avg, float* __restrict__ exp_avg_sq,
                    float* __restrict__ shards, float* __restrict__ gout, AdamCoef c) {
    const int n = NR > 0 ? NR : N;
    const float fN = (float)n;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nvec; q += stride) {
        const int64_t f = vbeg + q * 4;
        // every load of this vector before any arithmetic, as in the bf16 kernel
        constexpr int kW = NR > 0 ? NR : 8;
        uint4 w[kW];
        const int nfirst = NR > 0 ? NR : (n < 8 ? n : 8);
#pragma unroll
        for (int r = 0; r < kW; ++r)
            if (NR > 0 || r < nfirst) w[r] = ss::ld_stream_u4(static_cast<const float*>(grads.p[r]) + f);
        float4 t, m, v;
        if (ADAM) {
            t = ss::ld_rw_f4(MASTER ? master + f : shards + f);
            m = ss::ld_rw_f4(exp_avg + f);
            v = ss::ld_rw_f4(exp_avg_sq + f);
        }
        float s[4] = {__uint_as_float(w[0].x), __uint_as_float(w[0].y), __uint_as_float(w[0].z),
                      __uint_as_float(w[0].w)};
#pragma unroll
        for (int r = 1; r < kW; ++r) {
            if (NR > 0 || r < nfirst) {
                s[0] = __fadd_rn(s[0], __uint_as_float(w[r].x));
                s[1] = __fadd_rn(s[1], __uint_as_float(w[r].y));
                s[2] = __fadd_rn(s[2], __uint_as_float(w[r].z));
                s[3] = __fadd_rn(s[3], __uint_as_float(w[r].w));
            }
        }
        // ranks beyond the first 8 (N > 8), 8 loads in flight at a time,
        // added in rank order
        for (int r0 = 8; NR == 0 && r0 < n; r0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r0 + j < n) w[j] = ss::ld_stream_u4(static_cast<const float*>(grads.p[r0 + j]) + f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r0 + j < n) {
                    s[0] = __fadd_rn(s[0], __uint_as_float(w[j].x));
                    s[1] = __fadd_rn(s[1], __uint_as_float(w[j].y));
                    s[2] = __fadd_rn(s[2], __uint_as_float(w[j].z));
                    s[3] = __fadd_rn(s[3], __uint_as_float(w[j].w));
                }
            }
        }
        float g[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) g[k] = __fdiv_rn(s[k], fN);
        if (WRITE_G) ss::st_stream_f4(gout + f, make_float4(g[0], g[1], g[2], g[3]));
        if (ADAM) {
            float th[4] = {t.x, t.y, t.z, t.w}, mm[4] = {m.x, m.y, m.z, m.w},
                  vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw_elem(g[k], th[k], mm[k], vv[k], c);
            float4 tn = make_float4(th[0], th[1], th[2], th[3]);
            if (MASTER) ss::st_stream_f4(master + f, tn);
            ss::st_stream_f4(exp_avg + f, make_float4(mm[0], mm[1], mm[2], mm[3]));
            ss::st_stream_f4(exp_avg_sq + f, make_float4(vv[0], vv[1], vv[2], vv[3]));
            ss::st_stream_f4(shards + f, tn);
        }
    }
}

// ---------------------------------------------------------------------------
// scalar path for the unaligned head / tail of a range (< 8 elements each)
// ---------------------------------------------------------------------------

__global__ void rs_adamw_scalar_kernel(RankPtrs grads, int N, int eb, int64_t a0, int64_t a1,
                                       int64_t b0, int64_t b1, float* master, float* exp_avg,
                                       float* exp_avg_sq, void* shards, float* gout, AdamCoef c,
                                       int adam) {
    int64_t k = threadIdx.x;
    int64_t na = a1 - a0;
    int64_t f;
    if (k < na)
        f = a0 + k;
    else if (k - na < b1 - b0)
        f = b0 + (k - na);
    else
        return;
    float s;
    if (eb == 2) {
        s = ss::bf16_to_f32(static_cast<const uint16_t*>(grads.p[0])[f]);
        for (int r = 1; r < N; ++r)
            s = __fadd_rn(s, ss::bf16_to_f32(static_cast<const uint16_t*>(grads.p[r])[f]));
    } else {
        s = static_cast<const float*>(grads.p[0])[f];
        for (int r = 1; r < N; ++r) s = __fadd_rn(s, static_cast<const float*>(grads.p[r])[f]);
    }
    float g = __fdiv_rn(s, (float)N);
    if (gout) gout[f] = g;
    if (adam) {
        float th = master ? master[f]
                          : (eb == 2 ? ss::bf16_to_f32(static_cast<const uint16_t*>(shards)[f])
                                     : static_cast<const float*>(shards)[f]);
        float m = exp_avg[f], v = exp_avg_sq[f];
        adamw_elem(g, th, m, v, c);
        if (master) master[f] = th;
        exp_avg[f] = m;
        exp_avg_sq[f] = v;
        if (eb == 2)
            static_cast<uint16_t*>(shards)[f] = ss::f32_to_bf16(th);
        else
            static_cast<float*>(shards)[f] = th;
    }
}

// ---------------------------------------------------------------------------
// optimizer state init: master = widen(shard), moments = 0
// ---------------------------------------------------------------------------

__global__ void init_master_kernel(const void* shards, int eb, int64_t lo, int64_t hi,
                                   float* master, float* m, float* v) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t f = lo + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; f < hi; f += stride) {
        master[f] = eb == 2 ? ss::bf16_to_f32(static_cast<const uint16_t*>(shards)[f])
                            : static_cast<const float*>(shards)[f];
        m[f] = 0.0f;
        v[f] = 0.0f;
    }
}

// The same for 16-byte vectors of bf16 shards: elements [8*vlo, 8*vhi), one
// vector per thread (every buffer 16-byte aligned there).
__global__ void __launch_bounds__(kThreads)
init_master_bf16_vec_kernel(const uint16_t* __restrict__ shards, int64_t vlo, int64_t nvec,
                            float* __restrict__ master, float* __restrict__ m,
                            float* __restrict__ v) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nvec; q += stride) {
        const int64_t f = 8 * (vlo + q);
        const uint4 w = ss::ld_stream_u4(shards + f);
        ss::st_stream_f4(master + f, make_float4(ss::bf16_lo(w.x), ss::bf16_hi(w.x), ss::bf16_lo(w.y),
                                                 ss::bf16_hi(w.y)));
        ss::st_stream_f4(master + f + 4, make_float4(ss::bf16_lo(w.z), ss::bf16_hi(w.z),
                                                     ss::bf16_lo(w.w), ss::bf16_hi(w.w)));
        ss::st_stream_f4(m + f, z);
        ss::st_stream_f4(m + f + 4, z);
        ss::st_stream_f4(v + f, z);
        ss::st_stream_f4(v + f + 4, z);
    }
}

// ---------------------------------------------------------------------------
// dispatch
// ---------------------------------------------------------------------------

using BF16Kernel = void (*)(RankPtrs, int, int64_t, int64_t, float*, float*, float*, uint16_t*,
                            float*, AdamCoef, const float*, float);
using F32Kernel = void (*)(RankPtrs, int, int64_t, int64_t, float*, float*, float*, float*, float*,
                           AdamCoef);

template <bool ADAM, bool WG, bool M = true, bool A = false>
BF16Kernel pick_bf16(int N) {
    switch (N) {
        case 1: return rs_adamw_bf16_kernel<1, ADAM, WG, M, A>;
        case 2: return rs_adamw_bf16_kernel<2, ADAM, WG, M, A>;
        case 3: return rs_adamw_bf16_kernel<3, ADAM, WG, M, A>;
        case 4: return rs_adamw_bf16_kernel<4, ADAM, WG, M, A>;
        case 5: return rs_adamw_bf16_kernel<5, ADAM, WG, M, A>;
        case 6: return rs_adamw_bf16_kernel<6, ADAM, WG, M, A>;
        case 7: return rs_adamw_bf16_kernel<7, ADAM, WG, M, A>;
        case 8: return rs_adamw_bf16_kernel<8, ADAM, WG, M, A>;
        default: return rs_adamw_bf16_kernel<0, ADAM, WG, M, A>;
    }
}

template <bool ADAM, bool WG, bool M = true>
F32Kernel pick_f32(int N) {
    switch (N) {
        case 1: return rs_adamw_f32_kernel<1, ADAM, WG, M>;
        case 2: return rs_adamw_f32_kernel<2, ADAM, WG, M>;
        case 3: return rs_adamw_f32_kernel<3, ADAM, WG, M>;
        case 4: return rs_adamw_f32_kernel<4, ADAM, WG, M>;
        case 5: return rs_adamw_f32_kernel<5, ADAM, WG, M>;
        case 6: return rs_adamw_f32_kernel<6, ADAM, WG, M>;
        case 7: return rs_adamw_f32_kernel<7, ADAM, WG, M>;
        case 8: return rs_adamw_f32_kernel<8, ADAM, WG, M>;
        default: return rs_adamw_f32_kernel<0, ADAM, WG, M>;
    }
}

// One thread per vector (the kernels' grid-stride loop only runs more than
// once beyond 2^31 - 1 CTAs).
int grid_for(int64_t nvec) {
    const int64_t want = (nvec + kThreads - 1) / kThreads;
    const int64_t cap = 0x7FFFFFFF;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

AdamCoef make_coef(const ss_adamw* hp) {
    AdamCoef c;
    std::memset(&c, 0, sizeof c);
    if (!hp) return c;
    const double t = (double)hp->step;
    const double bc1 = 1.0 - std::pow(hp->beta1, t);
    const double bc2 = 1.0 - std::pow(hp->beta2, t);
    c.decay = (float)(1.0 - hp->lr * hp->weight_decay);
    c.b1 = (float)hp->beta1;
    c.omb1 = (float)(1.0 - hp->beta1);
    c.b2 = (float)hp->beta2;
    c.omb2 = (float)(1.0 - hp->beta2);
    c.step_size = (float)(hp->lr / bc1);
    c.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
    c.eps = (float)hp->eps;
    return c;
}

}  // namespace

extern "C" {

int fsdp_reduce_scatter_adamw(const ss_plan* plan, const void* const* rank_grads, float* master,
                              float* exp_avg, float* exp_avg_sq, void* param_shards,
                              const ss_adamw* hp, float* reduced_grad_out, int group,
                              ss_stream_t stream) {
    if (!plan || !rank_grads) return SS_EINVAL;
    if (!plan->has_dev) return SS_ENODEVICE;
    if (int drc = ss::check_device(plan)) return drc;
    int64_t lo, hi;
    if (!ss::group_range(plan, group, &lo, &hi)) return SS_EINVAL;
    const int N = plan->N;
    if (hp) {
        if (!exp_avg || !exp_avg_sq || !param_shards) return SS_EINVAL;
        if (hp->step < 1 || !(hp->beta1 >= 0.0 && hp->beta1 < 1.0) ||
            !(hp->beta2 >= 0.0 && hp->beta2 < 1.0) || !(hp->eps >= 0.0) || !std::isfinite(hp->lr) ||
            !std::isfinite(hp->weight_decay))
            return SS_EINVAL;
    } else if (!reduced_grad_out) {
        return SS_EINVAL;
    }
    RankPtrs rp;
    std::memset(&rp, 0, sizeof rp);
    for (int r = 0; r < N; ++r) {
        if (!rank_grads[r] && hi > lo) return SS_EINVAL;
        if (!ss::aligned(rank_grads[r], 16)) return SS_EALIGN;
        rp.p[r] = rank_grads[r];
    }
    const void* bufs[5] = {master, exp_avg, exp_avg_sq, param_shards, reduced_grad_out};
    for (const void* b : bufs)
        if (b && !ss::aligned(b, 16)) return SS_EALIGN;
    if (hi <= lo) return SS_OK;

    const AdamCoef c = make_coef(hp);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int vw = plan->eb == 2 ? 8 : 4;  // elements per 128-bit vector
    const int64_t vbeg = (lo + vw - 1) / vw * vw;
    const int64_t vend = hi / vw * vw;
    const bool adam = hp != nullptr, wg = reduced_grad_out != nullptr;
    const bool with_master = master != nullptr;

    if (vend > vbeg) {
        const int64_t nvec = (vend - vbeg) / vw;
        if (plan->eb == 2) {
            BF16Kernel fn = !adam ? pick_bf16<false, true>(N)
                            : with_master ? (wg ? pick_bf16<true, true>(N) : pick_bf16<true, false>(N))
                                          : (wg ? pick_bf16<true, true, false>(N)
                                                : pick_bf16<true, false, false>(N));
            int grid = grid_for(nvec);
            fn<<<grid, kThreads, 0, st>>>(rp, N, vbeg, nvec, master, exp_avg, exp_avg_sq,
                                          static_cast<uint16_t*>(param_shards), reduced_grad_out, c,
                                          nullptr, 1.0f);
        } else {
            F32Kernel fn = !adam ? pick_f32<false, true>(N)
                           : with_master ? (wg ? pick_f32<true, true>(N) : pick_f32<true, false>(N))
                                         : (wg ? pick_f32<true, true, false>(N)
                                               : pick_f32<true, false, false>(N));
            int grid = grid_for(nvec);
            fn<<<grid, kThreads, 0, st>>>(rp, N, vbeg, nvec, master, exp_avg, exp_avg_sq,
                                          static_cast<float*>(param_shards), reduced_grad_out, c);
        }
        int rc = ss::check_launch();
        if (rc) return rc;
    }
    // unaligned head [lo, min(vbeg, hi)) and tail [max(vend, lo), hi): fewer than 2*vw elements
    int64_t a0 = lo, a1 = vbeg < hi ? vbeg : hi;
    int64_t b0 = vend > a1 ? vend : a1, b1 = hi;
    if (vend <= vbeg) {  // range shorter than a vector: all of it goes through the scalar path
        a1 = hi;
        b0 = b1 = hi;
    }
    if (a1 > a0 || b1 > b0) {
        rs_adamw_scalar_kernel<<<1, 32, 0, st>>>(rp, N, plan->eb, a0, a1, b0, b1, master, exp_avg,
                                                 exp_avg_sq, param_shards, reduced_grad_out, c,
                                                 adam ? 1 : 0);
        int rc = ss::check_launch();
        if (rc) return rc;
    }
    return SS_OK;
}

int fsdp_init_master(const ss_plan* plan, const void* param_shards, float* master, float* exp_avg,
                     float* exp_avg_sq, int group, ss_stream_t stream) {
    if (!plan || !param_shards || !master || !exp_avg || !exp_avg_sq) return SS_EINVAL;
    if (!plan->has_dev) return SS_ENODEVICE;
    if (int drc = ss::check_device(plan)) return drc;
    int64_t lo, hi;
    if (!ss::group_range(plan, group, &lo, &hi)) return SS_EINVAL;
    const void* bufs[4] = {param_shards, master, exp_avg, exp_avg_sq};
    for (const void* b : bufs)
        if (!ss::aligned(b, 16)) return SS_EALIGN;
    if (hi <= lo) return SS_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t cap = (int64_t)ss::num_sms() * 8;
    auto scalar = [&](int64_t a0, int64_t a1) -> int {
        if (a1 <= a0) return SS_OK;
        const int64_t blocks = (a1 - a0 + kThreads - 1) / kThreads;
        init_master_kernel<<<(int)(blocks < cap ? blocks : cap), kThreads, 0, st>>>(
            param_shards, plan->eb, a0, a1, master, exp_avg, exp_avg_sq);
        return ss::check_launch();
    };
    if (plan->eb != 2) return scalar(lo, hi);
    // bf16: 16-byte vectors over the 8-aligned middle, scalar head and tail
    const int64_t vlo = (lo + 7) / 8, vhi = hi / 8;
    if (vhi <= vlo) return scalar(lo, hi);
    int rc = scalar(lo, 8 * vlo);
    if (rc) return rc;
    init_master_bf16_vec_kernel<<<grid_for(vhi - vlo), kThreads, 0, st>>>(
        static_cast<const uint16_t*>(param_shards), vlo, vhi - vlo, master, exp_avg, exp_avg_sq);
    rc = ss::check_launch();
    if (rc) return rc;
    return scalar(8 * vhi, hi);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gradient accumulation over micro-batches
// ---------------------------------------------------------------------------
//
// "Scaling data parallel", section 5 (gradient accumulation / no_sync) with
// section 9.2 (ZeRO-2 keeps an fp32 gradient for its own 1/N and adds each
// reduce-scatter into it): with k micro-batches per optimizer step,
//   acc_1 = RS_1,  acc_j = acc_{j-1} + RS_j   (fp32, micro-batch order)
//   g = acc_k / k, then AdamW as in fsdp_reduce_scatter_adamw.
// Micro-batches 1..k-1 run rs_accum_kernel (2N + 4 / 2N + 8 bytes per
// element); micro-batch k runs the RS+AdamW kernel with the accumulator as an
// extra input (2N + 4 + 26 bytes), so the accumulator is never re-read.

namespace {

template <int NR, bool FIRST>
__global__ void __launch_bounds__(kThreads)
rs_accum_kernel(RankPtrs grads, int N, int64_t vbeg, int64_t nvec, float* __restrict__ accum) {
    const int n = NR > 0 ? NR : N;
    const float fN = (float)n;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nvec; q += stride) {
        const int64_t f = vbeg + q * 8;
        constexpr int kW = NR > 0 ? NR : 8;
        uint4 w[kW];
        const int nfirst = NR > 0 ? NR : (n < 8 ? n : 8);
#pragma unroll
        for (int r = 0; r < kW; ++r)
            if (NR > 0 || r < nfirst)
                w[r] = ss::ld_stream_u4(static_cast<const uint16_t*>(grads.p[r]) + f);
        float4 a0, a1;
        if (!FIRST) {
            a0 = ss::ld_rw_f4(accum + f);
            a1 = ss::ld_rw_f4(accum + f + 4);
        }
        float s[8] = {ss::bf16_lo(w[0].x), ss::bf16_hi(w[0].x), ss::bf16_lo(w[0].y),
                      ss::bf16_hi(w[0].y), ss::bf16_lo(w[0].z), ss::bf16_hi(w[0].z),
                      ss::bf16_lo(w[0].w), ss::bf16_hi(w[0].w)};
#pragma unroll
        for (int r = 1; r < kW; ++r) {
            if (NR > 0 || r < nfirst) {
                s[0] = __fadd_rn(s[0], ss::bf16_lo(w[r].x));
                s[1] = __fadd_rn(s[1], ss::bf16_hi(w[r].x));
                s[2] = __fadd_rn(s[2], ss::bf16_lo(w[r].y));
                s[3] = __fadd_rn(s[3], ss::bf16_hi(w[r].y));
                s[4] = __fadd_rn(s[4], ss::bf16_lo(w[r].z));
                s[5] = __fadd_rn(s[5], ss::bf16_hi(w[r].z));
                s[6] = __fadd_rn(s[6], ss::bf16_lo(w[r].w));
                s[7] = __fadd_rn(s[7], ss::bf16_hi(w[r].w));
            }
        }
        // ranks beyond the first 8 (N > 8), 8 loads in flight at a time,
        // added in rank order
        for (int r0 = 8; NR == 0 && r0 < n; r0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (r0 + j < n) w[j] = ss::ld_stream_u4(static_cast<const uint16_t*>(grads.p[r0 + j]) + f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r0 + j < n) {
                    s[0] = __fadd_rn(s[0], ss::bf16_lo(w[j].x));
                    s[1] = __fadd_rn(s[1], ss::bf16_hi(w[j].x));
                    s[2] = __fadd_rn(s[2], ss::bf16_lo(w[j].y));
                    s[3] = __fadd_rn(s[3], ss::bf16_hi(w[j].y));
                    s[4] = __fadd_rn(s[4], ss::bf16_lo(w[j].z));
                    s[5] = __fadd_rn(s[5], ss::bf16_hi(w[j].z));
                    s[6] = __fadd_rn(s[6], ss::bf16_lo(w[j].w));
                    s[7] = __fadd_rn(s[7], ss::bf16_hi(w[j].w));
                }
            }
        }
        float o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = __fdiv_rn(s[k], fN);
        if (!FIRST) {
            const float acc[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = __fadd_rn(acc[k], o[k]);
        }
        ss::st_stream_f4(accum + f, make_float4(o[0], o[1], o[2], o[3]));
        ss::st_stream_f4(accum + f + 4, make_float4(o[4], o[5], o[6], o[7]));
    }
}

// Head / tail elements (< 8 each side) of every accumulation mode.
// mode 0: acc = RS; 1: acc += RS; 2: g = (acc + RS) / kdiv, AdamW.
__global__ void rs_accum_scalar_kernel(RankPtrs grads, int N, int64_t a0, int64_t a1, int64_t b0,
                                       int64_t b1, float* accum, int mode, float kdiv,
                                       float* master, float* exp_avg, float* exp_avg_sq,
                                       uint16_t* shards, float* gout, AdamCoef c) {
    const int64_t k = threadIdx.x, na = a1 - a0;
    int64_t f;
    if (k < na)
        f = a0 + k;
    else if (k - na < b1 - b0)
        f = b0 + (k - na);
    else
        return;
    float s = ss::bf16_to_f32(static_cast<const uint16_t*>(grads.p[0])[f]);
    for (int r = 1; r < N; ++r)
        s = __fadd_rn(s, ss::bf16_to_f32(static_cast<const uint16_t*>(grads.p[r])[f]));
    const float rs = __fdiv_rn(s, (float)N);
    if (mode == 0) {
        accum[f] = rs;
        return;
    }
    if (mode == 1) {
        accum[f] = __fadd_rn(accum[f], rs);
        return;
    }
    const float g = __fdiv_rn(__fadd_rn(accum[f], rs), kdiv);
    if (gout) gout[f] = g;
    float th = master ? master[f] : ss::bf16_to_f32(shards[f]);
    float m = exp_avg[f], v = exp_avg_sq[f];
    adamw_elem(g, th, m, v, c);
    if (master) master[f] = th;
    exp_avg[f] = m;
    exp_avg_sq[f] = v;
    shards[f] = ss::f32_to_bf16(th);
}

using AccKernel = void (*)(RankPtrs, int, int64_t, int64_t, float*);

template <bool FIRST>
AccKernel pick_acc(int N) {
    switch (N) {
        case 2: return rs_accum_kernel<2, FIRST>;
        case 4: return rs_accum_kernel<4, FIRST>;
        case 8: return rs_accum_kernel<8, FIRST>;
        default: return rs_accum_kernel<0, FIRST>;
    }
}

}  // namespace

extern "C" int fsdp_reduce_scatter_accumulate(const ss_plan* plan, const void* const* rank_grads,
                                              float* accum, int micro_step, int num_micro,
                                              float* master, float* exp_avg, float* exp_avg_sq,
                                              void* param_shards, const ss_adamw* hp,
                                              float* reduced_grad_out, int group,
                                              ss_stream_t stream) {
    if (!plan || !rank_grads) return SS_EINVAL;
    if (!plan->has_dev) return SS_ENODEVICE;
    if (int drc = ss::check_device(plan)) return drc;
    if (plan->eb != 2) return SS_EINVAL;
    if (num_micro < 1 || micro_step < 0 || micro_step >= num_micro) return SS_EINVAL;
    const bool last = micro_step == num_micro - 1;
    if (last && num_micro == 1)  // one micro-batch: the plain fused step
        return fsdp_reduce_scatter_adamw(plan, rank_grads, master, exp_avg, exp_avg_sq, param_shards,
                                         hp, reduced_grad_out, group, stream);
    if (!accum) return SS_EINVAL;
    if (last) {
        if (!hp || !exp_avg || !exp_avg_sq || !param_shards) return SS_EINVAL;
        if (hp->step < 1 || !(hp->beta1 >= 0.0 && hp->beta1 < 1.0) ||
            !(hp->beta2 >= 0.0 && hp->beta2 < 1.0) || !(hp->eps >= 0.0) || !std::isfinite(hp->lr) ||
            !std::isfinite(hp->weight_decay))
            return SS_EINVAL;
    }
    int64_t lo, hi;
    if (!ss::group_range(plan, group, &lo, &hi)) return SS_EINVAL;
    const int N = plan->N;
    RankPtrs rp;
    std::memset(&rp, 0, sizeof rp);
    for (int r = 0; r < N; ++r) {
        if (!rank_grads[r] && hi > lo) return SS_EINVAL;
        if (!ss::aligned(rank_grads[r], 16)) return SS_EALIGN;
        rp.p[r] = rank_grads[r];
    }
    const void* bufs[6] = {accum, master, exp_avg, exp_avg_sq, param_shards, reduced_grad_out};
    for (const void* b : bufs)
        if (b && !ss::aligned(b, 16)) return SS_EALIGN;
    if (hi <= lo) return SS_OK;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int64_t vbeg = (lo + 7) / 8 * 8, vend = hi / 8 * 8;
    const float kdiv = (float)num_micro;
    const AdamCoef c = last ? make_coef(hp) : AdamCoef{};
    uint16_t* sh = static_cast<uint16_t*>(param_shards);
    if (vend > vbeg) {
        const int64_t nvec = (vend - vbeg) / 8;
        const int grid = grid_for(nvec);
        if (!last) {
            AccKernel fn = micro_step == 0 ? pick_acc<true>(N) : pick_acc<false>(N);
            fn<<<grid, kThreads, 0, st>>>(rp, N, vbeg, nvec, accum);
        } else {
            const bool wg = reduced_grad_out != nullptr, m = master != nullptr;
            BF16Kernel fn = m ? (wg ? pick_bf16<true, true, true, true>(N)
                                    : pick_bf16<true, false, true, true>(N))
                              : (wg ? pick_bf16<true, true, false, true>(N)
                                    : pick_bf16<true, false, false, true>(N));
            fn<<<grid, kThreads, 0, st>>>(rp, N, vbeg, nvec, master, exp_avg, exp_avg_sq, sh,
                                          reduced_grad_out, c, accum, kdiv);
        }
        int rc = ss::check_launch();
        if (rc) return rc;
    }
    int64_t a0 = lo, a1 = vbeg < hi ? vbeg : hi;
    int64_t b0 = vend > a1 ? vend : a1, b1 = hi;
    if (vend <= vbeg) {
        a1 = hi;
        b0 = b1 = hi;
    }
    if (a1 > a0 || b1 > b0) {
        const int mode = last ? 2 : (micro_step == 0 ? 0 : 1);
        rs_accum_scalar_kernel<<<1, 32, 0, st>>>(rp, N, a0, a1, b0, b1, accum, mode, kdiv, master,
                                                 exp_avg, exp_avg_sq, sh, reduced_grad_out, c);
        int rc = ss::check_launch();
        if (rc) return rc;
    }
    return SS_OK;
}

