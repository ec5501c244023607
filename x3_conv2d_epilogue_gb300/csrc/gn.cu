// gn.cu -- finalize step of the GroupNorm -> scale -> max-pool -> clamp
// chain, shared by both conv paths.
//
// The conv kernels never write the normalised tensor.  They leave, per pooling
// window, the max and the min of y = conv + bias (the tf32 path only the one
// that the channel's slope sign selects, see below), and per (image, unit,
// group) the partial sums of y and y^2.  Because the normalisation and the scale are
// one affine map per channel,
//     z = ((y - mean) * rstd * gamma + beta) * scale = A * y + B,
//     A = gamma * scale * rstd,  B = (beta - gamma * mean * rstd) * scale,
// the pooled maximum of z is A * max(y) + B when A >= 0 and A * min(y) + B
// when A < 0.  As rstd > 0, the sign of A is that of gamma * scale, known
// before any statistic.  This is the GroupNorm affine fold of the p85 page
// (POPCORNBENCH Kimi-K2.6, level-2 problem 85: "effective_gamma = gamma *
// scale, effective_beta = beta * scale"), carried one step further so that the
// pool can run before the statistics are known.  Statistics follow the same
// page: biased variance over (C/groups, Ho, Wo) including the conv bias, eps
// inside the square root.
#include <math.h>

#include "gn_common.cuh"
#include "internal.h"

namespace conv_epi {
namespace {

constexpr int kThreads = 256;

struct GnArgs {
    GnWork gn;
    int N, C, Ho, Wo, groups;
    float eps, lo, hi;
    const float *gamma, *beta, *scale;
    float *out;
    int32_t *idx;
    int presel;      // 1: pmax already holds the extreme the slope's sign selects
    int nsl;         // with presel: the slots holding it for the parts of each band (1; 2: halves in pmax, pmin;
                     // 4: quarters in pmax, pmin and the index buffers, which the tensor-core path leaves free)
    double inv_cnt;  // 1 / (C/groups * Ho * Wo)
    float cnt;       // C/groups * Ho * Wo
    uint32_t per_magic;  // ceil(2^32 / (Hp * Wp)): exact f / (Hp * Wp) for f < 2^16
};

// the tensor-core path (presel) stores its partial sums as float pairs, the
// fp32 CUDA-core path as doubles
__device__ __forceinline__ void group_stats(const GnArgs &a, int n, int g, float &mean_f, float &rstd_f) {
    if (a.presel)
        gn_group_stats_f(reinterpret_cast<const float *>(a.gn.part), a.gn.units, a.groups, n, g, a.cnt, a.eps, mean_f,
                         rstd_f);
    else
        gn_group_stats(a.gn.part, a.gn.units, a.groups, n, g, a.inv_cnt, a.eps, mean_f, rstd_f);
}

// The tensor-core path's case: pmax holds, per channel, the extreme that the
// slope's sign selects, and no indices are wanted.  The group's C/groups
// pooled planes are one contiguous block of F = cpg * Hp * Wp floats (F a
// multiple of 4, 16-byte aligned: checked on the host), so every thread first
// issues its 16-byte loads of the block's first 4096 floats, then warp 0
// computes the statistics and each channel's coefficients while those loads
// are in flight; one barrier, then z = clamp(A * y + B) and 16-byte stores.
constexpr int kVec = 4;  // float4 loads in flight per thread
__global__ void __launch_bounds__(kThreads) gn_finalize_vec_kernel(const GnArgs a) {
    constexpr int kMaxCpg = 64;
    __shared__ float sA[kMaxCpg], sB[kMaxCpg];
    const int n = blockIdx.x / a.groups, g = blockIdx.x % a.groups;
    const int cpg = a.C / a.groups;
    const uint32_t per = (uint32_t)(a.gn.Hp * a.gn.Wp);
    const size_t base = ((size_t)n * a.C + (size_t)g * cpg) * per;
    const float4 *__restrict__ src = reinterpret_cast<const float4 *>(a.gn.pmax + base);
    // (bands in parts: the other slots)
    const float4 *__restrict__ src2 = reinterpret_cast<const float4 *>(a.gn.pmin + base);
    const float4 *__restrict__ src3 = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.gn.amax) + base);
    const float4 *__restrict__ src4 = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.gn.amin) + base);
    float4 *__restrict__ dst = reinterpret_cast<float4 *>(a.out + base);
    const int nv = (int)((size_t)cpg * per / 4);
    float4 v[kVec], w[kVec], w3[kVec], w4[kVec];
    auto load = [&](int k, int i) {
        v[k] = src[i];
        if (a.nsl > 1) w[k] = src2[i];
        if (a.nsl > 2) w3[k] = src3[i], w4[k] = src4[i];
    };
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        const int i = threadIdx.x + k * kThreads;
        if (i < nv) load(k, i);
    }
    if (threadIdx.x < 32) {
        // the channel parameters (at most two channels per lane) are loaded
        // before the fold, so their latency overlaps it
        float gm[kMaxCpg / 32], sc[kMaxCpg / 32], bt[kMaxCpg / 32];
#pragma unroll
        for (int k = 0; k < kMaxCpg / 32; ++k) {
            const int cl = threadIdx.x + 32 * k;
            if (cl < cpg) {
                const int c = g * cpg + cl;
                gm[k] = a.gamma[c], sc[k] = a.scale[c], bt[k] = a.beta[c];
            }
        }
        float mean, rstd;
        group_stats(a, n, g, mean, rstd);
#pragma unroll
        for (int k = 0; k < kMaxCpg / 32; ++k) {
            const int cl = threadIdx.x + 32 * k;
            if (cl < cpg) gn_coeffs(gm[k], bt[k], sc[k], mean, rstd, sA[cl], sB[cl]);
        }
    }
    __syncthreads();
    // (bands in parts: the band's extreme from its parts, by the slope's sign)
    auto apply = [&](float y, float y2, float y3, float y4, uint32_t f) {
        const uint32_t cl = __umulhi(f, a.per_magic);  // f / per
        if (a.nsl > 1) {
            const bool up = sA[cl] >= 0.0f;
            y = up ? fmaxf(y, y2) : fminf(y, y2);
            if (a.nsl > 2) y = up ? fmaxf(y, fmaxf(y3, y4)) : fminf(y, fminf(y3, y4));
        }
        return fminf(fmaxf(fmaf(sA[cl], y, sB[cl]), a.lo), a.hi);
    };
    for (int i0 = 0; i0 < nv; i0 += kVec * kThreads) {
        if (i0 > 0) {
#pragma unroll
            for (int k = 0; k < kVec; ++k) {
                const int i = i0 + threadIdx.x + k * kThreads;
                if (i < nv) load(k, i);
            }
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int i = i0 + threadIdx.x + k * kThreads;
            if (i < nv) {
                const uint32_t f = 4u * (uint32_t)i;
                dst[i] = make_float4(apply(v[k].x, w[k].x, w3[k].x, w4[k].x, f), apply(v[k].y, w[k].y, w3[k].y, w4[k].y, f + 1),
                                     apply(v[k].z, w[k].z, w3[k].z, w4[k].z, f + 2),
                                     apply(v[k].w, w[k].w, w3[k].w, w4[k].w, f + 3));
            }
        }
    }
}

// One CTA per (image, group).  Warp 0 folds the group's per-unit partial sums
// (fixed order: lanes take units lane, lane+32, ..., then a fixed shuffle
// tree; fp64 for the fp32 path's double partials, double-float for the
// tensor-core path's float pairs) into the mean and variance; the first C/groups threads turn
// them into each channel's affine coefficients (fp32; rstd = 1/sqrt(var +
// eps) from the variance).  Then the CTA writes the group's pooled
// outputs, channel by channel (C/groups consecutive [Hp][Wp] planes:
// contiguous loads and stores).  fp64 is kept to the fp32 path's fold: it is
// a slow pipe on this part, so no per-output or per-thread fp64 work.
__global__ void __launch_bounds__(kThreads) gn_finalize_kernel(const GnArgs a) {
    constexpr int kMaxCpg = 64;
    __shared__ float s_mean, s_rstd;
    __shared__ float sA[kMaxCpg], sB[kMaxCpg];
    const int n = blockIdx.x / a.groups, g = blockIdx.x % a.groups;
    const int cpg = a.C / a.groups;
    if (threadIdx.x < 32) {
        float mean, rstd;
        group_stats(a, n, g, mean, rstd);
        if (threadIdx.x == 0) s_mean = mean, s_rstd = rstd;
    }
    __syncthreads();
    const float mean = s_mean, rstd = s_rstd;
    for (int cl0 = 0; cl0 < cpg; cl0 += kMaxCpg) {
        const int ncl = min(kMaxCpg, cpg - cl0);
        if (cl0 > 0) __syncthreads();  // the previous batch's coefficients are no longer read
        if (threadIdx.x < ncl) {
            const int c = g * cpg + cl0 + threadIdx.x;
            gn_coeffs(a.gamma[c], a.beta[c], a.scale[c], mean, rstd, sA[threadIdx.x], sB[threadIdx.x]);
        }
        __syncthreads();
        const int per = a.gn.Hp * a.gn.Wp;
        for (int cl = 0; cl < ncl; ++cl) {
            const int c = g * cpg + cl0 + cl;
            const float A = sA[cl], B = sB[cl];
            const size_t base = ((size_t)n * a.C + c) * per;
            const float *__restrict__ src = ((a.presel || A >= 0.0f) ? a.gn.pmax : a.gn.pmin) + base;
            // (bands in parts: the other slots)
            const float *__restrict__ src2 = a.gn.pmin + base;
            const float *__restrict__ src3 = reinterpret_cast<const float *>(a.gn.amax) + base;
            const float *__restrict__ src4 = reinterpret_cast<const float *>(a.gn.amin) + base;
            float *__restrict__ dst = a.out + base;
            if (a.idx) {
                const int32_t *__restrict__ isrc = (A > 0.0f ? a.gn.amax : a.gn.amin) + base;
                for (int p = threadIdx.x; p < per; p += kThreads) {
                    dst[p] = fminf(fmaxf(fmaf(A, src[p], B), a.lo), a.hi);
                    a.idx[base + p] = A != 0.0f ? isrc[p] : 0;
                }
            } else {
                // four independent loads in flight per thread (bands in
                // parts: each the extreme of the band's parts by the slope's sign)
                auto y_at = [&](int q) {
                    float y = src[q];
                    if (a.nsl > 1) y = A >= 0.0f ? fmaxf(y, src2[q]) : fminf(y, src2[q]);
                    if (a.nsl > 2)
                        y = A >= 0.0f ? fmaxf(y, fmaxf(src3[q], src4[q])) : fminf(y, fminf(src3[q], src4[q]));
                    return y;
                };
                int p = threadIdx.x;
                for (; p + 3 * kThreads < per; p += 4 * kThreads) {
                    const float y0 = y_at(p), y1 = y_at(p + kThreads), y2 = y_at(p + 2 * kThreads), y3 = y_at(p + 3 * kThreads);
                    dst[p] = fminf(fmaxf(fmaf(A, y0, B), a.lo), a.hi);
                    dst[p + kThreads] = fminf(fmaxf(fmaf(A, y1, B), a.lo), a.hi);
                    dst[p + 2 * kThreads] = fminf(fmaxf(fmaf(A, y2, B), a.lo), a.hi);
                    dst[p + 3 * kThreads] = fminf(fmaxf(fmaf(A, y3, B), a.lo), a.hi);
                }
                for (; p < per; p += kThreads) dst[p] = fminf(fmaxf(fmaf(A, y_at(p), B), a.lo), a.hi);
            }
        }
    }
}

}  // namespace

conv_epi_status gn_finalize(conv_epi_handle h, const conv_epi_epilogue_desc &e, float *out, cudaStream_t s,
                            bool presel, int nslots) {
    GnArgs a;
    a.gn = h->gn;
    a.N = h->d.N, a.C = h->d.Cout, a.Ho = h->Ho, a.Wo = h->Wo, a.groups = e.groups;
    a.eps = e.eps, a.lo = e.clamp_lo, a.hi = e.clamp_hi;
    a.gamma = e.gamma, a.beta = e.beta, a.scale = e.chan_scale;
    a.out = out, a.idx = e.index_out;
    a.presel = presel ? 1 : 0;
    a.nsl = presel ? nslots : 1;
    a.inv_cnt = 1.0 / ((double)(a.C / a.groups) * a.Ho * a.Wo);
    a.cnt = (float)((double)(a.C / a.groups) * a.Ho * a.Wo);
    const uint32_t per = (uint32_t)(h->gn.Hp * h->gn.Wp);
    a.per_magic = (uint32_t)((((uint64_t)1 << 32) + per - 1) / per);
    const unsigned blocks = (unsigned)(a.N * a.groups);
    // the vector kernel: whole group blocks of float4 (F = cpg * per a multiple
    // of 4 keeps every block 16-byte aligned), flat indices below 2^16 for the
    // channel division, at most 64 channels per group
    const size_t F = (size_t)(a.C / a.groups) * per;
    const bool vec = presel && !e.index_out && F % 4 == 0 && F < (1u << 16) && a.C / a.groups <= 64 &&
                     (reinterpret_cast<uintptr_t>(out) & 15u) == 0 && (reinterpret_cast<uintptr_t>(h->gn.pmax) & 15u) == 0;
    if (vec) gn_finalize_vec_kernel<<<blocks, kThreads, 0, s>>>(a);
    else gn_finalize_kernel<<<blocks, kThreads, 0, s>>>(a);
    CE_CUDA(cudaGetLastError());
    return CONV_EPI_OK;
}

}  // namespace conv_epi
