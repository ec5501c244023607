// gn_common.cuh -- GroupNorm finalize arithmetic shared by the separate
// finalize kernels (gn.cu) and the tensor-core kernel's in-kernel finalize
// (tc.cu).  The statistics follow the GroupNorm definition the p85 page uses
// (POPCORNBENCH Kimi-K2.6, level-2 problem 85): biased variance over
// (C/groups, Ho, Wo) including the conv bias, eps inside the square root.
#pragma once

#include <math.h>
#include <stdint.h>

namespace conv_epi {

// Mean and rstd of group g of image n from the fp32 CUDA-core path's per-unit
// partial sums part[n][unit][group][2] (one warp: fixed order in fp64 --
// lanes take units lane, lane+32, ..., then a fixed xor tree, so every lane
// ends with the same bits).  fp64 only here: its rate on this part is low.
__device__ __forceinline__ void gn_group_stats(const double *part, int units, int groups, int n, int g,
                                               double inv_cnt, float eps, float &mean_f, float &rstd_f) {
    const int lane = threadIdx.x & 31;
    double s = 0.0, ss = 0.0;
    const double *p = part + ((size_t)n * units * groups + g) * 2;
    for (int u = lane; u < units; u += 32) s += p[(size_t)u * 2 * groups], ss += p[(size_t)u * 2 * groups + 1];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, off);
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    }
    const double mean = s * inv_cnt;
    double var = ss * inv_cnt - mean * mean;
    if (var < 0.0) var = 0.0;
    mean_f = (float)mean;
    rstd_f = rsqrtf((float)var + eps);
}

// Double-float arithmetic: a value hi + lo held as two floats with |lo| at
// most half an ulp of hi.  The sum keeps the exact rounding error of hi + hi
// (Knuth's TwoSum: no multiplication, so no contraction into an FMA can
// change it) and is commutative bit for bit, so a shuffle butterfly leaves
// every lane with the same result.
struct Df {
    float hi, lo;
};
__device__ __forceinline__ Df df_add(Df a, Df b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b.hi - bb);
    const float t = e + (a.lo + b.lo);
    const float h = s + t;
    return {h, t - (h - s)};
}
// (hi + lo) / n for a float n (the group's count, exact below 2^24): the
// remainder of the first quotient is exact through the FMA
__device__ __forceinline__ Df df_div(Df a, float n) {
    const float q1 = a.hi / n;
    const float r = fmaf(-q1, n, a.hi) + a.lo;
    const float q2 = r / n;
    const float h = q1 + q2;
    return {h, q2 - (h - q1)};
}

// The tensor-core path's statistics: per-unit partial sums stored as float
// pairs part_f[n][unit][group][2], folded in double-float (fp32 arithmetic
// only: fp64 is a slow pipe on this part and the fold sits on the finalize's
// critical path).  Lanes take units lane, lane + 32, ..., then a fixed xor
// tree; the mean and E[y^2] are divided in double-float and the variance
// E[y^2] - mean^2 formed with the product's exact error, so the cancellation
// of a large mean loses nothing to the fold.  cnt = C/groups * Ho * Wo.
__device__ __forceinline__ void gn_group_stats_f(const float *part, int units, int groups, int n, int g, float cnt,
                                                 float eps, float &mean_f, float &rstd_f) {
    const int lane = threadIdx.x & 31;
    Df s{0.0f, 0.0f}, ss{0.0f, 0.0f};
    const float *p = part + ((size_t)n * units * groups + g) * 2;
    for (int u = lane; u < units; u += 32) {
        const float2 v = *reinterpret_cast<const float2 *>(p + (size_t)u * 2 * groups);
        s = df_add(s, Df{v.x, 0.0f});
        ss = df_add(ss, Df{v.y, 0.0f});
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const Df so{__shfl_xor_sync(0xffffffffu, s.hi, off), __shfl_xor_sync(0xffffffffu, s.lo, off)};
        const Df sso{__shfl_xor_sync(0xffffffffu, ss.hi, off), __shfl_xor_sync(0xffffffffu, ss.lo, off)};
        s = df_add(s, so);
        ss = df_add(ss, sso);
    }
    const Df mean = df_div(s, cnt), e2 = df_div(ss, cnt);
    const float p2 = mean.hi * mean.hi;
    const float p2e = fmaf(mean.hi, mean.hi, -p2) + 2.0f * mean.hi * mean.lo;
    const Df var = df_add(e2, Df{-p2, -p2e});
    float v = var.hi + var.lo;
    if (v < 0.0f) v = 0.0f;
    mean_f = mean.hi + mean.lo;
    rstd_f = rsqrtf(v + eps);
}

// Channel c's affine map z = A * y + B of GroupNorm then the scale:
// A = gamma * scale * rstd, B = (beta - gamma * mean * rstd) * scale.
__device__ __forceinline__ void gn_coeffs(float gamma, float beta, float scale, float mean, float rstd, float &A,
                                          float &B) {
    A = gamma * scale * rstd;
    B = (beta - gamma * mean * rstd) * scale;
}

}  // namespace conv_epi
