// gn_common.cuh -- GroupNorm finalize arithmetic shared by the separate
// finalize kernels (gn.cu) and the tensor-core kernel's in-kernel finalize
// (tc.cu).  The statistics follow the GroupNorm definition the p85 page uses
// (POPCORNBENCH Kimi-K2.6, level-2 problem 85): biased variance over
// (C/groups, Ho, Wo) including the conv bias, eps inside the square root.
#pragma once

#include <math.h>
#include <stdint.h>

namespace conv_epi {

// Mean and rstd of group g of image n from the per-unit partial sums
// part[n][unit][group][2] (one warp: fixed order in fp64 -- lanes take units
// lane, lane+32, ..., then a fixed xor tree, so every lane ends with the same
// bits).  fp64 only here: its rate on this part is low.
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

// Channel c's affine map z = A * y + B of GroupNorm then the scale:
// A = gamma * scale * rstd, B = (beta - gamma * mean * rstd) * scale.
__device__ __forceinline__ void gn_coeffs(float gamma, float beta, float scale, float mean, float rstd, float &A,
                                          float &B) {
    A = gamma * scale * rstd;
    B = (beta - gamma * mean * rstd) * scale;
}

}  // namespace conv_epi
