// gn.cu -- finalize step of the GroupNorm -> scale -> max-pool -> clamp
// chain, shared by both conv paths.
//
// The conv kernels never write the normalised tensor.  They leave, per pooling
// window, the max and the min of y = conv + bias, and per (image, unit, group)
// the partial sums of y and y^2.  Because the normalisation and the scale are
// one affine map per channel,
//     z = ((y - mean) * rstd * gamma + beta) * scale = A * y + B,
//     A = gamma * scale * rstd,  B = (beta - gamma * mean * rstd) * scale,
// the pooled maximum of z is A * max(y) + B when A >= 0 and A * min(y) + B
// when A < 0.  This is the GroupNorm affine fold of the p85 page
// (POPCORNBENCH Kimi-K2.6, level-2 problem 85: "effective_gamma = gamma *
// scale, effective_beta = beta * scale"), carried one step further so that the
// pool can run before the statistics are known.  Statistics follow the same
// page: biased variance over (C/groups, Ho, Wo) including the conv bias, eps
// inside the square root.
#include <math.h>

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
};

// One thread per pooled output.  A CTA covers kThreads consecutive outputs
// of the [N][C][Hp][Wp] tensor, i.e. at most a few (n, c) planes; one warp
// per plane folds the partial sums of that plane's group (fixed order, fp64)
// into the channel's affine coefficients.
__global__ void __launch_bounds__(kThreads) gn_finalize_kernel(const GnArgs a) {
    constexpr int kMaxPlanes = kThreads + 1;  // (n, c) planes one CTA can touch
    __shared__ float sA[kMaxPlanes], sB[kMaxPlanes];
    const int per = a.gn.Hp * a.gn.Wp;
    const size_t total = (size_t)a.N * a.C * per;
    const size_t first = (size_t)blockIdx.x * kThreads;
    const size_t plane0 = first / per;
    const size_t last = min(total, first + kThreads) - 1;
    const int nplanes = (int)(last / per - plane0 + 1);
    // one warp per plane: lanes load the per-unit partial sums in parallel and
    // fold them in a fixed order (strided lane sums, then a fixed shuffle tree)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = warp; k < nplanes; k += kThreads / 32) {
        const size_t pl = plane0 + k;
        const int n = (int)(pl / a.C), c = (int)(pl % a.C);
        const int cpg = a.C / a.groups;
        const int g = c / cpg;
        double s = 0.0, ss = 0.0;
        const double *p = a.gn.part + ((size_t)n * a.gn.units * a.groups + g) * 2;
        for (int u = lane; u < a.gn.units; u += 32) s += p[(size_t)u * 2 * a.groups], ss += p[(size_t)u * 2 * a.groups + 1];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, off);
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
        }
        if (lane == 0) {
            const double cnt = (double)cpg * a.Ho * a.Wo;
            const double mean = s / cnt;
            double var = ss / cnt - mean * mean;
            if (var < 0.0) var = 0.0;
            const double rstd = 1.0 / sqrt(var + (double)a.eps);
            const double gm = a.gamma[c], sc = a.scale[c];
            sA[k] = (float)(gm * sc * rstd);
            sB[k] = (float)((a.beta[c] - gm * mean * rstd) * sc);
        }
    }
    __syncthreads();
    const size_t o = first + threadIdx.x;
    if (o >= total) return;
    const int k = (int)(o / per - plane0);
    const float A = sA[k];
    const float y = A >= 0.0f ? a.gn.pmax[o] : a.gn.pmin[o];
    a.out[o] = fminf(fmaxf(fmaf(A, y, sB[k]), a.lo), a.hi);
    if (a.idx) a.idx[o] = A > 0.0f ? a.gn.amax[o] : (A < 0.0f ? a.gn.amin[o] : 0);
}

}  // namespace

conv_epi_status gn_finalize(conv_epi_handle h, const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    GnArgs a;
    a.gn = h->gn;
    a.N = h->d.N, a.C = h->d.Cout, a.Ho = h->Ho, a.Wo = h->Wo, a.groups = e.groups;
    a.eps = e.eps, a.lo = e.clamp_lo, a.hi = e.clamp_hi;
    a.gamma = e.gamma, a.beta = e.beta, a.scale = e.chan_scale;
    a.out = out, a.idx = e.index_out;
    const size_t per = (size_t)h->gn.Hp * h->gn.Wp;
    const size_t total = (size_t)a.N * a.C * per;
    const unsigned blocks = (unsigned)((total + kThreads - 1) / kThreads);
    gn_finalize_kernel<<<blocks, kThreads, 0, s>>>(a);
    CE_CUDA(cudaGetLastError());
    return CONV_EPI_OK;
}

}  // namespace conv_epi
