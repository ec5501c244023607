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

constexpr int kChan = 16;  // channels per CTA

struct GnArgs {
    GnWork gn;
    int N, C, Ho, Wo, groups;
    float eps, lo, hi;
    const float *gamma, *beta, *scale;
    float *out;
    int32_t *idx;
};

__global__ void __launch_bounds__(256) gn_finalize_kernel(const GnArgs a) {
    __shared__ float sA[kChan], sB[kChan];
    const int n = blockIdx.x;
    const int c0 = blockIdx.y * kChan;
    const int nc = min(kChan, a.C - c0);
    if (threadIdx.x < nc) {
        const int c = c0 + threadIdx.x;
        const int cpg = a.C / a.groups;
        const int g = c / cpg;
        double s = 0.0, ss = 0.0;
        const double *p = a.gn.part + ((size_t)n * a.gn.units * a.groups + g) * 2;
        for (int u = 0; u < a.gn.units; ++u, p += 2 * a.groups) s += p[0], ss += p[1];
        const double cnt = (double)cpg * a.Ho * a.Wo;
        const double mean = s / cnt;
        double var = ss / cnt - mean * mean;
        if (var < 0.0) var = 0.0;
        const double rstd = 1.0 / sqrt(var + (double)a.eps);
        const double gm = a.gamma[c], sc = a.scale[c];
        sA[threadIdx.x] = (float)(gm * sc * rstd);
        sB[threadIdx.x] = (float)((a.beta[c] - gm * mean * rstd) * sc);
    }
    __syncthreads();
    const int per = a.gn.Hp * a.gn.Wp;
    for (int i = threadIdx.x; i < nc * per; i += blockDim.x) {
        const int cl = i / per;
        const size_t o = ((size_t)n * a.C + c0 + cl) * per + (i % per);
        const float A = sA[cl];
        const float y = A >= 0.0f ? a.gn.pmax[o] : a.gn.pmin[o];
        const float z = fmaf(A, y, sB[cl]);
        a.out[o] = fminf(fmaxf(z, a.lo), a.hi);
        if (a.idx) a.idx[o] = A > 0.0f ? a.gn.amax[o] : (A < 0.0f ? a.gn.amin[o] : 0);
    }
}

}  // namespace

conv_epi_status gn_finalize(conv_epi_handle h, const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    GnArgs a;
    a.gn = h->gn;
    a.N = h->d.N, a.C = h->d.Cout, a.Ho = h->Ho, a.Wo = h->Wo, a.groups = e.groups;
    a.eps = e.eps, a.lo = e.clamp_lo, a.hi = e.clamp_hi;
    a.gamma = e.gamma, a.beta = e.beta, a.scale = e.chan_scale;
    a.out = out, a.idx = e.index_out;
    dim3 grid(h->d.N, (h->d.Cout + kChan - 1) / kChan);
    gn_finalize_kernel<<<grid, 256, 0, s>>>(a);
    CE_CUDA(cudaGetLastError());
    return CONV_EPI_OK;
}

}  // namespace conv_epi
