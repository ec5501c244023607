// postpass.cu -- conv_epi_postpass: a chain applied as a separate pass over a
// stored conv output y[N][Cout][Ho][Wo] (bias included), in fp32 arithmetic.
//
// This is the structure every page starts from and plans its kernels for: the
// convolution stays a library call that writes the full conv output to
// memory, and the post-conv chain is one custom pass over it (POPCORNBENCH
// Kimi-K2.6, level 2: p25 "fused_min_tanh_tanh", a thread per output pixel
// looping over the channels; p32 the scale + channel-min kernel of the same
// shape; p54 the fused elementwise multiplier / LeakyReLU / GELU pass; p85 a
// GroupNorm statistics kernel, then one kernel that normalises, scales, max
// pools and clamps).  Written anew for sm_103a; the library offers it so that
// the fused forward can be compared with the unfused design on one machine,
// and for callers that already hold a conv output.
//
// Kernels (all memory-bound, coalesced):
//   min chains      one thread per output pixel, the channel loop four loads
//                   deep;
//   per-channel     16-byte loads and stores over each (image, channel) plane
//                   when a plane is whole float4s, else one float per thread;
//   GroupNorm       stats: one CTA per (image, group), fp32 per thread, fp64
//                   across the CTA in a fixed order; apply: one warp per
//                   pooled row, a lane per window, the window's max (or min,
//                   when the channel's slope gamma * scale is negative) of y
//                   by vector loads where the rows allow, then
//                   clamp(A y + B).
#include <math.h>

#include <type_traits>

#include "gn_common.cuh"
#include "internal.h"

namespace conv_epi {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float gelu_erf(float t) { return 0.5f * t * (1.0f + erff(t * 0.70710678118654752f)); }

// min over channels of scalar * y, then tanh(tanh(.)) when tanh2
__global__ void __launch_bounds__(kThreads) post_min(const float *__restrict__ y, float *__restrict__ out, int N, int C,
                                                    size_t plane, float scalar, int tanh2) {
    const size_t total = (size_t)N * plane;
    for (size_t p = blockIdx.x * (size_t)blockDim.x + threadIdx.x; p < total; p += (size_t)gridDim.x * blockDim.x) {
        const size_t n = p / plane, q = p - n * plane;
        const float *src = y + n * C * plane + q;
        float m = INFINITY;
        int c = 0;
        for (; c + 4 <= C; c += 4) {
            const float v0 = __ldg(src + (size_t)c * plane), v1 = __ldg(src + (size_t)(c + 1) * plane);
            const float v2 = __ldg(src + (size_t)(c + 2) * plane), v3 = __ldg(src + (size_t)(c + 3) * plane);
            m = fminf(m, fminf(fminf(scalar * v0, scalar * v1), fminf(scalar * v2, scalar * v3)));
        }
        for (; c < C; ++c) m = fminf(m, scalar * __ldg(src + (size_t)c * plane));
        if (tanh2) m = tanhf(tanhf(m));
        out[p] = m;
    }
}

// out = y (kind NONE) or GELU(LeakyReLU(y * mult[c])), plane by plane
template <bool kGelu>
__global__ void __launch_bounds__(kThreads) post_chan(const float *__restrict__ y, float *__restrict__ out, int N, int C,
                                                     size_t plane, const float *__restrict__ mult, float slope) {
    auto f = [&](float v, float m) {
        if (!kGelu) return v;
        float t = v * m;
        t = t > 0.0f ? t : slope * t;
        return gelu_erf(t);
    };
    const size_t planes = (size_t)N * C;
    if (plane % 4 == 0) {
        const size_t p4 = plane / 4, total = planes * p4;
        const float4 *s4 = reinterpret_cast<const float4 *>(y);
        float4 *d4 = reinterpret_cast<float4 *>(out);
        for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
            const int c = (int)((i / p4) % C);
            const float m = kGelu ? __ldg(&mult[c]) : 1.0f;
            const float4 v = __ldg(s4 + i);
            d4[i] = make_float4(f(v.x, m), f(v.y, m), f(v.z, m), f(v.w, m));
        }
    } else {
        const size_t total = planes * plane;
        for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
            const int c = (int)((i / plane) % C);
            out[i] = f(__ldg(y + i), kGelu ? __ldg(&mult[c]) : 1.0f);
        }
    }
}

// GroupNorm statistics of (image n, group g) = blockIdx.x: the group's cpg
// planes are one contiguous block; per-thread fp32 sums, then the CTA's
// threads folded in fp64 in a fixed order (warp xor trees, then the warps in
// order); stats[n][g] = (mean, rstd)
__global__ void __launch_bounds__(kThreads) post_gn_stats(const float *__restrict__ y, float *__restrict__ stats,
                                                         int groups, int cpg, size_t plane, double inv_cnt, float eps) {
    __shared__ double ws[2][kThreads / 32];
    const size_t len = (size_t)cpg * plane;
    const float *src = y + (size_t)blockIdx.x * len;
    float s = 0.0f, ss = 0.0f;
    for (size_t i = threadIdx.x; i < len; i += kThreads) {
        const float v = __ldg(src + i);
        s += v, ss = fmaf(v, v, ss);
    }
    double ds = s, dss = ss;
    for (int o = 16; o >= 1; o >>= 1) {
        ds += __shfl_xor_sync(0xffffffffu, ds, o);
        dss += __shfl_xor_sync(0xffffffffu, dss, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) ws[0][warp] = ds, ws[1][warp] = dss;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0, tt = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) t += ws[0][w], tt += ws[1][w];
        const double mean = t * inv_cnt;
        double var = tt * inv_cnt - mean * mean;
        if (var < 0.0) var = 0.0;
        stats[2 * blockIdx.x] = (float)mean;
        stats[2 * blockIdx.x + 1] = rsqrtf((float)var + eps);
    }
}

// one warp per pooled row (n, c, ph), its lanes over the row's windows pw:
// z = A y + B over the k x k window, pooled by its max (A's sign picks the
// max or the min of y), then clamped.  The row's index arithmetic and the
// channel's coefficients are taken once per row, and a lane's loads for its
// next windows (pw = lane + 32 j: 1, 2 or 4 of them for k = 4, 2..3 or 1) go
// out before any is reduced, so enough bytes are in flight to keep HBM busy.  VEC floats per load: 4 when k = 4
// and Wo is a multiple of 4, 2 when k is even and Wo is even (every window
// row then starts on a VEC-float boundary), else 1; K = 0 takes k at run
// time (one window at a time).
template <int K, int VEC>
__global__ void __launch_bounds__(kThreads) post_gn_pool(const float *__restrict__ y, float *__restrict__ out,
                                                        const float *__restrict__ stats, const float *__restrict__ gamma,
                                                        const float *__restrict__ beta, const float *__restrict__ scale,
                                                        int N, int C, int groups, int Ho, int Wo, int k_rt, int Hp,
                                                        int Wp, float lo, float hi) {
    const int k = K ? K : k_rt;
    const size_t rows = (size_t)N * C * Hp;
    const int cpg = C / groups, lane = threadIdx.x & 31;
    const size_t warps = (size_t)gridDim.x * (kThreads / 32);
    for (size_t r = blockIdx.x * (size_t)(kThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
        const size_t nc = r / Hp;
        const int ph = (int)(r - nc * Hp);
        const int c = (int)(nc % C), n = (int)(nc / C), g = c / cpg;
        const float mean = __ldg(&stats[2 * ((size_t)n * groups + g)]), rstd = __ldg(&stats[2 * ((size_t)n * groups + g) + 1]);
        float A, B;
        gn_coeffs(__ldg(&gamma[c]), __ldg(&beta[c]), __ldg(&scale[c]), mean, rstd, A, B);
        const float *w0 = y + (nc * Ho + (size_t)ph * k) * Wo;
        float *orow = out + r * Wp;
        if constexpr (K > 0) {
            constexpr int kJ = K >= 4 ? 1 : K >= 2 ? 2 : 4, kL = K / VEC;  // windows per lane per batch, loads per window row
            using V = typename std::conditional<VEC == 4, float4, typename std::conditional<VEC == 2, float2, float>::type>::type;
            for (int pb = 0; pb < Wp; pb += 32 * kJ) {
                V v[kJ][K][kL];
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
                    const int pw = pb + lane + 32 * j;
                    if (pw < Wp) {
#pragma unroll
                        for (int a = 0; a < K; ++a)
#pragma unroll
                            for (int l = 0; l < kL; ++l)
                                v[j][a][l] = __ldg(reinterpret_cast<const V *>(w0 + (size_t)a * Wo + (size_t)pw * K) + l);
                    }
                }
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
                    const int pw = pb + lane + 32 * j;
                    if (pw >= Wp) break;
                    float mx = -INFINITY, mn = INFINITY;
#pragma unroll
                    for (int a = 0; a < K; ++a)
#pragma unroll
                        for (int l = 0; l < kL; ++l) {
                            const float *e = reinterpret_cast<const float *>(&v[j][a][l]);
#pragma unroll
                            for (int i = 0; i < VEC; ++i) mx = fmaxf(mx, e[i]), mn = fminf(mn, e[i]);
                        }
                    orow[pw] = fminf(fmaxf(fmaf(A, A >= 0.0f ? mx : mn, B), lo), hi);
                }
            }
        } else {
            for (int pw = lane; pw < Wp; pw += 32) {
                const float *w = w0 + (size_t)pw * k;
                float mx = -INFINITY, mn = INFINITY;
                for (int a = 0; a < k; ++a)
                    for (int b = 0; b < k; ++b) {
                        const float v = __ldg(w + (size_t)a * Wo + b);
                        mx = fmaxf(mx, v), mn = fminf(mn, v);
                    }
                orow[pw] = fminf(fmaxf(fmaf(A, A >= 0.0f ? mx : mn, B), lo), hi);
            }
        }
    }
}

// The same statistics from the two-pass tensor-core form's per-unit sums:
// ystat[n][u][hc][L] = (sum y, sum y^2) of accumulator row L's valid outputs
// in unit u (column group hc); row L of a unit holds channel
// mt * Cg + L % Cg (mt: the unit's channel tile), so group g's entries are
// its cpg channels' rows of every row slot s < S, in the units of their
// tile.  Per-thread fp32 sums over a strided slice, then the CTA's threads in
// fp64 in a fixed order, as above.
__global__ void __launch_bounds__(kThreads) post_gn_stats_units(const float2 *__restrict__ ystat, float *__restrict__ stats,
                                                               int groups, int cpg, int upi, int S, int MT, int Cg,
                                                               double inv_cnt, float eps) {
    __shared__ double ws[2][kThreads / 32];
    const int n = blockIdx.x / groups, g = blockIdx.x % groups;
    const int per_unit = cpg * S * 2;  // entries of group g in one unit
    const int total = per_unit * upi;
    float s = 0.0f, ss = 0.0f;
    for (int i = threadIdx.x; i < total; i += kThreads) {
        const int u = i / per_unit, r = i - u * per_unit;
        const int cl = r % cpg, sl = (r / cpg) % S, hc = r / (cpg * S);
        const int c = g * cpg + cl;
        if (MT > 1 && u % MT != c / Cg) continue;  // another channel tile's unit
        const float2 v = __ldg(&ystat[(((size_t)n * upi + u) * 2 + hc) * 128 + sl * Cg + c % Cg]);
        s += v.x, ss += v.y;
    }
    double ds = s, dss = ss;
    for (int o = 16; o >= 1; o >>= 1) {
        ds += __shfl_xor_sync(0xffffffffu, ds, o);
        dss += __shfl_xor_sync(0xffffffffu, dss, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) ws[0][warp] = ds, ws[1][warp] = dss;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0, tt = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) t += ws[0][w], tt += ws[1][w];
        const double mean = t * inv_cnt;
        double var = tt * inv_cnt - mean * mean;
        if (var < 0.0) var = 0.0;
        stats[2 * blockIdx.x] = (float)mean;
        stats[2 * blockIdx.x + 1] = rsqrtf((float)var + eps);
    }
}

unsigned blocks_for(size_t work, int sm_count) {
    const size_t b = (work + kThreads - 1) / kThreads;
    const size_t cap = (size_t)sm_count * 8;
    return (unsigned)(b < cap ? (b ? b : 1) : cap);
}

// the pooling pass with the widest loads the window rows allow
void launch_gn_pool(conv_epi_handle h, const float *y, const conv_epi_epilogue_desc &e, float *out, int Hp, int Wp,
                    cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    const int Ho = h->Ho, Wo = h->Wo, k = e.pool_k;
    const size_t rows = (size_t)d.N * d.Cout * Hp;
    const unsigned grid = blocks_for(rows * 32, h->sm_count);
    auto go = [&](auto kern) {
        kern<<<grid, kThreads, 0, s>>>(y, out, h->post, e.gamma, e.beta, e.chan_scale, d.N, d.Cout, e.groups, Ho, Wo,
                                       k, Hp, Wp, e.clamp_lo, e.clamp_hi);
    };
    if (k == 4 && Wo % 4 == 0) go(post_gn_pool<4, 4>);
    else if (k == 4 && Wo % 2 == 0) go(post_gn_pool<4, 2>);
    else if (k == 4) go(post_gn_pool<4, 1>);
    else if (k == 2 && Wo % 2 == 0) go(post_gn_pool<2, 2>);
    else if (k == 2) go(post_gn_pool<2, 1>);
    else if (k == 1) go(post_gn_pool<1, 1>);
    else if (k == 3) go(post_gn_pool<3, 1>);
    else go(post_gn_pool<0, 1>);
}

}  // namespace

conv_epi_status ensure_post_stats(conv_epi_handle h, int groups) {
    const size_t need = (size_t)h->d.N * groups * 2 * sizeof(float);
    if (need > h->post_bytes) {
        if (h->post) {
            CE_CUDA(cudaDeviceSynchronize());
            CE_CUDA(cudaFree(h->post));
            h->post = nullptr, h->post_bytes = 0;
        }
        CE_CUDA(cudaMalloc(&h->post, need));
        h->post_bytes = need;
    }
    return CONV_EPI_OK;
}

conv_epi_status postpass_gn_units(conv_epi_handle h, const float *y, const float2 *ystat, int upi, int S, int MT, int Cg,
                                  const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    const size_t plane = (size_t)h->Ho * h->Wo;
    conv_epi_status st = ensure_post_stats(h, e.groups);
    if (st) return st;
    const int cpg = d.Cout / e.groups;
    post_gn_stats_units<<<(unsigned)(d.N * e.groups), kThreads, 0, s>>>(ystat, h->post, e.groups, cpg, upi, S, MT, Cg,
                                                                       1.0 / ((double)cpg * plane), e.eps);
    CE_CUDA(cudaGetLastError());
    const int Hp = (h->Ho - e.pool_k) / e.pool_k + 1, Wp = (h->Wo - e.pool_k) / e.pool_k + 1;
    launch_gn_pool(h, y, e, out, Hp, Wp, s);
    CE_CUDA(cudaGetLastError());
    h->last_launches = 2;
    return CONV_EPI_OK;
}

conv_epi_status postpass_forward(conv_epi_handle h, const float *y, const conv_epi_epilogue_desc &e, float *out,
                                 cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    const size_t plane = (size_t)h->Ho * h->Wo;
    h->last_launches = 0;
    switch (e.kind) {
    case CONV_EPI_MIN_TANH2:
    case CONV_EPI_SCALE_MIN:
        post_min<<<blocks_for((size_t)d.N * plane, h->sm_count), kThreads, 0, s>>>(
            y, out, d.N, d.Cout, plane, e.scalar, e.kind == CONV_EPI_MIN_TANH2 ? 1 : 0);
        break;
    case CONV_EPI_MUL_LRELU_GELU:
        post_chan<true><<<blocks_for((size_t)d.N * d.Cout * plane / 4, h->sm_count), kThreads, 0, s>>>(
            y, out, d.N, d.Cout, plane, e.chan_scale, e.lrelu_slope);
        break;
    case CONV_EPI_NONE:
        post_chan<false><<<blocks_for((size_t)d.N * d.Cout * plane / 4, h->sm_count), kThreads, 0, s>>>(
            y, out, d.N, d.Cout, plane, nullptr, 0.0f);
        break;
    case CONV_EPI_GN_SCALE_POOL_CLAMP: {
        conv_epi_status st = ensure_post_stats(h, e.groups);
        if (st) return st;
        const int cpg = d.Cout / e.groups;
        post_gn_stats<<<(unsigned)(d.N * e.groups), kThreads, 0, s>>>(y, h->post, e.groups, cpg, plane,
                                                                      1.0 / ((double)cpg * plane), e.eps);
        CE_CUDA(cudaGetLastError());
        const int Hp = (h->Ho - e.pool_k) / e.pool_k + 1, Wp = (h->Wo - e.pool_k) / e.pool_k + 1;
        launch_gn_pool(h, y, e, out, Hp, Wp, s);
        h->last_launches = 1;
        break;
    }
    default:
        return CONV_EPI_ERR_INVALID_ARG;
    }
    CE_CUDA(cudaGetLastError());
    h->last_launches += 1;
    return CONV_EPI_OK;
}

}  // namespace conv_epi
