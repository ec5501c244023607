/*
 * oracle.c -- fp64 CPU reference for the fused 3x3 conv + epilogue chains.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain loops in double precision;
 * the only "library" calls are tanh/erf/sqrt from <math.h>.  Threads only
 * split independent outputs between workers; no sum is reordered across
 * workers.
 *
 * Pages (POPCORNBENCH transcripts, model Kimi-K2.6, level 2):
 *   p25  Conv2d(16->64, k=3) -> min over channels (keepdim) -> tanh -> tanh
 *   p85  Conv2d(8->64, k=3) -> GroupNorm(16) -> x scale[C,1,1] -> MaxPool2d(4) -> clamp[0,1]
 *   p54  Conv2d(64->64, k=3) -> x multiplier[C,1,1] -> LeakyReLU(0.01) -> GELU
 *   p32  Conv2d(64->128, k=3) -> x 2.0 -> min over channels (keepdim)
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* a minimal parallel-for: tasks 0..ntasks-1 handed out by an atomic counter */
/* ------------------------------------------------------------------------ */
typedef void (*task_fn)(void *ctx, int64_t task);
typedef struct {
    task_fn fn;
    void *ctx;
    int64_t ntasks;
    atomic_llong next;
} pool_job;

static void *pool_worker(void *arg) {
    pool_job *job = (pool_job *)arg;
    for (;;) {
        int64_t t = atomic_fetch_add(&job->next, 1);
        if (t >= job->ntasks) break;
        job->fn(job->ctx, t);
    }
    return NULL;
}

static void parallel_for(int nthreads, int64_t ntasks, task_fn fn, void *ctx) {
    pool_job job;
    job.fn = fn;
    job.ctx = ctx;
    job.ntasks = ntasks;
    atomic_init(&job.next, 0);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > ntasks) nthreads = (int)(ntasks > 0 ? ntasks : 1);
    pthread_t th[256];
    int started = 0;
    for (int k = 1; k < nthreads; ++k)
        if (pthread_create(&th[started], NULL, pool_worker, &job) == 0) ++started;
    pool_worker(&job);
    for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
}

/* ------------------------------------------------------------------------ */
/* shapes                                                                   */
/* ------------------------------------------------------------------------ */

/* Conv2d with kernel 3, stride 1, padding 0, dilation 1: Ho = H - 3 + 1.
 * p85, reference-model analysis: "output size = H_out = H - k + 1 = 126";
 * p54, shape analysis: 256 - 3 + 1 = 254. */
int oracle_conv_out(int H, int W, int *Ho, int *Wo) {
    if (H < 3 || W < 3) return -1;
    *Ho = H - 3 + 1;
    *Wo = W - 3 + 1;
    return 0;
}

/* MaxPool2d(kernel k), stride k, padding 0, floor mode:
 * floor((Ho + 2*0 - 1*(k-1) - 1) / k + 1) = floor((Ho - k) / k) + 1.
 * p85, reference-model analysis: floor((126 - 4)/4 + 1) = 31. */
int oracle_pool_out(int Ho, int k) {
    if (k < 1 || Ho < k) return 0;
    return (Ho - k) / k + 1;
}

int oracle_output_shape(int N, int Cin, int H, int W, int Cout, const oracle_chain *c,
                        int64_t shape[4]) {
    int Ho, Wo;
    (void)Cin;
    if (!c || oracle_conv_out(H, W, &Ho, &Wo)) return -1;
    shape[0] = N;
    switch (c->kind) {
    case ORACLE_MIN_TANH2:
    case ORACLE_SCALE_MIN:
        /* keepdim=True: one channel */
        shape[1] = 1, shape[2] = Ho, shape[3] = Wo;
        return 0;
    case ORACLE_MUL_LRELU_GELU:
        shape[1] = Cout, shape[2] = Ho, shape[3] = Wo;
        return 0;
    case ORACLE_GN_SCALE_POOL_CLAMP:
        shape[1] = Cout;
        shape[2] = oracle_pool_out(Ho, c->pool_k);
        shape[3] = oracle_pool_out(Wo, c->pool_k);
        return 0;
    default:
        return -1;
    }
}

/* ------------------------------------------------------------------------ */
/* convolution                                                              */
/* ------------------------------------------------------------------------ */

/* One output of nn.Conv2d(Cin, Cout, 3) (bias=True, stride 1, no padding):
 * the bias plus the 3x3xCin window of x times the filter, as the p54 page
 * writes it out for its fused-conv design ("acc += in_val * w_val" over c_in,
 * kh, kw, then the per-channel chain). */
double oracle_conv_at(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                      int Cout, int n, int co, int i, int j) {
    (void)N;
    (void)Cout;
    double acc = (double)b[co];
    for (int ci = 0; ci < Cin; ++ci)
        for (int kh = 0; kh < 3; ++kh)
            for (int kw = 0; kw < 3; ++kw)
                acc += (double)w[((int64_t)co * Cin + ci) * 9 + kh * 3 + kw] *
                       (double)x[(((int64_t)n * Cin + ci) * H + (i + kh)) * W + (j + kw)];
    return acc;
}

typedef struct {
    const float *x, *w, *b;
    int N, Cin, H, W, Cout, Ho, Wo;
    int n0;          /* first image of this call */
    double *y;       /* [nimg][Cout][Ho][Wo] */
} conv_ctx;

static void conv_task(void *p, int64_t t) {
    conv_ctx *c = (conv_ctx *)p;
    int nl = (int)(t / c->Cout), co = (int)(t % c->Cout);
    double *yo = c->y + ((int64_t)nl * c->Cout + co) * c->Ho * c->Wo;
    for (int i = 0; i < c->Ho; ++i)
        for (int j = 0; j < c->Wo; ++j)
            yo[(int64_t)i * c->Wo + j] =
                oracle_conv_at(c->x, c->w, c->b, c->N, c->Cin, c->H, c->W, c->Cout, c->n0 + nl, co, i, j);
}

static int conv_images(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                       int Cout, int n0, int nimg, double *y, int nthreads) {
    conv_ctx c;
    c.x = x, c.w = w, c.b = b, c.N = N, c.Cin = Cin, c.H = H, c.W = W, c.Cout = Cout;
    if (oracle_conv_out(H, W, &c.Ho, &c.Wo)) return -1;
    c.n0 = n0, c.y = y;
    parallel_for(nthreads, (int64_t)nimg * Cout, conv_task, &c);
    return 0;
}

int oracle_conv3x3(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                   int Cout, double *y, int nthreads) {
    if (!x || !w || !b || !y || N < 0 || Cin < 1 || Cout < 1) return -1;
    return conv_images(x, w, b, N, Cin, H, W, Cout, 0, N, y, nthreads);
}

/* ------------------------------------------------------------------------ */
/* chains                                                                   */
/* ------------------------------------------------------------------------ */

/* p25 reference-model analysis: torch.min(x, dim=1, keepdim=True)[0], then
 * tanh applied twice (the page keeps both: it does not simplify tanh(tanh)).
 * p32 reference-model analysis: multiply by scale_factor (2.0) first, then
 * the channel min.  Here: m = min over c of (scalar * y[c]); tanh2 selects the
 * two tanh's.  argidx = the first channel that attains the minimum. */
static void min_chain_pixel(const double *ycol, int64_t cstride, int C, double scalar, int tanh2,
                            double *out, int32_t *arg) {
    double m = INFINITY;
    int32_t am = -1;
    for (int c = 0; c < C; ++c) {
        double v = scalar * ycol[(int64_t)c * cstride];
        if (am < 0 || v < m) { /* strict '<': ties keep the first channel */
            m = v;
            am = c;
        }
    }
    if (tanh2) m = tanh(tanh(m));
    *out = m;
    if (arg) *arg = am;
}

int oracle_chain_min(const double *y, int N, int C, int Ho, int Wo, double scalar, int tanh2,
                     double *out, int32_t *argidx) {
    if (!y || !out) return -1;
    int64_t hw = (int64_t)Ho * Wo;
    for (int n = 0; n < N; ++n)
        for (int64_t p = 0; p < hw; ++p)
            min_chain_pixel(y + (int64_t)n * C * hw + p, hw, C, scalar, tanh2, &out[(int64_t)n * hw + p],
                            argidx ? &argidx[(int64_t)n * hw + p] : NULL);
    return 0;
}

/* p54 reference-model analysis and fused-kernel passages:
 *   v = y * multiplier[c]              (multiplier has shape (C,1,1))
 *   v = LeakyReLU(v) = max(0,v) + slope * min(0,v), slope 0.01
 *   v = GELU(v) = 0.5 * v * (1 + erf(v / sqrt(2)))   (approximate='none')  */
static double mul_lrelu_gelu(double y, double mult, double slope) {
    double v = y * mult;
    v = (v > 0.0 ? v : 0.0) + slope * (v < 0.0 ? v : 0.0);
    return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
}

int oracle_chain_mul_lrelu_gelu(const double *y, int N, int C, int Ho, int Wo, const float *mult,
                                double slope, double *out) {
    if (!y || !out || !mult) return -1;
    int64_t hw = (int64_t)Ho * Wo;
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C; ++c)
            for (int64_t p = 0; p < hw; ++p) {
                int64_t k = ((int64_t)n * C + c) * hw + p;
                out[k] = mul_lrelu_gelu(y[k], (double)mult[c], slope);
            }
    return 0;
}

/* p85 GroupNorm passages: view the conv output as (N, G, C/G, H, W); per
 * (n, g) mean and biased variance (unbiased=False) over (C/G, H, W) -- the
 * conv bias stays inside these statistics, because a per-channel constant
 * changes the group variance; normalise (v - mean) / sqrt(var + eps); affine
 * v * gamma[c] + beta[c]; then v * scale[c]; MaxPool2d(k) with stride k,
 * no padding, floor mode (rows/cols past the last full window are dropped
 * from the pool but not from the statistics); clamp to [lo, hi].
 * Statistics here are two-pass in fp64.  argidx = offset kh*k + kw of the
 * first (row-major) window position holding the pooled maximum. */
static int gn_one(const double *yimg, int C, int Ho, int Wo, const oracle_chain *c, int g,
                  double *out_img, int32_t *arg_img, double *mean_o, double *rstd_o) {
    int cpg = C / c->groups;
    int64_t hw = (int64_t)Ho * Wo;
    const double *yg = yimg + (int64_t)g * cpg * hw;
    int64_t cnt = (int64_t)cpg * hw;
    double s = 0.0;
    for (int64_t k = 0; k < cnt; ++k) s += yg[k];
    double mean = s / (double)cnt;
    double ss = 0.0;
    for (int64_t k = 0; k < cnt; ++k) {
        double d = yg[k] - mean;
        ss += d * d;
    }
    double var = ss / (double)cnt;
    double rstd = 1.0 / sqrt(var + c->eps);
    if (mean_o) *mean_o = mean;
    if (rstd_o) *rstd_o = rstd;
    int k = c->pool_k;
    int Hp = oracle_pool_out(Ho, k), Wp = oracle_pool_out(Wo, k);
    for (int cl = 0; cl < cpg; ++cl) {
        int ch = g * cpg + cl;
        const double *yc = yg + (int64_t)cl * hw;
        for (int ph = 0; ph < Hp; ++ph)
            for (int pw = 0; pw < Wp; ++pw) {
                double best = -INFINITY;
                int32_t barg = -1;
                for (int a = 0; a < k; ++a)
                    for (int bb = 0; bb < k; ++bb) {
                        double v = yc[(int64_t)(ph * k + a) * Wo + (pw * k + bb)];
                        v = ((v - mean) * rstd * (double)c->gamma[ch] + (double)c->beta[ch]) * (double)c->scale[ch];
                        if (barg < 0 || v > best) {
                            best = v;
                            barg = a * k + bb;
                        }
                    }
                double o = best;
                if (o < c->clamp_lo) o = c->clamp_lo;
                if (o > c->clamp_hi) o = c->clamp_hi;
                int64_t oi = ((int64_t)ch * Hp + ph) * Wp + pw;
                out_img[oi] = o;
                if (arg_img) arg_img[oi] = barg;
            }
    }
    return 0;
}

static int gn_valid(int C, int Ho, int Wo, const oracle_chain *c) {
    return c && c->groups > 0 && C % c->groups == 0 && c->pool_k > 0 && Ho >= c->pool_k &&
           Wo >= c->pool_k && c->gamma && c->beta && c->scale;
}

int oracle_chain_gn_pool(const double *y, int N, int C, int Ho, int Wo, const oracle_chain *c,
                         double *out, int32_t *argidx, double *mean, double *rstd) {
    if (!y || !out || !gn_valid(C, Ho, Wo, c)) return -1;
    int Hp = oracle_pool_out(Ho, c->pool_k), Wp = oracle_pool_out(Wo, c->pool_k);
    int64_t hw = (int64_t)Ho * Wo, phw = (int64_t)Hp * Wp;
    for (int n = 0; n < N; ++n)
        for (int g = 0; g < c->groups; ++g)
            gn_one(y + (int64_t)n * C * hw, C, Ho, Wo, c, g, out + (int64_t)n * C * phw,
                   argidx ? argidx + (int64_t)n * C * phw : NULL, mean ? &mean[n * c->groups + g] : NULL,
                   rstd ? &rstd[n * c->groups + g] : NULL);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* whole forward, one image at a time                                       */
/* ------------------------------------------------------------------------ */
static int apply_chain(const double *y, int nimg, int C, int Ho, int Wo, const oracle_chain *c,
                       double *out, int32_t *arg) {
    switch (c->kind) {
    case ORACLE_MIN_TANH2:
        return oracle_chain_min(y, nimg, C, Ho, Wo, c->scalar, 1, out, arg);
    case ORACLE_SCALE_MIN:
        return oracle_chain_min(y, nimg, C, Ho, Wo, c->scalar, 0, out, arg);
    case ORACLE_MUL_LRELU_GELU:
        return oracle_chain_mul_lrelu_gelu(y, nimg, C, Ho, Wo, c->mult, c->lrelu_slope, out);
    case ORACLE_GN_SCALE_POOL_CLAMP:
        return oracle_chain_gn_pool(y, nimg, C, Ho, Wo, c, out, arg, NULL, NULL);
    default:
        return -1;
    }
}

int oracle_forward(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                   int Cout, const oracle_chain *c, double *out, int32_t *argidx, int nthreads) {
    int64_t shape[4];
    int Ho, Wo;
    if (!x || !w || !b || !out || !c || oracle_output_shape(N, Cin, H, W, Cout, c, shape) ||
        oracle_conv_out(H, W, &Ho, &Wo))
        return -1;
    if (c->kind == ORACLE_MUL_LRELU_GELU && !c->mult) return -1;
    if (c->kind == ORACLE_GN_SCALE_POOL_CLAMP && !gn_valid(Cout, Ho, Wo, c)) return -1;
    int64_t per_out = shape[1] * shape[2] * shape[3];
    double *y = (double *)malloc(sizeof(double) * (size_t)Cout * Ho * Wo);
    if (!y) return -1;
    for (int n = 0; n < N; ++n) {
        conv_images(x, w, b, N, Cin, H, W, Cout, n, 1, y, nthreads);
        if (apply_chain(y, 1, Cout, Ho, Wo, c, out + (int64_t)n * per_out,
                        argidx ? argidx + (int64_t)n * per_out : NULL)) {
            free(y);
            return -1;
        }
    }
    free(y);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* sampled evaluation                                                       */
/* ------------------------------------------------------------------------ */
int oracle_min_at(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                  int Cout, double scalar, int tanh2, int npts, const int32_t *n, const int32_t *i,
                  const int32_t *j, double *out, int32_t *argidx) {
    if (!x || !w || !b || !n || !i || !j || !out) return -1;
    double *col = (double *)malloc(sizeof(double) * (size_t)Cout);
    if (!col) return -1;
    for (int k = 0; k < npts; ++k) {
        for (int co = 0; co < Cout; ++co) col[co] = oracle_conv_at(x, w, b, N, Cin, H, W, Cout, n[k], co, i[k], j[k]);
        min_chain_pixel(col, 1, Cout, scalar, tanh2, &out[k], argidx ? &argidx[k] : NULL);
    }
    free(col);
    return 0;
}

int oracle_mul_lrelu_gelu_at(const float *x, const float *w, const float *b, int N, int Cin, int H,
                             int W, int Cout, const float *mult, double slope, int npts,
                             const int32_t *n, const int32_t *co, const int32_t *i,
                             const int32_t *j, double *out) {
    if (!x || !w || !b || !mult || !n || !co || !i || !j || !out) return -1;
    for (int k = 0; k < npts; ++k)
        out[k] = mul_lrelu_gelu(oracle_conv_at(x, w, b, N, Cin, H, W, Cout, n[k], co[k], i[k], j[k]),
                                (double)mult[co[k]], slope);
    return 0;
}

typedef struct {
    const float *x, *w, *b;
    int N, Cin, H, W, Cout, Ho, Wo, n, c0;
    double *slab; /* [Cout][Ho][Wo]; only channels c0.. are written */
} group_ctx;

static void group_row_task(void *p, int64_t t) {
    group_ctx *g = (group_ctx *)p;
    int cl = (int)(t / g->Ho), r = (int)(t % g->Ho);
    int co = g->c0 + cl;
    double *yo = g->slab + ((int64_t)co * g->Ho + r) * g->Wo;
    for (int s = 0; s < g->Wo; ++s)
        yo[s] = oracle_conv_at(g->x, g->w, g->b, g->N, g->Cin, g->H, g->W, g->Cout, g->n, co, r, s);
}

int oracle_gn_group(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                    int Cout, const oracle_chain *c, int n, int g, double *out, int32_t *argidx,
                    double *mean, double *rstd, int nthreads) {
    int Ho, Wo;
    if (!x || !w || !b || !out || oracle_conv_out(H, W, &Ho, &Wo) || !gn_valid(Cout, Ho, Wo, c) || n < 0 ||
        n >= N || g < 0 || g >= c->groups)
        return -1;
    int cpg = Cout / c->groups;
    int64_t hw = (int64_t)Ho * Wo;
    int Hp = oracle_pool_out(Ho, c->pool_k), Wp = oracle_pool_out(Wo, c->pool_k);
    int64_t phw = (int64_t)Hp * Wp;
    /* the image's conv output, of which only group g's channels are computed */
    double *slab = (double *)calloc((size_t)Cout * hw, sizeof(double));
    double *oimg = (double *)calloc((size_t)Cout * phw, sizeof(double));
    int32_t *aimg = argidx ? (int32_t *)calloc((size_t)Cout * phw, sizeof(int32_t)) : NULL;
    if (!slab || !oimg || (argidx && !aimg)) {
        free(slab), free(oimg), free(aimg);
        return -1;
    }
    group_ctx gc;
    gc.x = x, gc.w = w, gc.b = b, gc.N = N, gc.Cin = Cin, gc.H = H, gc.W = W, gc.Cout = Cout;
    gc.Ho = Ho, gc.Wo = Wo, gc.n = n, gc.c0 = g * cpg, gc.slab = slab;
    parallel_for(nthreads, (int64_t)cpg * Ho, group_row_task, &gc);
    gn_one(slab, Cout, Ho, Wo, c, g, oimg, aimg, mean, rstd);
    memcpy(out, oimg + (int64_t)g * cpg * phw, sizeof(double) * (size_t)cpg * phw);
    if (argidx) memcpy(argidx, aimg + (int64_t)g * cpg * phw, sizeof(int32_t) * (size_t)cpg * phw);
    free(slab), free(oimg), free(aimg);
    return 0;
}
