/*
 * oracle.h -- fp64 CPU reference for the fused 3x3 conv + epilogue chains.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this code.  It shares no
 * code, header, table or helper with the CUDA library, and neither includes
 * nor calls the other.
 *
 * Every function is the plain definition of what it computes, in double
 * precision, from float32 inputs:
 *
 *   y[n,co,i,j] = b[co] + sum_{ci,kh,kw} w[co,ci,kh,kw] * x[n,ci,i+kh,j+kw]
 *
 * for a 3x3 kernel, stride 1, no padding (so Ho = H - 2, Wo = W - 2), followed
 * by one of four chains.  The sources are four kernel-writing transcripts
 * (POPCORNBENCH, model Kimi-K2.6, level-2 problems 25, 85, 54 and 32);
 * each function names the page and the passage it follows.
 *
 * Pins (tests/test_oracle_pins.py): every function here is checked against a
 * library routine (torch CPU fp64 conv2d / group_norm / max_pool2d / gelu /
 * leaky_relu), brute force, closed forms and invariants.  No function is
 * "parity unpinned".
 *
 * Layouts: all tensors are dense, row-major, NCHW; w is [Cout][Cin][3][3].
 * Index outputs (argidx) are optional (NULL skips them).
 * Return value: 0 on success, -1 on a bad argument.
 */
#ifndef CONV_EPI_ORACLE_H
#define CONV_EPI_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Chain selectors (same numbering as the workload recipes). */
#define ORACLE_MIN_TANH2 1
#define ORACLE_SCALE_MIN 2
#define ORACLE_MUL_LRELU_GELU 3
#define ORACLE_GN_SCALE_POOL_CLAMP 4

typedef struct {
    int kind;
    double scalar;          /* MIN_TANH2 / SCALE_MIN: y is multiplied by it before the min */
    const float *mult;      /* MUL_LRELU_GELU: per-channel multiplier [Cout] */
    double lrelu_slope;     /* MUL_LRELU_GELU: LeakyReLU negative slope */
    int groups;             /* GN: number of groups */
    double eps;             /* GN: epsilon inside the square root */
    const float *gamma;     /* GN weight [Cout] */
    const float *beta;      /* GN bias [Cout] */
    const float *scale;     /* per-channel scale after GN [Cout] */
    int pool_k;             /* max-pool kernel = stride */
    double clamp_lo, clamp_hi;
} oracle_chain;

/* Output spatial sizes: conv Ho = H-2; pool floor((Ho-k)/k)+1. */
int oracle_conv_out(int H, int W, int *Ho, int *Wo);
int oracle_pool_out(int Ho, int k);
/* Output shape [4] of the whole chain. */
int oracle_output_shape(int N, int Cin, int H, int W, int Cout, const oracle_chain *c, int64_t shape[4]);

/* Full conv, y [N][Cout][Ho][Wo] in fp64; threaded over (n, co). */
int oracle_conv3x3(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                   int Cout, double *y, int nthreads);

/* Chains applied to a full fp64 conv output. */
int oracle_chain_min(const double *y, int N, int C, int Ho, int Wo, double scalar, int tanh2,
                     double *out, int32_t *argidx);
int oracle_chain_mul_lrelu_gelu(const double *y, int N, int C, int Ho, int Wo, const float *mult,
                                double slope, double *out);
int oracle_chain_gn_pool(const double *y, int N, int C, int Ho, int Wo, const oracle_chain *c,
                         double *out, int32_t *argidx, double *mean, double *rstd);

/* Whole forward (conv + chain) one image at a time, so memory stays at one
 * image's conv output per worker.  out has oracle_output_shape(); argidx is
 * the chain's index output (channel for the min chains, window offset
 * kh*pool_k+kw for the pool chain) or NULL.  Threads: over (n, co) for the
 * conv, over images for the chain. */
int oracle_forward(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                   int Cout, const oracle_chain *c, double *out, int32_t *argidx, int nthreads);

/* Point evaluations for sampled checks on full-size problems. */
double oracle_conv_at(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                      int Cout, int n, int co, int i, int j);
/* Min chains at npts pixels (n[k], i[k], j[k]). */
int oracle_min_at(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                  int Cout, double scalar, int tanh2, int npts, const int32_t *n, const int32_t *i,
                  const int32_t *j, double *out, int32_t *argidx);
/* Per-channel chain at npts points (n[k], co[k], i[k], j[k]). */
int oracle_mul_lrelu_gelu_at(const float *x, const float *w, const float *b, int N, int Cin, int H,
                             int W, int Cout, const float *mult, double slope, int npts,
                             const int32_t *n, const int32_t *co, const int32_t *i,
                             const int32_t *j, double *out);
/* GN chain for one (n, g): out [C/groups][Hp][Wp] for channels g*C/groups.. */
int oracle_gn_group(const float *x, const float *w, const float *b, int N, int Cin, int H, int W,
                    int Cout, const oracle_chain *c, int n, int g, double *out, int32_t *argidx,
                    double *mean, double *rstd, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
