/*
 * conv_epi.h -- fused 3x3 Conv2d + epilogue for NVIDIA GB300 (sm_103a).
 *
 * One call computes, for a float32 input x[N][Cin][H][W] (NCHW; in tf32 mode
 * also channels last, x[N][H][W][Cin], see conv_epi_layout), filter
 * w[Cout][Cin][3][3] and bias b[Cout],
 *
 *     y[n,co,i,j] = b[co] + sum_{ci,kh,kw} w[co,ci,kh,kw] * x[n,ci,i+kh,j+kw]
 *
 * (kernel 3, stride 1, no padding: Ho = H-2, Wo = W-2) as an implicit GEMM
 * with K = Cin*9, and applies one post-conv chain inside the GEMM epilogue.
 * The full conv output y never reaches memory when the chain reduces it.
 *
 * The chains are the four models of the POPCORNBENCH kernel-writing
 * transcripts (model Kimi-K2.6, level 2), problems
 *   p25  min over channels (keepdim) -> tanh -> tanh       CONV_EPI_MIN_TANH2
 *   p32  x scalar -> min over channels (keepdim)            CONV_EPI_SCALE_MIN
 *   p54  x multiplier[C] -> LeakyReLU -> GELU (exact erf)   CONV_EPI_MUL_LRELU_GELU
 *   p85  GroupNorm -> x scale[C] -> MaxPool(k) -> clamp     CONV_EPI_GN_SCALE_POOL_CLAMP
 * Each page states its problem as a module built with the model's arguments
 * whose forward(x) uses the module's parameters and returns the model's
 * output; here the parameters travel in the arguments of conv_epi_forward.
 *
 * Conventions for every entry point:
 *   - Tensors are dense, contiguous, row-major (NCHW; x may be NHWC, as the
 *     description's layout says), float32, and must start on a 16-byte
 *     boundary.  "device pointer" means memory the current CUDA
 *     device can read (cudaMalloc, torch CUDA tensors); "host pointer" means
 *     ordinary (ideally pinned) host memory.
 *   - The caller owns every tensor it passes; the library owns the handle and
 *     its workspace (packed weights, GroupNorm partial sums, pooled max/min,
 *     the padded copy of x for tf32 NCHW rows whose W is not a multiple of 4,
 *     and the device staging of conv_epi_forward_host).
 *   - Calls are asynchronous on the given stream unless stated otherwise and
 *     return a status; no C++ exception crosses this boundary.
 *   - A handle serves one caller at a time: its calls share its workspace,
 *     so forwards on one handle must be ordered (one stream, or streams
 *     joined by events); concurrent work takes one handle each.  Calls on
 *     different handles are independent.
 *   - There is no CPU fallback: without a usable sm_103a device, calls that
 *     compute return CONV_EPI_ERR_CUDA or CONV_EPI_ERR_UNSUPPORTED.
 *   - An empty batch (N = 0) is valid.  Its forwards check the chain as usual
 *     and return CONV_EPI_OK without device work; x and out may then be null.
 */
#ifndef CONV_EPI_H
#define CONV_EPI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONV_EPI_API __attribute__((visibility("default")))

typedef struct conv_epi_handle_s *conv_epi_handle; /* opaque, library-owned */

typedef enum {
    CONV_EPI_OK = 0,
    CONV_EPI_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad chain parameters */
    CONV_EPI_ERR_UNSUPPORTED = 2,  /* shape/chain outside what the chosen mode implements */
    CONV_EPI_ERR_ALIGNMENT = 3,    /* a tensor does not start on a 16-byte boundary */
    CONV_EPI_ERR_CUDA = 4,         /* a CUDA runtime call failed (see conv_epi_last_cuda_error) */
    CONV_EPI_ERR_TIMEOUT = 5,      /* a kernel gave up waiting on a pipeline barrier */
    CONV_EPI_ERR_NO_MEMORY = 6,    /* workspace allocation failed */
    CONV_EPI_ERR_DEVICE = 7        /* a kernel raised its own error flag */
} conv_epi_status;

/* Arithmetic of the convolution. */
typedef enum {
    CONV_EPI_MODE_TF32 = 0, /* 5th-gen tensor cores (tcgen05), tf32 operands, fp32 accumulate */
    CONV_EPI_MODE_FP32 = 1  /* CUDA cores, fp32 fused multiply-add (strict-tolerance mode) */
} conv_epi_mode;

/* Memory layout of the input x (the filter is [Cout][Cin][3][3] and every
 * output NCHW in both). */
typedef enum {
    CONV_EPI_LAYOUT_NCHW = 0, /* x[N][Cin][H][W], the layout the problem is stated in */
    CONV_EPI_LAYOUT_NHWC = 1  /* x[N][H][W][Cin] (channels last).  fp32 mode: any Cin; a first
                                 kernel transposes x into a handle-owned NCHW copy (one more read
                                 and write of x), so results equal the NCHW run's bit for bit.
                                 tf32 mode: Cin a multiple of 4 (else CONV_EPI_ERR_UNSUPPORTED).
                                 Each input tile is copied straight into the tensor core's
                                 operand layout (four channels of a position are adjacent in both),
                                 so no conversion pass runs: the tensor core uses the top 19 bits
                                 of each fp32 input (its low 13 mantissa bits are dropped, i.e.
                                 truncated toward zero) where the NCHW path rounds to nearest.  The
                                 filter is rounded to nearest in both layouts. */
} conv_epi_layout;

/* Problem description.  Kernel 3x3, stride 1, padding 0 are implied. */
typedef struct {
    int N, Cin, H, W, Cout; /* input [N][Cin][H][W] (or [N][H][W][Cin]), filter [Cout][Cin][3][3] */
    int mode;               /* conv_epi_mode */
    int layout;             /* conv_epi_layout of x; 0 = NCHW */
} conv_epi_desc;

typedef enum {
    CONV_EPI_MIN_TANH2 = 1,          /* out[n,0,i,j] = tanh(tanh(min_c scalar*y[n,c,i,j]))   [N,1,Ho,Wo] */
    CONV_EPI_SCALE_MIN = 2,          /* out[n,0,i,j] = min_c scalar*y[n,c,i,j]               [N,1,Ho,Wo] */
    CONV_EPI_MUL_LRELU_GELU = 3,     /* t = y*chan_scale[c]; t = max(t,0)+slope*min(t,0);
                                        out = 0.5 t (1 + erf(t/sqrt 2))                     [N,Cout,Ho,Wo] */
    CONV_EPI_GN_SCALE_POOL_CLAMP = 4, /* z = ((y-mean_ng)*rstd_ng*gamma[c] + beta[c]) * chan_scale[c],
                                        mean/biased var over (C/groups, Ho, Wo) of each (n, group),
                                        rstd = 1/sqrt(var+eps); out = clamp(maxpool_k(z), lo, hi)
                                        with stride k, floor mode                  [N,Cout,Hp,Wp] */
    CONV_EPI_NONE = 5                /* out = y, the conv output itself (bias added), no chain:
                                        on every page the reference model's first layer is this
                                        nn.Conv2d, whose output the chain then consumes (p25, the
                                        analysis of the reference model)            [N,Cout,Ho,Wo] */
} conv_epi_kind;

/* Post-conv chain.  Parameter tensors are device pointers of Cout floats
 * (host pointers for conv_epi_forward_host). */
typedef struct {
    int kind;                 /* conv_epi_kind */
    float scalar;             /* MIN kinds: multiplier before the min (any sign; 1 = none) */
    const float *chan_scale;  /* MUL_LRELU_GELU: multiplier[Cout]; GN kind: scale[Cout] after the norm */
    float lrelu_slope;        /* MUL_LRELU_GELU: LeakyReLU negative slope (0.01 on the page) */
    int groups;               /* GN: number of groups, divides Cout */
    float eps;                /* GN: added to the variance inside the square root */
    const float *gamma;       /* GN: weight[Cout] */
    const float *beta;        /* GN: bias[Cout] */
    int pool_k;               /* GN: max-pool kernel and stride (>= 1) */
    float clamp_lo, clamp_hi; /* GN: clamp bounds after the pool (lo <= hi) */
    int32_t *index_out;       /* optional device pointer, NULL to skip; same shape as out:
                                 MIN kinds -> channel of the minimum (first on ties);
                                 GN kind   -> window offset a*k+b of the pooled value
                                              (first row-major on ties);
                                 MUL_LRELU_GELU, NONE -> not produced (must be NULL).
                                 Only CONV_EPI_MODE_FP32 produces indices. */
} conv_epi_epilogue_desc;

/* Output shape of a chain: shape[4] = {N, C, Ho', Wo'}.  Pure host call.
 * The min chains reduce with keepdim (C = 1); without keepdim the same
 * N*Ho*Wo floats are the [N][Ho][Wo] tensor, so one output serves both. */
CONV_EPI_API conv_epi_status conv_epi_output_shape(const conv_epi_desc *desc,
                                                   const conv_epi_epilogue_desc *epi,
                                                   int64_t shape[4]);

/* Create a handle for one problem size and mode on the current CUDA device.
 * This is the construction step of the problem as every page states it: a
 * module built once with the model's arguments (in_channels, out_channels,
 * kernel_size 3 and the chain's constants; p85 and p54, the ModelNew module
 * and its __init__), here the sizes of x and the filter and the arithmetic
 * mode.  desc: read during the call only (the handle keeps a copy).
 * *out: receives the new handle, or NULL when the call fails.
 * Errors: INVALID_ARG (null pointer, sizes < 1, H or W < 3, unknown mode or
 * layout), UNSUPPORTED (shape or device outside the chosen mode, a tensor of
 * 2^31 or more elements, a device that is not sm_103a), CUDA / NO_MEMORY
 * (workspace allocation). 
 * Validates the description and allocates the workspace every chain needs
 * except the GN chain's pooled buffers, which are allocated on the first GN
 * forward (conv_epi_reserve allocates them up front).  Synchronous.
 *
 * Shapes:
 *   CONV_EPI_MODE_FP32: any N, Cin, Cout and H, W >= 3.
 *     GN chain: fused into the fp32 kernel for pool_k 1, 2 or 4 and at
 *     most 64 groups (window indices available); any other pool_k or group
 *     count runs as two passes, the fp32 conv writing y into a handle-owned
 *     buffer (conv_epi_reserve or the first GN forward allocates it) and the
 *     chain's post-pass, without indices (index_out: UNSUPPORTED).
 *   CONV_EPI_MODE_TF32: any N, Cin, Cout and H, W >= 3.
 *     GN chain: fused into the conv kernel for groups of a power-of-two
 *     number of channels up to 64 and either pool_k = 4 with Cout <= 64 and
 *     W <= 64 or W >= 66 (wider than 256 as column tiles of 252 outputs), or
 *     with Cout > 64 and
 *     W <= 64 or 66 <= W <= 128 (more than 128 channels as channel tiles of
 *     128), or with 64 < Cout <= 128 and 130 <= W <= 256, or
 *     pool_k = 2 with Cout <= 128 and W <= 128 (not 65), or Cout <= 64 and
 *     130 <= W <= 256 where its pooled tile fits the shared memory beside
 *     the smallest rings (NCHW with Cin <= 8: W <= 240; channels last: up
 *     to 256);
 *     any other GN
 *     shape runs as two passes, the tensor-core conv
 *     writing y (bias added) and its per-unit sums of y and y^2 into a
 *     handle-owned buffer (conv_epi_plan.ybuf_bytes; allocated by
 *     conv_epi_reserve or the first GN forward), then the statistics folded
 *     from those sums and the normalise-scale-pool-clamp pass over y (fp32).
 *     Rows wider than 256 run as column tiles, more than 128 output channels
 *     as channel tiles.  NCHW rows whose W is not a multiple of 4 are first
 *     copied, by a small kernel, into a handle-owned buffer of rows padded to
 *     a multiple of 4 floats (the tensor load needs 16-byte row strides):
 *     one more read and write of x.  The GN chain runs as one cooperative
 *     launch (every CTA resident) that finalizes inside the kernel; where the
 *     device refuses that launch, a second finalize kernel follows.
 *   Other shapes return CONV_EPI_ERR_UNSUPPORTED: at create, or at the first
 *   forward for chain-specific limits.
 * Debug mode: with the environment variable CONV_EPI_DEBUG set to "1" when
 * the handle is created, every conv_epi_forward on it waits for its stream
 * and returns the device-side status itself (as conv_epi_sync would), so a
 * barrier timeout surfaces at the call that caused it.  Such forwards cannot
 * be captured into a CUDA graph. */
CONV_EPI_API conv_epi_status conv_epi_create(const conv_epi_desc *desc, conv_epi_handle *out);

/* Allocate, ahead of the first forward, whatever workspace `epi` will need
 * (so that forward itself never allocates, e.g. before graph capture). */
CONV_EPI_API conv_epi_status conv_epi_reserve(conv_epi_handle h, const conv_epi_epilogue_desc *epi);

/* Run conv + chain on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  This is the module's forward(x) as the pages state it (p85 and
 * p54, ModelNew.forward: the conv with the module's weight and bias, then
 * the model's chain, returning the chain's output); the parameters the
 * module would hold travel as arguments: w [Cout][Cin][3][3], b [Cout] and
 * the chain's tensors in `epi`.  x, w, b, the chain's parameter tensors and
 * out are device pointers owned by the caller, read (x, w, b, parameters) or
 * written (out, index_out) by kernels on `stream` after the call returns;
 * out must hold conv_epi_output_shape() floats.  Asynchronous: argument
 * errors are returned at once (INVALID_ARG, ALIGNMENT, UNSUPPORTED), launch
 * failures as CUDA, device-side errors (a barrier wait that timed out) by
 * conv_epi_sync(). */
CONV_EPI_API conv_epi_status conv_epi_forward(conv_epi_handle h, const float *x, const float *w,
                                              const float *b, const conv_epi_epilogue_desc *epi,
                                              float *out, void *stream);

/* Same computation from HOST buffers.  Every pointer (including those inside
 * `epi`) is a host pointer; pinned memory lets the copies run asynchronously.
 * w, b and the chain's parameters are copied on `stream` into library-owned
 * device staging (kept by the handle, grown to the largest call, freed by
 * conv_epi_destroy).  The batch then goes in up to eight slices of whole
 * images (one slice when an image is not a whole number of 16-byte units in
 * or out): slice k's input copy runs on a library-owned copy stream while
 * slice k-1 is computed on `stream` and slice k-2's result copies back on a
 * second library-owned stream, joined by events.  Synchronous: returns after
 * the last result copy, with the device-side status as conv_epi_sync(). */
CONV_EPI_API conv_epi_status conv_epi_forward_host(conv_epi_handle h, const float *x, const float *w,
                                                   const float *b, const conv_epi_epilogue_desc *epi,
                                                   float *out, void *stream);

/* Forward for callers that cannot allocate device memory (no counterpart on
 * the pages: it exists for users of this library).  Code that runs inside a
 * custom allocator or memory-pool callback, code that must not grow the
 * device's memory footprint after start-up, or a runtime that lends this
 * library only its input and output buffers cannot call conv_epi_create,
 * which allocates the scratch the tensor-core kernel needs.  This call takes
 * the problem description instead of a handle and keeps that scratch (the
 * packed tf32 filter) in a fixed 1 MiB array inside the library's device
 * image, which every GPU that loads the library holds until the process
 * exits.  It allocates and frees nothing.
 *   desc: as for conv_epi_create; mode must be CONV_EPI_MODE_TF32.
 *   x, w, b, the chain's parameters, out: device pointers as for
 *   conv_epi_forward.  Chains MIN_TANH2, SCALE_MIN, MUL_LRELU_GELU and NONE
 *   (the GroupNorm chain needs a larger workspace); index_out must be NULL.
 * The description and the chain are checked exactly as conv_epi_create and
 * conv_epi_forward check them, with the same statuses.
 * Returns CONV_EPI_ERR_UNSUPPORTED when the packed filter of the problem does
 * not fit the array (Cin rounded up to a multiple of 8, times 3*(2S+1)*Cout
 * floats, plus one 8-channel chunk, with S = 128/Cout), when an NCHW input's W
 * is not a multiple of 4 (that needs the padded copy's buffer), or when the
 * shape is outside the tensor-core path.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress) and
 * clears its error word with a synchronous cudaMemset, so make that first
 * call before any stream capture.  Every call on a device shares the array
 * and the array keeps the last call's contents; each call rewrites the part
 * it reads, so nothing needs to start at zero, but calls whose kernels
 * overlap on the GPU (unordered streams) race on it.  Asynchronous on
 * `stream` like conv_epi_forward; a device-side barrier timeout is recorded
 * in an error word beside the array (one per device), which
 * conv_epi_noalloc_sync reports and clears. */
CONV_EPI_API conv_epi_status conv_epi_forward_noalloc(const conv_epi_desc *desc, const float *x, const float *w,
                                                      const float *b, const conv_epi_epilogue_desc *epi, float *out,
                                                      void *stream);

/* Wait for `stream`, then report and clear the error word of the
 * allocation-free forwards on the current device: CONV_EPI_ERR_TIMEOUT when
 * one of their kernels gave up waiting on a pipeline barrier since the last
 * call (its output is then undefined), else CONV_EPI_OK.  The word is shared
 * by every allocation-free forward on the device.  Allocates nothing
 * (the first call on a device looks up the word's address, as the first
 * forward does).  Synchronous. */
CONV_EPI_API conv_epi_status conv_epi_noalloc_sync(void *stream);

/* The chain alone, as a separate pass over a conv output that is already in
 * memory: the structure each page designs its kernels for, with the
 * convolution left to a library call that writes y in full (p25 and p32: a
 * post-pass that takes the channel minimum per pixel; p54: one elementwise
 * pass; p85: a GroupNorm statistics kernel, then one kernel that
 * normalises, scales, max-pools and clamps).  For comparing the fused
 * forward with that design on one machine, and for callers that hold y.
 *   h: a handle for the problem (its description gives N, Cout, Ho, Wo; the
 *      mode and layout do not matter here: the pass computes in fp32).
 *   y: device pointer, the conv output [N][Cout][Ho][Wo] float32 with the
 *      bias added, 16-byte aligned; read only.
 *   epi: the chain, as for conv_epi_forward; index_out must be NULL.
 *   out: device pointer, conv_epi_output_shape() floats, 16-byte aligned.
 * Asynchronous on `stream`.  The GroupNorm chain keeps its statistics in a
 * handle-owned buffer allocated on the first such call.  Returns
 * INVALID_ARG / ALIGNMENT for bad arguments, UNSUPPORTED when index_out is
 * set, CUDA or NO_MEMORY on a failing CUDA call. */
CONV_EPI_API conv_epi_status conv_epi_postpass(conv_epi_handle h, const float *y, const conv_epi_epilogue_desc *epi,
                                               float *out, void *stream);

/* The tensor-core kernel's plan for one problem and chain, as a forward on
 * a handle would launch it: tiling, ring stages, the shared-memory layout,
 * the tensor-load box and the filter operand layout.  For diagnostics and
 * host-side tests of the kernel's index ranges; a pure host call (no device
 * is needed).  Every field is an int64_t; sizes are in bytes unless stated. */
typedef struct {
    int64_t struct_bytes;    /* sizeof(conv_epi_plan), set by the call */
    int64_t gemm_cout;       /* output channels per channel tile of the GEMM: 64 or 128 */
    int64_t S;               /* output rows stacked in the 128 accumulator lanes (128 / gemm_cout) */
    int64_t P;               /* positions per accumulator row (the MMA's N) */
    int64_t U;               /* accumulator row sets per unit */
    int64_t RU;              /* output rows per unit (U * S) */
    int64_t Rin;             /* input rows staged per unit (RU + 2) */
    int64_t PL;              /* 16-byte rows per 4-channel group of a B plane */
    int64_t ucol;            /* tensor-memory columns per accumulator row set */
    int64_t chunks;          /* 8-channel K chunks */
    int64_t CT;              /* column tiles per output row */
    int64_t CW;              /* output columns per column tile */
    int64_t BW;              /* staged row width, floats (NCHW) */
    int64_t MT;              /* channel tiles */
    int64_t units_per_image; /* row blocks x column tiles x channel tiles */
    int64_t resident;        /* 1: the whole packed filter stays in shared memory */
    int64_t na, nb, nr;      /* ring stages: filter chunks, B planes, staged input tiles */
    int64_t a_bytes, b_bytes, raw_bytes, scratch_bytes;  /* one stage of each ring; the epilogue scratch */
    int64_t a_off, b_off, raw_off, bar_off, scratch_off; /* shared-memory offsets */
    int64_t bar_bytes;       /* the mbarriers */
    int64_t smem;            /* dynamic shared memory per CTA */
    int64_t smem_limit;      /* the most the kernel requests */
    int64_t a_plane_bytes, a_lbo, a_kw_stride;  /* filter operand: one plane, K-group stride, tap stride */
    int64_t x_pitch;         /* floats between input rows as the tensor load reads them (NCHW) */
    int64_t box[4];          /* tensor-load box: NCHW (BW, Rin, 8, 1); NHWC (4, P, Rin, 1) */
    int64_t acc_cols;        /* tensor-memory columns per accumulator buffer (two buffers) */
    int64_t tmem_cols;       /* tensor-memory columns the kernel allocates */
    int64_t conv_items;      /* converter work items the kernel holds per chunk */
    int64_t wpack_bytes;     /* the handle's packed-filter buffer */
    int64_t xpad_bytes;      /* the handle's padded copy of x (0 unless NCHW rows need it) */
    int64_t gn_two_pass;     /* 1: a GroupNorm shape the fused epilogue does not take; the plan is
                                that of the plain conv (CONV_EPI_NONE), its first pass */
    int64_t ybuf_bytes;      /* the handle's buffer for that two-pass form (else 0): the conv output, then
                                the conv kernel's per-unit sums of y and y^2 that the statistics fold */
} conv_epi_plan;

/* Fill *plan for desc (mode must be CONV_EPI_MODE_TF32) and epi.  Returns
 * CONV_EPI_ERR_INVALID_ARG for a null pointer or an invalid description or
 * chain, CONV_EPI_ERR_UNSUPPORTED where the tensor-core kernel refuses the
 * shape (as conv_epi_create / conv_epi_forward would; *plan is then filled
 * as far as a plan exists, else zero), else CONV_EPI_OK. */
CONV_EPI_API conv_epi_status conv_epi_plan_query(const conv_epi_desc *desc, const conv_epi_epilogue_desc *epi,
                                                 conv_epi_plan *plan);

/* Wait for `stream` and report any device-side error flag the library's
 * kernels raised on this handle since the last call (then clear it). */
CONV_EPI_API conv_epi_status conv_epi_sync(conv_epi_handle h, void *stream);

/* Test hook for the bounded barrier waits (tf32 mode only).  The next
 * conv_epi_forward on this handle has each CTA's producer skip one copy: the
 * staged input tile with index `tile` in that CTA's own sequence (0 = its
 * first).  The copy is neither issued nor announced on its barrier, so the
 * converters waiting on that slot give up after the wait limit (2 s), raise
 * the timeout bit and every role of the CTA drains and returns;
 * conv_epi_sync() then reports CONV_EPI_ERR_TIMEOUT and the context stays
 * usable.  The output of that forward is undefined.  tile = -1 cancels; the
 * setting applies to one forward only.  Returns CONV_EPI_ERR_UNSUPPORTED on
 * an fp32-mode handle (whose kernels have no barrier rings).  With h = NULL
 * the setting applies to the next conv_epi_forward_noalloc made by the
 * calling thread instead (conv_epi_noalloc_sync then reports the timeout). */
CONV_EPI_API conv_epi_status conv_epi_test_drop_tile(conv_epi_handle h, int tile);

/* Release the handle and its workspace (synchronises the device first):
 * the end of the module's life (p85 and p54, the ModelNew module, whose
 * parameters and buffers go with it).  The handle must not be used after
 * the call.  Returns INVALID_ARG for a null handle, CUDA when the
 * synchronisation reports an error (the handle is released all the same). */
CONV_EPI_API conv_epi_status conv_epi_destroy(conv_epi_handle h);

/* Bytes of device workspace the handle holds now. */
CONV_EPI_API size_t conv_epi_workspace_bytes(conv_epi_handle h);

/* Number of kernel launches the last conv_epi_forward issued. */
CONV_EPI_API int conv_epi_last_launch_count(conv_epi_handle h);

/* Static strings; never NULL. */
CONV_EPI_API const char *conv_epi_status_string(conv_epi_status s);
CONV_EPI_API const char *conv_epi_last_cuda_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
CONV_EPI_API int conv_epi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CONV_EPI_H */
