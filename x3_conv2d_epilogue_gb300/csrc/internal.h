// internal.h -- declarations shared by the translation units of libconv_epi.
// Nothing here is visible through the C ABI (include/conv_epi.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "conv_epi.h"

namespace conv_epi {

// Device error word bits (ORed by kernels into handle->dev_err[0]).
enum : unsigned {
    ERRBIT_TIMEOUT = 1u,  // a bounded barrier wait ran out
    ERRBIT_BOUNDS = 2u,   // a kernel's own bounds check refused an access
    ERRBIT_TMEM = 4u,     // tensor-memory allocation returned an unexpected address
};

// Where the bounded waits give up (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// GroupNorm-chain workspace, written by either conv path and read by the
// finalize kernel.  For each (n, c, ph, pw) of the pooled output:
//   pmax / pmin : max / min of y = conv + bias over the k x k window (the
//                 tf32 path leaves only the one the channel's slope selects,
//                 in pmax);
//   amax / amin : window offset a*k+b of the first max / min (fp32 mode only);
// and for each (n, unit, group) the partial sums of y and y^2 (double) over
// the rows/cols the unit covered.
struct GnWork {
    float *pmax = nullptr, *pmin = nullptr;
    int32_t *amax = nullptr, *amin = nullptr;
    double *part = nullptr;  // [N][units][groups][2]
    unsigned *arrive = nullptr;  // grid-wide arrival counter of the tf32 kernel's in-kernel finalize
    int units = 0;           // partial-sum slots per image
    int Hp = 0, Wp = 0;
};

}  // namespace conv_epi

struct conv_epi_handle_s {
    conv_epi_desc d{};
    int Ho = 0, Wo = 0;
    int device = 0;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int coop = 0;  // the device takes cooperative launches
    unsigned *dev_err = nullptr;  // device error word

    // packed tf32 weights for the tensor-core path
    float *wpack = nullptr;
    size_t wpack_bytes = 0;

    // tf32 mode, NCHW rows that are not whole 16-byte units (W not a multiple
    // of 4): x is copied here first, rows padded to a multiple of 4 floats,
    // because the tensor load needs 16-byte row strides
    float *xpad = nullptr;
    size_t xpad_bytes = 0;

    // GroupNorm workspace (allocated on demand / by conv_epi_reserve)
    void *gn_mem = nullptr;
    size_t gn_bytes = 0;
    int gn_pool_k = 0, gn_groups = 0, gn_units = 0;
    conv_epi::GnWork gn;

    // device staging for conv_epi_forward_host, and the two streams and the
    // events that pipeline its copies with the forward
    void *stage = nullptr;
    size_t stage_bytes = 0;
    static constexpr int kHostSlices = 8;
    cudaStream_t host_copy = nullptr, host_back = nullptr;
    cudaEvent_t ev_entry = nullptr, ev_done = nullptr;
    cudaEvent_t ev_in[kHostSlices] = {}, ev_out[kHostSlices] = {};

    // tf32 GroupNorm shapes the fused epilogue does not take: the conv output
    // y [N][Cout][Ho][Wo] between the two passes (by conv_epi_reserve)
    float *ybuf = nullptr;
    size_t ybuf_bytes = 0;

    // conv_epi_postpass: the GroupNorm statistics [N][groups][2] (on demand)
    float *post = nullptr;
    size_t post_bytes = 0;

    int last_launches = 0;

    // CONV_EPI_DEBUG=1 at create: every forward waits for its stream and
    // returns the device-side status itself
    int debug = 0;

    // conv_epi_test_drop_tile: the next tf32 forward skips this staged tile
    int test_drop_tile = -1;
};

namespace conv_epi {

// Argument checks shared by every entry point (api.cu), so that they refuse
// the same inputs with the same status: the problem description, and the
// chain description against it (not its pointers' alignment).
bool aligned16(const void *p);
conv_epi_status check_desc(const conv_epi_desc *d);
conv_epi_status check_epi(const conv_epi_desc &d, const conv_epi_epilogue_desc *e);
// the tile conv_epi_test_drop_tile(NULL, tile) armed for the next
// allocation-free forward on the calling thread (-1: none); reading disarms it
int take_noalloc_drop_tile();

// records a failing CUDA call for conv_epi_last_cuda_error()
conv_epi_status cuda_fail(cudaError_t e, const char *what);
#define CE_CUDA(call)                                             \
    do {                                                          \
        cudaError_t e_ = (call);                                  \
        if (e_ != cudaSuccess) return conv_epi::cuda_fail(e_, #call); \
    } while (0)

// GN workspace sizing shared by the two conv paths (units = partial-sum slots
// per image, a function of the path's tiling).
conv_epi_status ensure_gn_workspace(conv_epi_handle h, int pool_k, int groups, int units);

// fp32 CUDA-core path (simt.cu)
conv_epi_status simt_supported(const conv_epi_desc &d, const conv_epi_epilogue_desc &e);
// the fp32 mode's GroupNorm workspace, or (shapes its kernel does not take)
// the buffer of y and the statistics of the two-pass form
conv_epi_status simt_reserve(conv_epi_handle h, const conv_epi_epilogue_desc &e);
int simt_gn_units(const conv_epi_desc &d, int Ho, int pool_k);
conv_epi_status simt_forward(conv_epi_handle h, const float *x, const float *w, const float *b,
                             const conv_epi_epilogue_desc &e, float *out, cudaStream_t s);

// tcgen05 tf32 path (tc.cu)
conv_epi_status tc_supported(const conv_epi_desc &d, const conv_epi_epilogue_desc *e);
size_t tc_xpad_bytes(const conv_epi_desc &d);  // 0 unless the input rows need the padded copy
// the plan a forward would launch (pure host; conv_epi_plan_query)
conv_epi_status tc_plan_query(const conv_epi_desc &d, const conv_epi_epilogue_desc &e, conv_epi_plan &q);
size_t tc_wpack_bytes(const conv_epi_desc &d);
int tc_gn_units(const conv_epi_desc &d, int Ho, int pool_k);
// the GroupNorm chain fused into the conv kernel (else two passes through a
// buffer of the conv output); workspace for a chain ahead of a forward
bool tc_gn_fused(const conv_epi_desc &d, const conv_epi_epilogue_desc &e);
conv_epi_status tc_reserve(conv_epi_handle h, const conv_epi_epilogue_desc &e);
conv_epi_status tc_forward(conv_epi_handle h, const float *x, const float *w, const float *b,
                           const conv_epi_epilogue_desc &e, float *out, cudaStream_t s);

// The chain as a separate pass over a stored conv output (postpass.cu), and
// the buffer of its GroupNorm statistics, N * groups (mean, rstd) pairs.
conv_epi_status ensure_post_stats(conv_epi_handle h, int groups);
// The GroupNorm chain's second pass for the two-pass tensor-core form: the
// statistics folded from the conv kernel's per-unit sums (ystat, units per
// image upi, S accumulator row slots, MT channel tiles of Cg), then the
// normalise-scale-pool-clamp pass over y.
conv_epi_status postpass_gn_units(conv_epi_handle h, const float *y, const float2 *ystat, int upi, int S, int MT, int Cg,
                                  const conv_epi_epilogue_desc &e, float *out, cudaStream_t s);
conv_epi_status postpass_forward(conv_epi_handle h, const float *y, const conv_epi_epilogue_desc &e, float *out,
                                 cudaStream_t s);

// GroupNorm finalize (gn.cu): pooled max/min + statistics -> output.
// presel: the conv path left in pmax, per channel, the window extreme that the
// sign of gamma * scale selects (max when it is >= 0, else min), and no pmin;
// nslots: with presel, 1, or 2 (pmax and pmin hold that extreme of each half
// of a band, its two row pairs) or 4 (pmax, pmin and the index buffers hold
// it for each quarter, one row each), to be folded the same way.
conv_epi_status gn_finalize(conv_epi_handle h, const conv_epi_epilogue_desc &e, float *out,
                            cudaStream_t s, bool presel, int nslots = 1);

}  // namespace conv_epi
