// api.cu -- the C ABI of libconv_epi: argument validation, workspace
// ownership, dispatch to the tf32 tensor-core path or the fp32 CUDA-core
// path, host-buffer forward and device error reporting.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "internal.h"

namespace {

thread_local char g_cuda_err[512] = "no CUDA error recorded";

// conv_epi_test_drop_tile(NULL, k): the tile the next allocation-free
// forward on this thread skips (-1: none)
thread_local int g_noalloc_drop_tile = -1;

}  // namespace

namespace conv_epi {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int take_noalloc_drop_tile() {
    const int t = g_noalloc_drop_tile;
    g_noalloc_drop_tile = -1;
    return t;
}

conv_epi_status check_desc(const conv_epi_desc *d) {
    if (!d) return CONV_EPI_ERR_INVALID_ARG;
    if (d->N < 0 || d->Cin < 1 || d->Cout < 1 || d->H < 3 || d->W < 3) return CONV_EPI_ERR_INVALID_ARG;
    if (d->mode != CONV_EPI_MODE_TF32 && d->mode != CONV_EPI_MODE_FP32) return CONV_EPI_ERR_INVALID_ARG;
    if (d->layout != CONV_EPI_LAYOUT_NCHW && d->layout != CONV_EPI_LAYOUT_NHWC) return CONV_EPI_ERR_INVALID_ARG;
    // element counts and offsets are kept in 64-bit, but every single tensor
    // must stay below 2^31 elements
    const int64_t nx = (int64_t)d->N * d->Cin * d->H * d->W;
    const int64_t ny = (int64_t)d->N * d->Cout * (d->H - 2) * (d->W - 2);
    if (nx >= (1ll << 31) || ny >= (1ll << 31)) return CONV_EPI_ERR_UNSUPPORTED;
    return CONV_EPI_OK;
}

// Validates the chain description itself (not its pointers' alignment).
conv_epi_status check_epi(const conv_epi_desc &d, const conv_epi_epilogue_desc *e) {
    if (!e) return CONV_EPI_ERR_INVALID_ARG;
    const int Ho = d.H - 2, Wo = d.W - 2;
    switch (e->kind) {
    case CONV_EPI_MIN_TANH2:
    case CONV_EPI_SCALE_MIN:
        if (!isfinite(e->scalar)) return CONV_EPI_ERR_INVALID_ARG;
        return CONV_EPI_OK;
    case CONV_EPI_MUL_LRELU_GELU:
        if (!e->chan_scale || !isfinite(e->lrelu_slope)) return CONV_EPI_ERR_INVALID_ARG;
        if (e->index_out) return CONV_EPI_ERR_INVALID_ARG;  // this chain has no index output
        return CONV_EPI_OK;
    case CONV_EPI_NONE:
        if (e->index_out) return CONV_EPI_ERR_INVALID_ARG;  // no reduction, no index output
        return CONV_EPI_OK;
    case CONV_EPI_GN_SCALE_POOL_CLAMP:
        if (!e->chan_scale || !e->gamma || !e->beta) return CONV_EPI_ERR_INVALID_ARG;
        if (e->groups < 1 || d.Cout % e->groups != 0) return CONV_EPI_ERR_INVALID_ARG;
        if (e->pool_k < 1 || e->pool_k > Ho || e->pool_k > Wo) return CONV_EPI_ERR_INVALID_ARG;
        if (!(e->eps >= 0.0f) || !isfinite(e->eps)) return CONV_EPI_ERR_INVALID_ARG;
        if (!(e->clamp_lo <= e->clamp_hi)) return CONV_EPI_ERR_INVALID_ARG;
        return CONV_EPI_OK;
    default:
        return CONV_EPI_ERR_INVALID_ARG;
    }
}

// bytes of the fp32 kernel's packed filter (simt.cu)
size_t simt_wpack_bytes(const conv_epi_desc &d);

}  // namespace conv_epi

namespace {

using conv_epi::aligned16;
using conv_epi::check_desc;
using conv_epi::check_epi;

int pool_out(int n, int k) { return (n - k) / k + 1; }

void shape_of(const conv_epi_desc &d, const conv_epi_epilogue_desc &e, int64_t s[4]) {
    const int Ho = d.H - 2, Wo = d.W - 2;
    s[0] = d.N;
    if (e.kind == CONV_EPI_MIN_TANH2 || e.kind == CONV_EPI_SCALE_MIN) {
        s[1] = 1, s[2] = Ho, s[3] = Wo;
    } else if (e.kind == CONV_EPI_MUL_LRELU_GELU || e.kind == CONV_EPI_NONE) {
        s[1] = d.Cout, s[2] = Ho, s[3] = Wo;
    } else {
        s[1] = d.Cout, s[2] = pool_out(Ho, e.pool_k), s[3] = pool_out(Wo, e.pool_k);
    }
}

conv_epi_status check_mode_support(const conv_epi_desc &d, const conv_epi_epilogue_desc *e) {
    // channels-last input feeds the tensor core directly, so a position's
    // channels must start on 16-byte boundaries there (the fp32 mode takes
    // any Cin: it works on an NCHW copy)
    if (d.layout == CONV_EPI_LAYOUT_NHWC && d.mode == CONV_EPI_MODE_TF32 && d.Cin % 4 != 0)
        return CONV_EPI_ERR_UNSUPPORTED;
    if (d.mode == CONV_EPI_MODE_FP32)
        return e ? conv_epi::simt_supported(d, *e) : CONV_EPI_OK;
    return conv_epi::tc_supported(d, e);
}

// An empty batch (N = 0) computes nothing: its forwards validate the chain
// against the handle's problem and return without touching the device (the
// tensor pointers may then be null).
conv_epi_status empty_batch(const conv_epi_desc &d, const conv_epi_epilogue_desc *e) {
    const conv_epi_status st = check_epi(d, e);
    return st ? st : check_mode_support(d, e);
}

conv_epi_status forward_checks(conv_epi_handle h, const float *x, const float *w, const float *b,
                               const conv_epi_epilogue_desc *e, const float *out) {
    if (!h || !x || !w || !b || !out || !e) return CONV_EPI_ERR_INVALID_ARG;
    conv_epi_status st = check_epi(h->d, e);
    if (st) return st;
    if (!aligned16(x) || !aligned16(w) || !aligned16(b) || !aligned16(out)) return CONV_EPI_ERR_ALIGNMENT;
    if (e->index_out && (reinterpret_cast<uintptr_t>(e->index_out) & 3u)) return CONV_EPI_ERR_ALIGNMENT;
    if (e->index_out && h->d.mode != CONV_EPI_MODE_FP32) return CONV_EPI_ERR_UNSUPPORTED;
    return check_mode_support(h->d, e);
}

}  // namespace

namespace conv_epi {

conv_epi_status cuda_fail(cudaError_t e, const char *what) {
    snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
    (void)cudaGetLastError();  // clear a sticky-free error so later calls can proceed
    return e == cudaErrorMemoryAllocation ? CONV_EPI_ERR_NO_MEMORY : CONV_EPI_ERR_CUDA;
}

conv_epi_status ensure_gn_workspace(conv_epi_handle h, int pool_k, int groups, int units) {
    const conv_epi_desc &d = h->d;
    if (h->gn_mem && h->gn_pool_k == pool_k && h->gn_groups == groups && h->gn_units == units)
        return CONV_EPI_OK;
    const int Hp = pool_out(h->Ho, pool_k), Wp = pool_out(h->Wo, pool_k);
    const size_t npool = (size_t)d.N * d.Cout * Hp * Wp;
    const size_t npart = (size_t)d.N * units * groups * 2;
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t bytes = 2 * up(npool * sizeof(float)) + 2 * up(npool * sizeof(int32_t)) + up(npart * sizeof(double)) +
                         256;  // + the arrival counter
    if (h->gn_mem && bytes <= h->gn_bytes) {
        // reuse the larger buffer
    } else {
        if (h->gn_mem) {
            CE_CUDA(cudaDeviceSynchronize());
            CE_CUDA(cudaFree(h->gn_mem));
            h->gn_mem = nullptr, h->gn_bytes = 0;
        }
        CE_CUDA(cudaMalloc(&h->gn_mem, bytes));
        h->gn_bytes = bytes;
    }
    char *p = static_cast<char *>(h->gn_mem);
    h->gn.pmax = reinterpret_cast<float *>(p), p += up(npool * sizeof(float));
    h->gn.pmin = reinterpret_cast<float *>(p), p += up(npool * sizeof(float));
    h->gn.amax = reinterpret_cast<int32_t *>(p), p += up(npool * sizeof(int32_t));
    h->gn.amin = reinterpret_cast<int32_t *>(p), p += up(npool * sizeof(int32_t));
    h->gn.part = reinterpret_cast<double *>(p), p += up(npart * sizeof(double));
    h->gn.arrive = reinterpret_cast<unsigned *>(p);
    h->gn.units = units, h->gn.Hp = Hp, h->gn.Wp = Wp;
    h->gn_pool_k = pool_k, h->gn_groups = groups, h->gn_units = units;
    return CONV_EPI_OK;
}

}  // namespace conv_epi

extern "C" {

CONV_EPI_API const char *conv_epi_status_string(conv_epi_status s) {
    switch (s) {
    case CONV_EPI_OK: return "ok";
    case CONV_EPI_ERR_INVALID_ARG: return "invalid argument";
    case CONV_EPI_ERR_UNSUPPORTED: return "unsupported shape, chain or device for this mode";
    case CONV_EPI_ERR_ALIGNMENT: return "tensor not aligned to 16 bytes";
    case CONV_EPI_ERR_CUDA: return "CUDA runtime error";
    case CONV_EPI_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case CONV_EPI_ERR_NO_MEMORY: return "out of device memory";
    case CONV_EPI_ERR_DEVICE: return "kernel raised an error flag";
    }
    return "unknown status";
}

CONV_EPI_API const char *conv_epi_last_cuda_error(void) { return g_cuda_err; }

CONV_EPI_API int conv_epi_version(void) { return 10200; }

CONV_EPI_API conv_epi_status conv_epi_output_shape(const conv_epi_desc *desc, const conv_epi_epilogue_desc *epi,
                                                   int64_t shape[4]) {
    if (!shape) return CONV_EPI_ERR_INVALID_ARG;
    conv_epi_status st = check_desc(desc);
    if (st) return st;
    if ((st = check_epi(*desc, epi))) return st;
    shape_of(*desc, *epi, shape);
    return CONV_EPI_OK;
}

CONV_EPI_API conv_epi_status conv_epi_create(const conv_epi_desc *desc, conv_epi_handle *out) {
    if (!out) return CONV_EPI_ERR_INVALID_ARG;
    *out = nullptr;
    conv_epi_status st = check_desc(desc);
    if (st) return st;
    if ((st = check_mode_support(*desc, nullptr))) return st;
    int dev = 0;
    CE_CUDA(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CE_CUDA(cudaGetDeviceProperties(&prop, dev));
    // every kernel of this library is built for sm_103a only
    if (!(prop.major == 10 && prop.minor == 3)) return CONV_EPI_ERR_UNSUPPORTED;
    conv_epi_handle h = new (std::nothrow) conv_epi_handle_s();
    if (!h) return CONV_EPI_ERR_NO_MEMORY;
    h->d = *desc;
    h->Ho = desc->H - 2, h->Wo = desc->W - 2;
    h->device = dev;
    h->sm_count = prop.multiProcessorCount;
    h->cc_major = prop.major, h->cc_minor = prop.minor;
    h->coop = prop.cooperativeLaunch;
    const char *dbg = getenv("CONV_EPI_DEBUG");
    h->debug = dbg && dbg[0] == '1' && dbg[1] == '\0';
    cudaError_t e = cudaMalloc(&h->dev_err, 256);
    if (e == cudaSuccess) e = cudaMemset(h->dev_err, 0, 256);
    // the packed filter: tf32 operands for the tensor-core kernel, or the fp32
    // kernel's staging order
    if (e == cudaSuccess) {
        h->wpack_bytes = desc->mode == CONV_EPI_MODE_TF32 ? conv_epi::tc_wpack_bytes(*desc)
                                                          : conv_epi::simt_wpack_bytes(*desc);
        e = cudaMalloc(&h->wpack, h->wpack_bytes);
    }
    // tf32 NCHW rows not a multiple of 4 floats: room for the padded copy of
    // x; fp32 channels-last input: room for its NCHW copy
    h->xpad_bytes = desc->mode == CONV_EPI_MODE_TF32 ? conv_epi::tc_xpad_bytes(*desc)
                    : desc->layout == CONV_EPI_LAYOUT_NHWC
                        ? (size_t)desc->N * desc->Cin * desc->H * desc->W * sizeof(float)
                        : 0;
    if (e == cudaSuccess && h->xpad_bytes != 0) e = cudaMalloc(&h->xpad, h->xpad_bytes);
    if (e != cudaSuccess) {
        st = conv_epi::cuda_fail(e, "conv_epi_create workspace");
        cudaFree(h->dev_err);
        cudaFree(h->wpack);
        cudaFree(h->xpad);
        delete h;
        return st;
    }
    *out = h;
    return CONV_EPI_OK;
}

CONV_EPI_API conv_epi_status conv_epi_reserve(conv_epi_handle h, const conv_epi_epilogue_desc *epi) {
    if (!h) return CONV_EPI_ERR_INVALID_ARG;
    conv_epi_status st = check_epi(h->d, epi);
    if (st) return st;
    if ((st = check_mode_support(h->d, epi))) return st;
    if (epi->kind != CONV_EPI_GN_SCALE_POOL_CLAMP) return CONV_EPI_OK;
    CE_CUDA(cudaSetDevice(h->device));
    if (h->d.mode == CONV_EPI_MODE_TF32) return conv_epi::tc_reserve(h, *epi);
    return conv_epi::simt_reserve(h, *epi);
}

CONV_EPI_API conv_epi_status conv_epi_forward(conv_epi_handle h, const float *x, const float *w, const float *b,
                                              const conv_epi_epilogue_desc *epi, float *out, void *stream) {
    if (h && h->d.N == 0) {
        h->last_launches = 0;
        return empty_batch(h->d, epi);
    }
    conv_epi_status st = forward_checks(h, x, w, b, epi, out);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    h->last_launches = 0;
    if (epi->kind == CONV_EPI_GN_SCALE_POOL_CLAMP) {
        if ((st = conv_epi_reserve(h, epi))) return st;
    }
    st = h->d.mode == CONV_EPI_MODE_FP32 ? conv_epi::simt_forward(h, x, w, b, *epi, out, s)
                                         : conv_epi::tc_forward(h, x, w, b, *epi, out, s);
    // debug handles report device-side errors (a barrier timeout) here
    if (st == CONV_EPI_OK && h->debug) st = conv_epi_sync(h, stream);
    return st;
}

CONV_EPI_API conv_epi_status conv_epi_forward_host(conv_epi_handle h, const float *x, const float *w,
                                                   const float *b, const conv_epi_epilogue_desc *epi, float *out,
                                                   void *stream) {
    if (h && h->d.N == 0) {
        h->last_launches = 0;
        return empty_batch(h->d, epi);
    }
    if (!h || !x || !w || !b || !epi || !out) return CONV_EPI_ERR_INVALID_ARG;
    conv_epi_status st = check_epi(h->d, epi);
    if (st) return st;
    const conv_epi_desc &d = h->d;
    int64_t shp[4];
    shape_of(d, *epi, shp);
    const size_t nx = (size_t)d.N * d.Cin * d.H * d.W, nw = (size_t)d.Cout * d.Cin * 9, nc = (size_t)d.Cout;
    const size_t no = (size_t)(shp[0] * shp[1] * shp[2] * shp[3]);
    auto up = [](size_t v) { return (v + 63) & ~(size_t)63; };  // 256-byte steps of floats
    const size_t need = sizeof(float) * (up(nx) + up(nw) + 4 * up(nc) + up(no)) + sizeof(int32_t) * up(no);
    CE_CUDA(cudaSetDevice(h->device));
    if (need > h->stage_bytes) {
        if (h->stage) {
            CE_CUDA(cudaDeviceSynchronize());
            CE_CUDA(cudaFree(h->stage));
            h->stage = nullptr, h->stage_bytes = 0;
        }
        CE_CUDA(cudaMalloc(&h->stage, need));
        h->stage_bytes = need;
    }
    float *dx = static_cast<float *>(h->stage);
    float *dw = dx + up(nx), *db = dw + up(nw), *dp0 = db + up(nc), *dp1 = dp0 + up(nc), *dp2 = dp1 + up(nc);
    float *dout = dp2 + up(nc);
    int32_t *didx = reinterpret_cast<int32_t *>(dout + up(no));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the filter, bias and chain parameters first, on the caller's stream
    CE_CUDA(cudaMemcpyAsync(dw, w, nw * sizeof(float), cudaMemcpyHostToDevice, s));
    CE_CUDA(cudaMemcpyAsync(db, b, nc * sizeof(float), cudaMemcpyHostToDevice, s));
    conv_epi_epilogue_desc de = *epi;
    if (epi->chan_scale) {
        CE_CUDA(cudaMemcpyAsync(dp0, epi->chan_scale, nc * sizeof(float), cudaMemcpyHostToDevice, s));
        de.chan_scale = dp0;
    }
    if (epi->gamma) {
        CE_CUDA(cudaMemcpyAsync(dp1, epi->gamma, nc * sizeof(float), cudaMemcpyHostToDevice, s));
        de.gamma = dp1;
    }
    if (epi->beta) {
        CE_CUDA(cudaMemcpyAsync(dp2, epi->beta, nc * sizeof(float), cudaMemcpyHostToDevice, s));
        de.beta = dp2;
    }
    // The batch in slices of whole images (every step of every chain is
    // independent per image): slice k's input copy, on a copy stream, runs
    // while slice k-1 is computed on the caller's stream and slice k-2's
    // result copies back on a third stream, so the transfer, which takes the
    // longest, hides the compute.
    if (!h->host_copy) {
        CE_CUDA(cudaStreamCreateWithFlags(&h->host_copy, cudaStreamNonBlocking));
        CE_CUDA(cudaStreamCreateWithFlags(&h->host_back, cudaStreamNonBlocking));
        CE_CUDA(cudaEventCreateWithFlags(&h->ev_entry, cudaEventDisableTiming));
        CE_CUDA(cudaEventCreateWithFlags(&h->ev_done, cudaEventDisableTiming));
        for (int k = 0; k < conv_epi_handle_s::kHostSlices; ++k) {
            CE_CUDA(cudaEventCreateWithFlags(&h->ev_in[k], cudaEventDisableTiming));
            CE_CUDA(cudaEventCreateWithFlags(&h->ev_out[k], cudaEventDisableTiming));
        }
    }
    const size_t xi = nx / d.N, oi = no / d.N;  // elements per image
    // slices start on 16-byte boundaries only when an image is a whole number
    // of float4s in and out; otherwise the batch goes as one slice
    int K = d.N < conv_epi_handle_s::kHostSlices ? d.N : conv_epi_handle_s::kHostSlices;
    if (xi % 4 != 0 || oi % 4 != 0) K = 1;
    // the GroupNorm workspace belongs to the handle: allocate it here, not in
    // a slice's copy of the handle
    if (epi->kind == CONV_EPI_GN_SCALE_POOL_CLAMP && (st = conv_epi_reserve(h, epi))) return st;
    CE_CUDA(cudaEventRecord(h->ev_entry, s));   // work already on the caller's stream comes first
    CE_CUDA(cudaStreamWaitEvent(h->host_copy, h->ev_entry, 0));
    CE_CUDA(cudaStreamWaitEvent(h->host_back, h->ev_entry, 0));
    for (int k = 0; k < K; ++k) {
        const size_t n0 = (size_t)d.N * k / K, n1 = (size_t)d.N * (k + 1) / K;
        CE_CUDA(cudaMemcpyAsync(dx + n0 * xi, x + n0 * xi, (n1 - n0) * xi * sizeof(float), cudaMemcpyHostToDevice,
                                h->host_copy));
        CE_CUDA(cudaEventRecord(h->ev_in[k], h->host_copy));
    }
    const int drop = h->test_drop_tile;
    int launches = 0;
    for (int k = 0; k < K; ++k) {
        const size_t n0 = (size_t)d.N * k / K, n1 = (size_t)d.N * (k + 1) / K;
        conv_epi_handle_s sub = *h;  // the same workspace, for images n0 .. n1-1
        sub.d.N = (int)(n1 - n0);
        sub.test_drop_tile = k == 0 ? drop : -1;
        conv_epi_epilogue_desc dk = de;
        if (epi->index_out) dk.index_out = didx + n0 * oi;
        CE_CUDA(cudaStreamWaitEvent(s, h->ev_in[k], 0));
        st = conv_epi_forward(&sub, dx + n0 * xi, dw, db, &dk, dout + n0 * oi, stream);
        if (st) return st;
        launches += sub.last_launches;
        CE_CUDA(cudaEventRecord(h->ev_out[k], s));
        CE_CUDA(cudaStreamWaitEvent(h->host_back, h->ev_out[k], 0));
        CE_CUDA(cudaMemcpyAsync(out + n0 * oi, dout + n0 * oi, (n1 - n0) * oi * sizeof(float), cudaMemcpyDeviceToHost,
                                h->host_back));
        if (epi->index_out)
            CE_CUDA(cudaMemcpyAsync(epi->index_out + n0 * oi, didx + n0 * oi, (n1 - n0) * oi * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, h->host_back));
    }
    h->test_drop_tile = -1;
    h->last_launches = launches;
    CE_CUDA(cudaEventRecord(h->ev_done, h->host_back));
    CE_CUDA(cudaStreamWaitEvent(s, h->ev_done, 0));
    return conv_epi_sync(h, stream);
}

CONV_EPI_API conv_epi_status conv_epi_postpass(conv_epi_handle h, const float *y, const conv_epi_epilogue_desc *epi,
                                               float *out, void *stream) {
    if (!h) return CONV_EPI_ERR_INVALID_ARG;
    conv_epi_status st = check_epi(h->d, epi);
    if (st) return st;
    if (epi->index_out) return CONV_EPI_ERR_UNSUPPORTED;  // no index output on this pass
    if (h->d.N == 0) {
        h->last_launches = 0;
        return CONV_EPI_OK;
    }
    if (!y || !out) return CONV_EPI_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out)) return CONV_EPI_ERR_ALIGNMENT;
    CE_CUDA(cudaSetDevice(h->device));
    return conv_epi::postpass_forward(h, y, *epi, out, static_cast<cudaStream_t>(stream));
}

CONV_EPI_API conv_epi_status conv_epi_sync(conv_epi_handle h, void *stream) {
    if (!h) return CONV_EPI_ERR_INVALID_ARG;
    CE_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    unsigned word = 0;
    CE_CUDA(cudaMemcpy(&word, h->dev_err, sizeof word, cudaMemcpyDeviceToHost));
    if (word) {
        CE_CUDA(cudaMemset(h->dev_err, 0, sizeof word));
        return (word & conv_epi::ERRBIT_TIMEOUT) ? CONV_EPI_ERR_TIMEOUT : CONV_EPI_ERR_DEVICE;
    }
    return CONV_EPI_OK;
}

CONV_EPI_API conv_epi_status conv_epi_plan_query(const conv_epi_desc *desc, const conv_epi_epilogue_desc *epi,
                                                 conv_epi_plan *plan) {
    if (!plan) return CONV_EPI_ERR_INVALID_ARG;
    *plan = conv_epi_plan{};
    plan->struct_bytes = (int64_t)sizeof(conv_epi_plan);
    conv_epi_status st = check_desc(desc);
    if (st) return st;
    if ((st = check_epi(*desc, epi))) return st;
    if (desc->mode != CONV_EPI_MODE_TF32) return CONV_EPI_ERR_UNSUPPORTED;
    if (desc->layout == CONV_EPI_LAYOUT_NHWC && desc->Cin % 4 != 0) return CONV_EPI_ERR_UNSUPPORTED;
    return conv_epi::tc_plan_query(*desc, *epi, *plan);
}

CONV_EPI_API conv_epi_status conv_epi_test_drop_tile(conv_epi_handle h, int tile) {
    if (tile < -1) return CONV_EPI_ERR_INVALID_ARG;
    if (!h) {  // the next allocation-free forward on this thread
        g_noalloc_drop_tile = tile;
        return CONV_EPI_OK;
    }
    if (h->d.mode != CONV_EPI_MODE_TF32) return CONV_EPI_ERR_UNSUPPORTED;
    h->test_drop_tile = tile;
    return CONV_EPI_OK;
}

CONV_EPI_API conv_epi_status conv_epi_destroy(conv_epi_handle h) {
    if (!h) return CONV_EPI_ERR_INVALID_ARG;
    cudaSetDevice(h->device);
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(h->dev_err);
    cudaFree(h->wpack);
    cudaFree(h->xpad);
    cudaFree(h->gn_mem);
    cudaFree(h->stage);
    cudaFree(h->post);
    cudaFree(h->ybuf);
    if (h->host_copy) {
        cudaStreamDestroy(h->host_copy);
        cudaStreamDestroy(h->host_back);
        cudaEventDestroy(h->ev_entry);
        cudaEventDestroy(h->ev_done);
        for (int k = 0; k < conv_epi_handle_s::kHostSlices; ++k) {
            cudaEventDestroy(h->ev_in[k]);
            cudaEventDestroy(h->ev_out[k]);
        }
    }
    delete h;
    return e == cudaSuccess ? CONV_EPI_OK : conv_epi::cuda_fail(e, "conv_epi_destroy");
}

CONV_EPI_API size_t conv_epi_workspace_bytes(conv_epi_handle h) {
    if (!h) return 0;
    return 256 + h->wpack_bytes + h->xpad_bytes + h->gn_bytes + h->stage_bytes + h->post_bytes + h->ybuf_bytes;
}

CONV_EPI_API int conv_epi_last_launch_count(conv_epi_handle h) { return h ? h->last_launches : 0; }

}  // extern "C"
