// noalloc.cu -- conv_epi_forward_noalloc: the tf32 tensor-core forward for
// callers that cannot allocate device memory.
//
// The ordinary entry points keep their scratch (the packed tf32 filter the
// tensor-core kernel streams from, the device error word) in memory that
// conv_epi_create allocates with cudaMalloc.  Some callers cannot do that:
// code that runs inside a custom allocator or a memory-pool callback, code
// that must not change the device's memory footprint after start-up, or a
// runtime that hands this library only the input and output buffers.  This
// entry point takes the problem description directly (no handle) and keeps
// its scratch in a fixed-size array that lives in the library's own device
// image: every GPU that loads the library holds kNoAllocScratchBytes of it
// until the process exits, and no call allocates or frees anything.
//
// Limits and sharing: the packed filter of a problem must fit the array
// (Cin * 3 * (2*S+1) * Cout floats plus one chunk of padding, S = 128/Cout;
// 1 MiB covers Cin = 64 with Cout = 128, or Cin = 128 with Cout = 64), and
// only the chains whose only scratch is that filter are offered (the
// GroupNorm chain also needs its pooled workspace and is refused).  All calls
// on a device share the one array and its contents persist between calls;
// each call rewrites the whole filter region it uses before reading it, so
// nothing has to start at zero.  Two calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on the array.
#include <math.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

// the scratch itself, and the error word its kernels report into (read and
// cleared by conv_epi_noalloc_sync)
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static __device__ __align__(256) unsigned g_noalloc_err[64];

// Device addresses of the two arrays, looked up once per device.  In host
// code the names above stand for host-side shadows, never for the device
// memory itself, so only these looked-up addresses are passed to kernels.
struct DeviceSlot {
    bool ready = false;
    void *scratch = nullptr;
    unsigned *err = nullptr;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
};
std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];

conv_epi_status setup_device(int dev, DeviceSlot *&out) {
    if (dev < 0 || dev >= kMaxDevices) return CONV_EPI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSlot &sl = g_slots[dev];
    if (!sl.ready) {
        void *p = nullptr, *q = nullptr;
        CE_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
        CE_CUDA(cudaGetSymbolAddress(&q, g_noalloc_err));
        CE_CUDA(cudaDeviceGetAttribute(&sl.sm_count, cudaDevAttrMultiProcessorCount, dev));
        CE_CUDA(cudaDeviceGetAttribute(&sl.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
        CE_CUDA(cudaDeviceGetAttribute(&sl.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
        CE_CUDA(cudaMemset(q, 0, sizeof(unsigned)));
        sl.scratch = p;
        sl.err = static_cast<unsigned *>(q);
        sl.ready = true;
    }
    out = &sl;
    return CONV_EPI_OK;
}

}  // namespace

extern "C" CONV_EPI_API conv_epi_status conv_epi_forward_noalloc(const conv_epi_desc *desc, const float *x,
                                                                 const float *w, const float *b,
                                                                 const conv_epi_epilogue_desc *epi, float *out,
                                                                 void *stream) {
    // the same description and chain checks, with the same statuses, as
    // conv_epi_create and conv_epi_forward
    conv_epi_status st = conv_epi::check_desc(desc);
    if (st) return st;
    const conv_epi_desc &d = *desc;
    if ((st = conv_epi::check_epi(d, epi))) return st;
    if (d.N > 0 && (!x || !w || !b || !out)) return CONV_EPI_ERR_INVALID_ARG;  // an empty batch may pass nulls
    // what this entry point adds: tensor-core mode only, and nothing that
    // would need a workspace beyond the static array
    if (d.mode != CONV_EPI_MODE_TF32) return CONV_EPI_ERR_UNSUPPORTED;
    if (d.layout == CONV_EPI_LAYOUT_NHWC && d.Cin % 4 != 0) return CONV_EPI_ERR_UNSUPPORTED;
    // NCHW rows that are not whole 16-byte units need a padded copy of x
    if (d.layout == CONV_EPI_LAYOUT_NCHW && d.W % 4 != 0) return CONV_EPI_ERR_UNSUPPORTED;
    if (epi->kind == CONV_EPI_GN_SCALE_POOL_CLAMP) return CONV_EPI_ERR_UNSUPPORTED;  // needs the pooled workspace
    if (epi->index_out) return CONV_EPI_ERR_UNSUPPORTED;  // indices come from the fp32 mode only
    if ((st = conv_epi::tc_supported(d, epi))) return st;
    if (conv_epi::tc_wpack_bytes(d) > kNoAllocScratchBytes) return CONV_EPI_ERR_UNSUPPORTED;  // scratch too small
    if (d.N == 0) return CONV_EPI_OK;  // an empty batch: the same refusals, then nothing to compute
    if (!conv_epi::aligned16(x) || !conv_epi::aligned16(w) || !conv_epi::aligned16(b) || !conv_epi::aligned16(out))
        return CONV_EPI_ERR_ALIGNMENT;

    int dev = 0;
    CE_CUDA(cudaGetDevice(&dev));
    DeviceSlot *sl = nullptr;
    if ((st = setup_device(dev, sl))) return st;
    if (!(sl->cc_major == 10 && sl->cc_minor == 3)) return CONV_EPI_ERR_UNSUPPORTED;

    // a handle on the stack that points at the static scratch
    conv_epi_handle_s h;
    h.d = d;
    h.Ho = d.H - 2, h.Wo = d.W - 2;
    h.device = dev;
    h.sm_count = sl->sm_count;
    h.cc_major = sl->cc_major, h.cc_minor = sl->cc_minor;
    h.dev_err = sl->err;
    h.wpack = static_cast<float *>(sl->scratch);
    h.wpack_bytes = kNoAllocScratchBytes;
    h.test_drop_tile = conv_epi::take_noalloc_drop_tile();
    return conv_epi::tc_forward(&h, x, w, b, *epi, out, static_cast<cudaStream_t>(stream));
}

extern "C" CONV_EPI_API conv_epi_status conv_epi_noalloc_sync(void *stream) {
    int dev = 0;
    CE_CUDA(cudaGetDevice(&dev));
    CE_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    DeviceSlot *sl = nullptr;
    conv_epi_status st = setup_device(dev, sl);
    if (st) return st;
    unsigned word = 0;
    CE_CUDA(cudaMemcpy(&word, sl->err, sizeof word, cudaMemcpyDeviceToHost));
    if (word) {
        CE_CUDA(cudaMemset(sl->err, 0, sizeof word));
        return (word & conv_epi::ERRBIT_TIMEOUT) ? CONV_EPI_ERR_TIMEOUT : CONV_EPI_ERR_DEVICE;
    }
    return CONV_EPI_OK;
}
