// tc.cu -- tf32 tensor-core path (CONV_EPI_MODE_TF32): the 3x3 convolution
// as an implicit GEMM on the 5th-generation tensor cores (tcgen05), with the
// post-conv chain fused into the epilogue that drains tensor memory.
//
// GEMM view.  For one image n, flatten an input plane row-major with a row
// pitch P >= W (P a multiple of 16): position q = h*P + w.  Output (i, j) sits
// at q_out = i*P + j and tap (kh, kw) reads q_out + kh*P + kw, so
//     D[co, q_out] = sum_{ci, kh, kw} W[co, ci, kh, kw] * X[ci, q_out + kh*P + kw]
// is a GEMM with M = Cout, N = positions, K = Cin*9 in which every tap is the
// same operand shifted by kh*P + kw positions.  (The pages' im2col view,
// POPCORNBENCH Kimi-K2.6 level-2 problems 85 and 54, "conv = GEMM with
// K = C_in*9"; on those pages the GEMM itself is left to cuDNN.)
//
// Operands in shared memory, both "K-major, no swizzle" with a 16-byte row:
//   B (positions x 8 channels): plane[ci4][q][4 floats] -- position rows are
//      16 bytes apart, so a tap shift of kh*P + kw positions is a plain
//      (16-byte aligned) change of the descriptor's start address.  NCHW has
//      positions contiguous per channel, so converter warps transpose the
//      input tile on the way in (global -> registers -> shared), rounding to
//      tf32 (round-to-nearest) as they go.
//   A (128 rows x 8 channels): packed filter planes, loaded by the bulk-copy
//      engine (cp.async.bulk) from a buffer the prep kernel writes each call.
// Accumulators live in tensor memory (128 lanes x 512 columns, fp32).
//
// Row slots.  The MMA's M is 128.  With Cout = 128 a tile is one output row
// per accumulator.  With Cout = 64 the 128 accumulator lanes hold TWO output
// rows (lanes 0-63: row r, lanes 64-127: row r+1): the A tile for the
// position shift "sk" stacks W(kh = sk) over W(kh = sk-1), so one MMA feeds
// both rows from the same input window.  Shifts sk = 0..3 cover kh = 0..2 of
// both rows; the two missing (kh = -1, kh = 3) blocks are zero, so 12 MMAs do
// the work of 9 full-height ones -- still 1.5x the rate of the M = 64 shape.
//
// One CTA per SM (persistent), 16 warps:
//   warp 0      tensor-memory allocator + single-thread MMA issuer
//   warp 1      filter producer (bulk copies into the stage ring)
//   warps 2-7   converters (input tile -> B plane)
//   warps 8-15  epilogue (tensor memory -> chain -> global), two warps per
//               32-lane quadrant, alternating 16-column chunks
// Stages: a ring of (A, B) buffers with full/empty mbarriers; two
// accumulator buffers in tensor memory so the epilogue of one unit overlaps
// the main loop of the next.  Every wait is bounded (2 s of %globaltimer);
// on expiry the kernel raises an error bit, drains what it has in flight and
// returns, so the context stays usable.
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace conv_epi {
namespace {

constexpr int kThreads = 512;
// Warp roles per chain: the min chains need 4 epilogue warps, the per-channel
// and GroupNorm chains 8; the converters take the warps in between.
template <int KIND>
struct Roles {
    static constexpr bool kMinKind = KIND == CONV_EPI_MIN_TANH2 || KIND == CONV_EPI_SCALE_MIN;
    static constexpr int kEpiWarps = kMinKind ? 4 : 8;
    static constexpr int kEpiWarp0 = 16 - kEpiWarps;  // a multiple of 4 (tensor-memory quadrants)
    static constexpr int kConvWarp0 = 2;
    static constexpr int kConvWarps = kEpiWarp0 - kConvWarp0;
    static constexpr int kConvThreads = kConvWarps * 32;
    static constexpr int kEpiThreads = kEpiWarps * 32;
    static constexpr int kColGroups = kEpiWarps / 4;  // epilogue warps per quadrant
    static constexpr int kNBMax = kMinKind ? 2 : 3;   // 4x4 blocks per converter thread per chunk
};
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;     // columns per accumulator buffer
constexpr int kMaxStages = 6;
constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA
constexpr int kStgPitch = 17;       // epilogue transpose staging pitch (floats)

struct TcArgs {
    const float *x, *b, *wpack;
    float *out;
    unsigned *err;
    int N, Cin, H, W, Cout, Ho, Wo;
    int S, P, U, RU, PL;
    int ucol;          // tensor-memory columns between the unit's accumulators (multiple of 32)
    uint32_t p_magic;  // ceil(2^32 / P), exact division for q < 2^16
    int chunks, units_per_img, total_units, stages;
    uint32_t a_bytes, b_bytes, stage_bytes, scratch_off;
    int resident;          // 1: every filter chunk stays in shared memory for the whole kernel
    uint32_t stage0_off;   // byte offset of stage 0 (after the resident filter, if any)
    uint32_t b_off;        // byte offset of B inside a stage (0 when the filter is resident)
    uint32_t a_kw_stride, a_lbo, a_plane_bytes;
    uint32_t idesc;
    float scalar;
    const float *chan_scale;
    float slope;
    int groups, pool_k, Hp, Wp;
    GnWork gn;
};

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ uint32_t f32_to_tf32(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
template <int NT>
__device__ __forceinline__ void epi_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
// barrier over the epilogue warps that also ORs a flag across them, so they
// all take the same branch after it
template <int NT>
__device__ __forceinline__ bool epi_bar_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(NT)
        : "memory");
    return r != 0;
}

// tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, M=128, kind::tf32, fp32 accumulate
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every MMA this thread issued before has completed
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns; wait folded in so that no use of
// the registers can be scheduled before the load has landed
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, K-major, no swizzle (canonical layout
// ((8,m),(4,2)) : ((16B, SBO), (4B, LBO)) for 32-bit elements):
//   bits  0-13 start address >> 4     bits 16-29 LBO >> 4 (K-direction core-matrix stride)
//   bits 32-45 SBO >> 4 (8-row group stride)   bits 46-47 = 1 (descriptor version)
//   bits 49-51 base offset = 0, bit 52 LBO mode = 0, bits 61-63 swizzle = 0 (none)
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46);
}

// bounded wait: true when the phase completed, false on timeout or (when
// honor_abort) once another role has given up
__device__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err,
                         bool honor_abort = true) {
    for (int i = 0; i < 64; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honor_abort && *abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(err, ERRBIT_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// --------------------------------------------------------------- roles ----
struct Bars {
    uint32_t base;
    int stages;
    __device__ uint32_t full_w(int s) const { return base + 8u * s; }
    __device__ uint32_t full_x(int s) const { return base + 8u * (stages + s); }
    __device__ uint32_t empty(int s) const { return base + 8u * (2 * stages + s); }
    __device__ uint32_t acc_full(int ab) const { return base + 8u * (3 * stages + ab); }
    __device__ uint32_t acc_empty(int ab) const { return base + 8u * (3 * stages + 2 + ab); }
    __device__ uint32_t final_bar() const { return base + 8u * (3 * stages + 4); }
    __device__ uint32_t wres() const { return base + 8u * (3 * stages + 5); }
    static constexpr int count(int stages) { return 3 * stages + 6; }
};

__device__ void mma_role(const TcArgs &a, uint32_t sbase, const Bars &bars, uint32_t tmem, volatile int *abort_flag) {
    int it = 0, j = 0;
    bool ok = true;
    if (a.resident) ok = wait_bar(bars.wres(), 0, abort_flag, a.err);
    for (int unit = blockIdx.x; ok && unit < a.total_units; unit += gridDim.x, ++j) {
        const int ab = j & 1;
        if (!wait_bar(bars.acc_empty(ab), ((j >> 1) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t dcol = tmem + ab * kAccStride;
        for (int c = 0; c < a.chunks; ++c, ++it) {
            const int s = it % a.stages;
            const uint32_t ph = (it / a.stages) & 1;
            if ((!a.resident && !wait_bar(bars.full_w(s), ph, abort_flag, a.err)) ||
                !wait_bar(bars.full_x(s), ph, abort_flag, a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t S0 = sbase + a.stage0_off + s * a.stage_bytes;
            const uint32_t A0 = a.resident ? sbase + c * a.a_bytes : S0;
            const uint32_t B0 = S0 + a.b_off;
            for (int u = 0; u < a.U; ++u) {
                for (int sk = 0; sk <= a.S + 1; ++sk) {
#pragma unroll
                    for (int kw = 0; kw < 3; ++kw) {
                        const uint64_t ad = smem_desc(A0 + kw * a.a_kw_stride + (a.S + 1 - sk) * a.a_plane_bytes,
                                                      a.a_lbo, 128);
                        const uint64_t bd = smem_desc(B0 + 16u * ((u * a.S + sk) * a.P + kw), 16u * a.PL, 128);
                        mma_tf32(dcol + u * a.ucol, ad, bd, a.idesc, (c | sk | kw) != 0);
                    }
                }
            }
            mma_commit(bars.empty(s));  // stage s may be refilled once these MMAs are done
        }
        if (!ok) break;
        mma_commit(bars.acc_full(ab));  // accumulator ab is complete
    }
    // drain: every MMA issued above completes before the CTA releases tensor memory
    mma_commit(bars.final_bar());
    wait_bar(bars.final_bar(), 0, abort_flag, a.err, false);
}

__device__ void weight_role(const TcArgs &a, uint32_t sbase, const Bars &bars, volatile int *abort_flag) {
    const char *wsrc = reinterpret_cast<const char *>(a.wpack);
    if (a.resident) {
        // the whole packed filter, once
        const uint32_t total = a.chunks * a.a_bytes;
        mbar_arrive_expect_tx(bars.wres(), total);
        for (uint32_t off = 0; off < total; off += 16384u)
            bulk_g2s(sbase + off, wsrc + off, min(16384u, total - off), bars.wres());
        wait_bar(bars.wres(), 0, abort_flag, a.err, false);
        return;
    }
    int it = 0;
    int last_par[kMaxStages];
    bool issued[kMaxStages];
    for (int s = 0; s < kMaxStages; ++s) issued[s] = false, last_par[s] = 0;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < a.total_units; unit += gridDim.x) {
        for (int c = 0; c < a.chunks; ++c, ++it) {
            const int s = it % a.stages;
            const uint32_t ph = (it / a.stages) & 1;
            if (!wait_bar(bars.empty(s), ph ^ 1, abort_flag, a.err)) {
                ok = false;
                break;
            }
            const uint32_t dst = sbase + a.stage0_off + s * a.stage_bytes;
            const char *src = wsrc + (size_t)c * a.a_bytes;
            mbar_arrive_expect_tx(bars.full_w(s), a.a_bytes);
            for (uint32_t off = 0; off < a.a_bytes; off += 16384u) {
                const uint32_t n = min(16384u, a.a_bytes - off);
                bulk_g2s(dst + off, src + off, n, bars.full_w(s));
            }
            issued[s] = true, last_par[s] = ph;
        }
    }
    // copies still in flight land before the CTA exits
    for (int s = 0; s < a.stages; ++s)
        if (issued[s]) wait_bar(bars.full_w(s), last_par[s], abort_flag, a.err, false);
}

// Converter warps: x[n][8c .. 8c+7][r0 .. r0+Rin-1][0 .. W-1] -> B plane
// [ci4][q][4] of a stage.  Work item = one 4x4 block: 4 consecutive positions
// (one 16-byte global load per channel) x 4 channels; a register transpose
// turns it into 4 position rows of 16 bytes, rounded to tf32.  The rows are
// stored in a per-thread rotated order so that the 8 threads of a store phase
// hit 8 different bank groups.  Positions outside the image are zero.
// Registers hold two chunks: the loads of chunk it+1 are in flight while the
// thread waits for its stage and stores chunk it.
template <int NB>
struct ConvRegs {
    float4 v[NB][4];
    int row[NB];  // first B-plane row of the block (jg*PL + q), -1 when absent
};

__device__ __forceinline__ float pick(const float4 &v, int p) {
    return p == 0 ? v.x : (p == 1 ? v.y : (p == 2 ? v.z : v.w));
}

template <int NT, int NB>
__device__ __forceinline__ void conv_issue(const TcArgs &a, ConvRegs<NB> &r, int t, int flat) {
    const int unit = blockIdx.x + (flat / a.chunks) * gridDim.x;
    const int c = flat % a.chunks;
    const int n = unit / a.units_per_img;
    const int r0 = (unit % a.units_per_img) * a.RU;
    const size_t HW = (size_t)a.H * a.W;
    const int qpp = a.PL >> 2;  // 4-position groups per ci4 plane
#pragma unroll
    for (int k = 0; k < NB; ++k) {
        const int b = t + k * NT;
        r.row[k] = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) r.v[k][e] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < 2 * qpp) {
            const int jg = b >= qpp ? 1 : 0;
            const int q = 4 * (b - jg * qpp);
            const int rr = __umulhi((uint32_t)q, a.p_magic);
            const int w = q - rr * a.P;
            const int h = r0 + rr;
            r.row[k] = jg * a.PL + q;
            if (h < a.H && w < a.W) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    a.x + (((size_t)n * a.Cin + 8 * c + 4 * jg) * HW + (size_t)h * a.W + w));
#pragma unroll
                for (int e = 0; e < 4; ++e) r.v[k][e] = __ldg(src + e * (HW >> 2));
            }
        }
    }
}

template <int NB>
__device__ __forceinline__ void conv_store(const TcArgs &a, const ConvRegs<NB> &r, uint8_t *plane) {
#pragma unroll
    for (int k = 0; k < NB; ++k) {
        if (r.row[k] < 0) continue;
        const int rot = (r.row[k] >> 3) & 3;  // (position group / 2) mod 4
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = (i + rot) & 3;
            uint4 o;
            o.x = f32_to_tf32(pick(r.v[k][0], p));
            o.y = f32_to_tf32(pick(r.v[k][1], p));
            o.z = f32_to_tf32(pick(r.v[k][2], p));
            o.w = f32_to_tf32(pick(r.v[k][3], p));
            reinterpret_cast<uint4 *>(plane)[r.row[k] + p] = o;
        }
    }
}

template <int NT, int NB>
__device__ void converter_role(const TcArgs &a, uint8_t *smem, const Bars &bars, volatile int *abort_flag,
                               int t) {
    const int my_units = a.total_units > (int)blockIdx.x ? (a.total_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_units * a.chunks;
    ConvRegs<NB> ra, rb;
    auto finish = [&](const ConvRegs<NB> &r, int it) -> bool {
        const int s = it % a.stages;
        const uint32_t ph = (it / a.stages) & 1;
        if (!wait_bar(bars.empty(s), ph ^ 1, abort_flag, a.err)) return false;
        conv_store<NB>(a, r, smem + a.stage0_off + s * a.stage_bytes + a.b_off);
        fence_proxy_async_smem();  // make the generic-proxy stores visible to the tensor core
        mbar_arrive(bars.full_x(s));
        return true;
    };
    if (total > 0) conv_issue<NT, NB>(a, ra, t, 0);
    for (int it = 0; it < total; it += 2) {
        if (it + 1 < total) conv_issue<NT, NB>(a, rb, t, it + 1);
        if (!finish(ra, it)) return;
        if (it + 1 >= total) break;
        if (it + 2 < total) conv_issue<NT, NB>(a, ra, t, it + 2);
        if (!finish(rb, it + 1)) return;
    }
}

// min (or max, sgn < 0) of 16 columns over the warp's 32 lanes, reduce-scatter:
// on return lanes 2c and 2c+1 hold column c's result in v[0]
__device__ __forceinline__ float rs_op(float x, float y, int sgn) { return sgn >= 0 ? fminf(x, y) : fmaxf(x, y); }
__device__ __forceinline__ void reduce_scatter16(float (&v)[16], int lane, int sgn) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float send = b4 ? v[i] : v[i + 8], keep = b4 ? v[i + 8] : v[i];
        v[i] = rs_op(keep, __shfl_xor_sync(0xffffffffu, send, 16), sgn);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b3 ? v[i] : v[i + 4], keep = b3 ? v[i + 4] : v[i];
        v[i] = rs_op(keep, __shfl_xor_sync(0xffffffffu, send, 8), sgn);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b2 ? v[i] : v[i + 2], keep = b2 ? v[i + 2] : v[i];
        v[i] = rs_op(keep, __shfl_xor_sync(0xffffffffu, send, 4), sgn);
    }
    {
        const float send = b1 ? v[0] : v[1], keep = b1 ? v[1] : v[0];
        v[0] = rs_op(keep, __shfl_xor_sync(0xffffffffu, send, 2), sgn);
    }
    v[0] = rs_op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1), sgn);
}

__device__ __forceinline__ float gelu_erf(float t) { return 0.5f * t * (1.0f + erff(t * 0.70710678118654752f)); }

template <int KIND>
__device__ void epilogue_role(const TcArgs &a, float *scratch, const Bars &bars, uint32_t tmem,
                              volatile int *abort_flag) {
    using R = Roles<KIND>;
    constexpr int NH = R::kColGroups;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ew = warp - R::kEpiWarp0;
    const int et = threadIdx.x - R::kEpiWarp0 * 32;
    const int qd = warp & 3;          // tensor-memory lane quadrant
    const int hc = ew >> 2;           // which 16-column chunks: cc = hc, hc + NH, ...
    const int L = qd * 32 + lane;     // accumulator row
    const int slot = L / a.Cout, co = L % a.Cout;
    const float bias = __ldg(&a.b[co]);
    const int sgn = a.scalar > 0.0f ? 1 : (a.scalar < 0.0f ? -1 : 0);
    constexpr bool kMin = KIND == CONV_EPI_MIN_TANH2 || KIND == CONV_EPI_SCALE_MIN;
    constexpr bool kGN = KIND == CONV_EPI_GN_SCALE_POOL_CLAMP;
    float mult = 0.0f;
    if (KIND == CONV_EPI_MUL_LRELU_GELU) mult = __ldg(&a.chan_scale[co]);
    const int nchunks = a.P / 16;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    int j = 0;
    for (int unit = blockIdx.x; unit < a.total_units; unit += gridDim.x, ++j) {
        const int n = unit / a.units_per_img;
        const int ru = unit % a.units_per_img;
        const int r0 = ru * a.RU;
        const int ab = j & 1;
        const bool ok = wait_bar(bars.acc_full(ab), (j >> 1) & 1, abort_flag, a.err);
        if (epi_bar_any<R::kEpiThreads>(!ok)) break;  // all epilogue warps leave together
        tc_fence_after();

        // GN per-thread state (registers): pooled max/min of this thread's
        // 4-column windows (4 per 16-column chunk, at most 4 chunks: P <= 128)
        constexpr int kMaxWin = 16;
        float pmx[kMaxWin], pmn[kMaxWin];
        float ls = 0.0f, lss = 0.0f;
        if (kGN) {
#pragma unroll
            for (int k = 0; k < kMaxWin; ++k) pmx[k] = -INFINITY, pmn[k] = INFINITY;
        }

        for (int u = 0; u < a.U; ++u) {
            const int row = r0 + u * a.S + slot;  // the same for the whole warp
            if constexpr (kGN) {
#pragma unroll
                for (int kc = 0; kc < kMaxWin / 4; ++kc) {
                    const int cc = hc + NH * kc;
                    if (cc >= nchunks) break;
                    const int col0 = cc * 16;
                    float v[16];
                    tmem_ld16(tmem + lane_off + ab * kAccStride + u * a.ucol + col0, v);
                    if (row < a.Ho) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            v[i] += bias;
                            if (col0 + i < a.Wo) {
                                ls += v[i];
                                lss = fmaf(v[i], v[i], lss);
                            }
                        }
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            const float mx = fmaxf(fmaxf(v[4 * wi], v[4 * wi + 1]), fmaxf(v[4 * wi + 2], v[4 * wi + 3]));
                            const float mn = fminf(fminf(v[4 * wi], v[4 * wi + 1]), fminf(v[4 * wi + 2], v[4 * wi + 3]));
                            pmx[4 * kc + wi] = fmaxf(pmx[4 * kc + wi], mx);
                            pmn[4 * kc + wi] = fminf(pmn[4 * kc + wi], mn);
                        }
                    }
                }
            } else {
            for (int cc = hc; cc < nchunks; cc += NH) {
                const int col0 = cc * 16;
                float v[16];
                tmem_ld16(tmem + lane_off + ab * kAccStride + u * a.ucol + col0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] += bias;
                if (kMin) {
                    reduce_scatter16(v, lane, sgn);
                    if ((lane & 1) == 0) scratch[(u * 4 + qd) * a.P + col0 + (lane >> 1)] = v[0];
                } else if (KIND == CONV_EPI_MUL_LRELU_GELU) {
                    float *stg = scratch + ew * 32 * kStgPitch;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float t = v[i] * mult;
                        t = t > 0.0f ? t : a.slope * t;
                        stg[lane * kStgPitch + i] = gelu_erf(t);
                    }
                    __syncwarp();
                    const int c = lane & 15;
                    if (row < a.Ho && col0 + c < a.Wo) {
#pragma unroll 4
                        for (int rp = 0; rp < 16; ++rp) {
                            const int rr = 2 * rp + (lane >> 4);
                            const int cor = (qd * 32 + rr) % a.Cout;
                            a.out[(((size_t)n * a.Cout + cor) * a.Ho + row) * a.Wo + col0 + c] = stg[rr * kStgPitch + c];
                        }
                    }
                    __syncwarp();
                }
            }
            }
        }
        // tensor memory of this unit is no longer needed
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.acc_empty(ab));

        if (kMin) {
            epi_bar<R::kEpiThreads>();
            const int qps = 4 / a.S;  // quadrants per slot
            for (int idx = et; idx < a.U * a.S * a.P; idx += R::kEpiThreads) {
                const int u = idx / (a.S * a.P), rem = idx % (a.S * a.P);
                const int s = rem / a.P, col = rem % a.P;
                const int row = r0 + u * a.S + s;
                if (row >= a.Ho || col >= a.Wo) continue;
                float m = scratch[(u * 4 + s * qps) * a.P + col];
                for (int k = 1; k < qps; ++k) m = rs_op(m, scratch[(u * 4 + s * qps + k) * a.P + col], sgn);
                float o = sgn == 0 ? 0.0f * m : a.scalar * m;
                if (KIND == CONV_EPI_MIN_TANH2) o = tanhf(tanhf(o));
                a.out[((size_t)n * a.Ho + row) * a.Wo + col] = o;
            }
            epi_bar<R::kEpiThreads>();
        } else if (kGN) {
            // pool: combine the two row slots (S == 2) through shared memory
            float *xg = scratch;                                  // [8 warps][32 lanes][kMaxWin][2]
            float *st = scratch + R::kEpiWarps * 32 * kMaxWin * 2;  // [8 warps][32 lanes][2]
            st[(ew * 32 + lane) * 2] = ls;
            st[(ew * 32 + lane) * 2 + 1] = lss;
#pragma unroll
            for (int k = 0; k < kMaxWin; ++k) {
                xg[((ew * 32 + lane) * kMaxWin + k) * 2] = pmx[k];
                xg[((ew * 32 + lane) * kMaxWin + k) * 2 + 1] = pmn[k];
            }
            epi_bar<R::kEpiThreads>();
            if (slot == 0 && ru < a.Hp) {
                const int ew1 = hc * 4 + qd + 2;  // warp holding the same channel in row slot 1
#pragma unroll
                for (int k = 0; k < kMaxWin; ++k) {
                    const int cc = hc + NH * (k / 4);
                    const int pw = cc * 4 + (k % 4);
                    if (cc >= nchunks || pw >= a.Wp) continue;
                    float mx = pmx[k], mn = pmn[k];
                    if (a.S == 2) {
                        mx = fmaxf(mx, xg[((ew1 * 32 + lane) * kMaxWin + k) * 2]);
                        mn = fminf(mn, xg[((ew1 * 32 + lane) * kMaxWin + k) * 2 + 1]);
                    }
                    const size_t o = (((size_t)n * a.Cout + co) * a.Hp + ru) * a.Wp + pw;
                    a.gn.pmax[o] = mx;
                    a.gn.pmin[o] = mn;
                }
            }
            // statistics: fixed-order sum per group
            const int cpg = a.Cout / a.groups;
            for (int g = et; g < a.groups; g += R::kEpiThreads) {
                double s0 = 0.0, s1 = 0.0;
                for (int s = 0; s < a.S; ++s)
                    for (int h2 = 0; h2 < 2; ++h2)
                        for (int c2 = g * cpg; c2 < (g + 1) * cpg; ++c2) {
                            const int LL = s * a.Cout + c2;
                            const int e2 = h2 * 4 + (LL >> 5);
                            s0 += st[(e2 * 32 + (LL & 31)) * 2];
                            s1 += st[(e2 * 32 + (LL & 31)) * 2 + 1];
                        }
                double *dst = a.gn.part + (((size_t)n * a.units_per_img + ru) * a.groups + g) * 2;
                dst[0] = s0;
                dst[1] = s1;
            }
            epi_bar<R::kEpiThreads>();
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) tc_conv_epi(const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    Bars bars;
    bars.base = sbase + a.stage0_off + a.stages * a.stage_bytes;
    bars.stages = a.stages;
    uint32_t *tmem_slot =
        reinterpret_cast<uint32_t *>(smem + a.stage0_off + a.stages * a.stage_bytes + 8 * Bars::count(a.stages));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *scratch = reinterpret_cast<float *>(smem + a.scratch_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(bars.full_w(s), 1);
            mbar_init(bars.full_x(s), Roles<KIND>::kConvThreads);
            mbar_init(bars.empty(s), 1);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(bars.acc_full(ab), 1);
            mbar_init(bars.acc_empty(ab), Roles<KIND>::kEpiWarps);
        }
        mbar_init(bars.final_bar(), 1);
        mbar_init(bars.wres(), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if ((tmem & 0xFFFFu) != 0 && threadIdx.x == 0) atomicOr(a.err, ERRBIT_TMEM);

    if (warp == 0) {
        if (lane == 0) mma_role(a, sbase, bars, tmem, abort_flag);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) weight_role(a, sbase, bars, abort_flag);
        __syncwarp();
    } else if (warp < Roles<KIND>::kEpiWarp0) {
        converter_role<Roles<KIND>::kConvThreads, Roles<KIND>::kNBMax>(
            a, smem, bars, abort_flag, threadIdx.x - Roles<KIND>::kConvWarp0 * 32);
    } else {
        epilogue_role<KIND>(a, scratch, bars, tmem, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------ filter packing ----
// wpack[c][kw][jg][p][co][e] = tf32(w[co][8c + 4jg + e][kh][kw]) with
// kh = S+1-p when 0 <= kh <= 2, else 0 (the zero planes that pad the
// stacked row slots).
__global__ void pack_weights(const float *__restrict__ w, float *__restrict__ wp, int Cin, int Cout, int S) {
    const int planes = 2 * S + 1;
    const size_t total = (size_t)Cin * 3 * planes * Cout;  // = chunks*3*2*planes*Cout*4
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        size_t r = i;
        const int e = r % 4;
        r /= 4;
        const int co = r % Cout;
        r /= Cout;
        const int p = r % planes;
        r /= planes;
        const int jg = r % 2;
        r /= 2;
        const int kw = r % 3;
        const int c = (int)(r / 3);
        const int kh = S + 1 - p;
        float v = 0.0f;
        if (kh >= 0 && kh <= 2) v = w[(((size_t)co * Cin + 8 * c + 4 * jg + e) * 3 + kh) * 3 + kw];
        wp[i] = __uint_as_float(f32_to_tf32(v));
    }
}

// ----------------------------------------------------------- planning ----
struct Plan {
    int S, P, U, RU, Rin, PL, chunks, ucol;
    uint32_t a_bytes, b_bytes, stage_bytes, scratch_bytes, scratch_off, stage0_off, b_off;
    int stages, resident;
    size_t smem;
};

uint32_t scratch_bytes_for(int kind, int U, int P) {
    switch (kind) {
    case CONV_EPI_MIN_TANH2:
    case CONV_EPI_SCALE_MIN:
        return (uint32_t)(U * 4 * P * sizeof(float));
    case CONV_EPI_MUL_LRELU_GELU:
        return (uint32_t)(Roles<CONV_EPI_MUL_LRELU_GELU>::kEpiWarps * 32 * kStgPitch * sizeof(float));
    case CONV_EPI_GN_SCALE_POOL_CLAMP: {
        constexpr int ew = Roles<CONV_EPI_GN_SCALE_POOL_CLAMP>::kEpiWarps;
        return (uint32_t)((ew * 32 * 16 * 2 + ew * 32 * 2) * sizeof(float));
    }
    }
    return 0;
}

int conv_threads_for(int kind) {
    switch (kind) {
    case CONV_EPI_MIN_TANH2: return Roles<CONV_EPI_MIN_TANH2>::kConvThreads * Roles<CONV_EPI_MIN_TANH2>::kNBMax;
    case CONV_EPI_SCALE_MIN: return Roles<CONV_EPI_SCALE_MIN>::kConvThreads * Roles<CONV_EPI_SCALE_MIN>::kNBMax;
    case CONV_EPI_MUL_LRELU_GELU:
        return Roles<CONV_EPI_MUL_LRELU_GELU>::kConvThreads * Roles<CONV_EPI_MUL_LRELU_GELU>::kNBMax;
    default:
        return Roles<CONV_EPI_GN_SCALE_POOL_CLAMP>::kConvThreads * Roles<CONV_EPI_GN_SCALE_POOL_CLAMP>::kNBMax;
    }
}

// Shared memory: [resident filter][stages x (A? + B)][mbarriers][tmem slot, abort][scratch]
bool make_plan(const conv_epi_desc &d, int kind, Plan &pl) {
    if (!(d.Cout == 64 || d.Cout == 128)) return false;
    if (d.Cin % 8 != 0 || d.W % 4 != 0 || d.W > 256 || d.H < 3) return false;
    pl.S = 128 / d.Cout;
    pl.P = (d.W + 15) / 16 * 16;
    pl.ucol = (pl.P + 31) / 32 * 32;
    pl.U = kAccStride / pl.ucol;
    pl.RU = pl.U * pl.S;
    pl.Rin = pl.RU + 2;
    pl.PL = (pl.Rin * pl.P + 4 + 7) / 8 * 8;
    pl.chunks = d.Cin / 8;
    if (pl.PL >= (1 << 16)) return false;
    // every 4x4 block of a chunk's B plane has a converter slot
    if (pl.PL / 2 > conv_threads_for(kind)) return false;
    pl.a_bytes = 3u * 2u * (2 * pl.S + 1) * d.Cout * 16u;
    pl.b_bytes = 2u * pl.PL * 16u;
    pl.scratch_bytes = scratch_bytes_for(kind, pl.U, pl.P);
    auto fits = [&](int st, uint32_t stage, uint32_t res) {
        const size_t bars_end = (size_t)res + (size_t)st * stage + 8u * Bars::count(st) + 8u;
        return ((bars_end + 15) & ~(size_t)15) + pl.scratch_bytes <= (size_t)kSmemLimit;
    };
    // keep the whole filter resident when it leaves room for at least 3 stages of B
    const uint32_t res_bytes = (pl.chunks * pl.a_bytes + 1023u) & ~1023u;
    const uint32_t b_stage = (pl.b_bytes + 1023u) & ~1023u;
    if (fits(3, b_stage, res_bytes)) {
        pl.resident = 1;
        pl.stage_bytes = b_stage;
        pl.stage0_off = res_bytes;
        pl.b_off = 0;
    } else {
        pl.resident = 0;
        pl.stage_bytes = (pl.a_bytes + pl.b_bytes + 1023u) & ~1023u;
        pl.stage0_off = 0;
        pl.b_off = pl.a_bytes;
    }
    int st = kMaxStages;
    while (st >= 2 && !fits(st, pl.stage_bytes, pl.stage0_off)) --st;
    if (st < 2) return false;
    pl.stages = st;
    pl.scratch_off = (pl.stage0_off + (uint32_t)st * pl.stage_bytes + 8u * Bars::count(st) + 8u + 15u) & ~15u;
    pl.smem = pl.scratch_off + pl.scratch_bytes;
    return true;
}

uint32_t make_idesc(int M, int N) {
    // kind::tf32 instruction descriptor: D fp32 (bits 4-5 = 1), A tf32 (bits 7-9 = 2),
    // B tf32 (bits 10-12 = 2), both K-major (bits 15, 16 = 0), N>>3 at bits 17-22,
    // M>>4 at bits 24-28; dense, no negation, no saturation.
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int KIND>
conv_epi_status launch_tc(const TcArgs &a, const Plan &pl, int grid, cudaStream_t s) {
    auto k = tc_conv_epi<KIND>;
    CE_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem));
    k<<<grid, kThreads, pl.smem, s>>>(a);
    CE_CUDA(cudaGetLastError());
    return CONV_EPI_OK;
}

}  // namespace

conv_epi_status tc_supported(const conv_epi_desc &d, const conv_epi_epilogue_desc *e) {
    Plan pl;
    const int kind = e ? e->kind : CONV_EPI_MIN_TANH2;
    if (!make_plan(d, kind, pl)) return CONV_EPI_ERR_UNSUPPORTED;
    if (e && e->kind == CONV_EPI_GN_SCALE_POOL_CLAMP) {
        // the epilogue pools 4x4 windows over one band of 4 rows per unit,
        // with at most 4 sixteen-column chunks per epilogue warp
        if (e->pool_k != 4 || pl.RU != 4 || pl.P > 128 || pl.S != 2) return CONV_EPI_ERR_UNSUPPORTED;
    }
    return CONV_EPI_OK;
}

size_t tc_wpack_bytes(const conv_epi_desc &d) {
    const int S = d.Cout >= 128 ? 1 : 2;
    return (size_t)d.Cin * 3 * (2 * S + 1) * d.Cout * sizeof(float) + 256;
}

int tc_gn_units(const conv_epi_desc &d, int Ho, int pool_k) {
    Plan pl;
    if (!make_plan(d, CONV_EPI_GN_SCALE_POOL_CLAMP, pl)) return (Ho + pool_k - 1) / pool_k;
    return (Ho + pl.RU - 1) / pl.RU;
}

conv_epi_status tc_forward(conv_epi_handle h, const float *x, const float *w, const float *b,
                           const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    Plan pl;
    if (!make_plan(d, e.kind, pl)) return CONV_EPI_ERR_UNSUPPORTED;
    // 1) pack the filter for this call
    {
        const size_t total = (size_t)d.Cin * 3 * (2 * pl.S + 1) * d.Cout;
        const int threads = 256;
        const int blocks = (int)((total + threads - 1) / threads);
        pack_weights<<<blocks, threads, 0, s>>>(w, h->wpack, d.Cin, d.Cout, pl.S);
        CE_CUDA(cudaGetLastError());
    }
    TcArgs a{};
    a.x = x, a.b = b, a.wpack = h->wpack, a.out = out, a.err = h->dev_err;
    a.N = d.N, a.Cin = d.Cin, a.H = d.H, a.W = d.W, a.Cout = d.Cout, a.Ho = h->Ho, a.Wo = h->Wo;
    a.S = pl.S, a.P = pl.P, a.U = pl.U, a.RU = pl.RU, a.PL = pl.PL, a.ucol = pl.ucol;
    a.p_magic = (uint32_t)((((uint64_t)1 << 32) + pl.P - 1) / pl.P);
    a.chunks = pl.chunks;
    a.units_per_img = (h->Ho + pl.RU - 1) / pl.RU;
    a.total_units = d.N * a.units_per_img;
    a.stages = pl.stages;
    a.a_bytes = pl.a_bytes, a.b_bytes = pl.b_bytes, a.stage_bytes = pl.stage_bytes, a.scratch_off = pl.scratch_off;
    a.resident = pl.resident, a.stage0_off = pl.stage0_off, a.b_off = pl.b_off;
    a.a_plane_bytes = (uint32_t)d.Cout * 16u;
    a.a_lbo = (uint32_t)(2 * pl.S + 1) * a.a_plane_bytes;
    a.a_kw_stride = 2u * a.a_lbo;
    a.idesc = make_idesc(128, pl.P);
    a.scalar = e.scalar, a.chan_scale = e.chan_scale, a.slope = e.lrelu_slope;
    a.groups = e.groups, a.pool_k = e.pool_k;
    if (e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP) {
        a.gn = h->gn;
        a.Hp = h->gn.Hp, a.Wp = h->gn.Wp;
        if (h->gn.units != a.units_per_img) return CONV_EPI_ERR_INVALID_ARG;
    }
    const int grid = a.total_units < h->sm_count ? a.total_units : h->sm_count;
    conv_epi_status st;
    switch (e.kind) {
    case CONV_EPI_MIN_TANH2: st = launch_tc<CONV_EPI_MIN_TANH2>(a, pl, grid, s); break;
    case CONV_EPI_SCALE_MIN: st = launch_tc<CONV_EPI_SCALE_MIN>(a, pl, grid, s); break;
    case CONV_EPI_MUL_LRELU_GELU: st = launch_tc<CONV_EPI_MUL_LRELU_GELU>(a, pl, grid, s); break;
    case CONV_EPI_GN_SCALE_POOL_CLAMP: st = launch_tc<CONV_EPI_GN_SCALE_POOL_CLAMP>(a, pl, grid, s); break;
    default: return CONV_EPI_ERR_INVALID_ARG;
    }
    if (st) return st;
    h->last_launches = 2;
    if (e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP) {
        if ((st = gn_finalize(h, e, out, s))) return st;
        h->last_launches = 3;
    }
    return CONV_EPI_OK;
}

}  // namespace conv_epi
