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
//      (16-byte aligned) change of the descriptor's start address.
//   A (128 rows x 8 channels): packed filter planes (bulk copy engine).
// Accumulators live in tensor memory (128 lanes x 512 columns, fp32).
//
// Input path.  The TMA engine loads each raw NCHW tile (8 channels x the
// unit's input rows x W) into a ring of staging buffers, zero-filling rows past
// the image.  Converter warps rewrite a staged tile shared->shared into the
// B plane (each lane gathers one position's four channels, rounds them to
// tf32 and stores one 16-byte plane row), so their proxy fence before handing
// the plane to the tensor core covers only short shared-memory stores --
// never global loads in flight.  Channels-last input (x as [N][H][W][Cin])
// skips both: its 4-channel boxes land straight in the B planes, whose
// 16-byte position rows they already match.  A tensor map's row stride must
// be a multiple of 16 bytes, so NCHW rows whose W is not a multiple of 4 are
// read from a padded copy of x (pad_rows, before the conv kernel).
//
// Row slots.  The MMA's M is 128.  With Cout = 128 a tile is one output row
// per accumulator.  With Cout = 64 the 128 accumulator lanes hold TWO output
// rows (lanes 0-63: row r, lanes 64-127: row r+1): the A tile for the
// position shift "sk" stacks W(kh = sk) over W(kh = sk-1), so one MMA feeds
// both rows from the same input window.  Shifts sk = 0..3 cover kh = 0..2 of
// both rows; the two missing (kh = -1, kh = 3) blocks are zero, so 12 MMAs do
// the work of 9 full-height ones -- still 1.5x the rate of the M = 64 shape.
//
// One CTA per SM (persistent), 16 warps; warp w issues on sub-partition w % 4:
//   warp 0      tensor-memory allocator + single-thread MMA issuer
//   warp 4      producer: TMA tensor loads of input tiles into the staging
//               ring and bulk copies of the filter (streamed per chunk, or
//               loaded once when it stays resident)
//   warps 1-3, 5-7  converters (staged tile -> B plane)
//   warps 8-15  epilogue (tensor memory -> chain -> global), two warps per
//               32-lane quadrant, alternating column chunks
// The MMA thread's instruction stream (descriptor steps, MMA issue, commits)
// is on the tensor pipe's critical path, so its sub-partition carries no
// converter: only the mostly waiting producer and two epilogue warps.
// Rings (mbarrier full/empty pairs): filter stages, B planes, staged tiles;
// two accumulator buffers in tensor memory so the epilogue of one unit
// overlaps the main loop of the next.  Every wait is bounded (2 s of
// %globaltimer); on expiry the kernel raises an error bit, drains what it has
// in flight and returns, so the context stays usable.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "gn_common.cuh"
#include "internal.h"

namespace conv_epi {
namespace {

constexpr int kThreads = 512;
constexpr int kProducerWarp = 4, kConvWarps = 6;
// converter index 0..5 of warps 1-3, 5-7
__device__ __forceinline__ int conv_index(int warp) { return warp < kProducerWarp ? warp - 1 : warp - 2; }
constexpr int kEpiWarp0 = 8, kEpiWarps = 8, kEpiThreads = kEpiWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;     // columns per accumulator buffer
constexpr int kMaxRing = 4;
constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA
constexpr int kPoolPitch = 33;      // GroupNorm pooled tile pitch (floats)
// Internal kind: the conv output y (as CONV_EPI_NONE) plus each thread's sums
// of y and y^2 per unit, the first pass of the two-pass GroupNorm form.
constexpr int kKindConvStats = 6;
// Internal kind: the GroupNorm chain beyond the page's 64 stacked channels --
// fewer than 64 (zero filters past Co) or 65..128 (no stacking, half a band
// per unit).  A separate instantiation, so that the page's shape keeps the
// lean kernel: with these cases compiled into it, it measured 8-10 us slower
// (86.5 -> 96 us for C5), its registers at the cap.
constexpr int kKindGnX = 7;
// ... and its one-band rows of 64..95 outputs (P = 80 or 96), which mask one
// chunk more: an instantiation of their own, so the wider rows keep one mask
// (measured: the second mask cost Cout 128 at W 128 9 %).
constexpr int kKindGnXNarrow = 8;
// ... and rows of 130..256 columns with Cout <= 64 (P 144..256): one row pair,
// half a band, per unit, its up to 63 windows in two passes of 4 chunks per
// warp (the second masked).
constexpr int kKindGnWide = 9;
// ... and 2 x 2 pooling windows (Cout <= 64, rows of 64..126 outputs, or of
// up to 62 in the four-u instantiation): each of a unit's row pairs is a
// pooling band, 8 windows per 16-column chunk.
constexpr int kKindGnPool2 = 10;
// ... and more than 128 channels (rows of up to 64 or of 64..126 outputs):
// channel tiles of 128, each unit one tile's band or half band (with the
// tile handling compiled into the kind above, its Cout 128 shapes measured
// 5 % slower).
constexpr int kKindGnTiles = 11;
// ... and rows wider than 256 columns (Cout <= 64): column tiles of 252
// outputs (63 whole windows), each unit one tile of one row pair, as in the
// 130..256-column kind but with each unit's column masks and window offset
// (also rows of 127 outputs, whose first pass needs the mask).
constexpr int kKindGnColTiles = 12;
// ... and 2 x 2 windows over 65..128 channels (rows of 64..126 outputs, or
// of up to 62 with four u): no row stacking, each pair of a unit's 1-row u
// one band (compiled into the kind of 2 x 2 windows above, the stacking
// checks cost its shapes 8 %).
constexpr int kKindGnPool2S1 = 13;
// ... and 2 x 2 windows on rows of 130..240 columns (Cout <= 64): one row
// pair, one band, per unit, its up to 119 windows gathered in two passes of
// four chunks per warp (the second masked) straight into the tile (with
// rows of 256 staged columns the two-slot tile and the minimal rings exceed
// shared memory).
constexpr int kKindGnWideP2 = 14;
// ... and 65..128 channels on rows of 130..256 columns: no row stacking, so
// a unit is one row, a quarter of a 4-row band; its extremes go to one of
// four workspace slots (pmax, pmin and the index buffers, which this path
// leaves free), folded by the finalize.
constexpr int kKindGnWideS1 = 15;
__host__ __device__ constexpr bool is_gnx(int kind) {
    return kind == kKindGnX || kind == kKindGnXNarrow || kind == kKindGnWide || kind == kKindGnPool2 ||
           kind == kKindGnTiles || kind == kKindGnColTiles || kind == kKindGnPool2S1 || kind == kKindGnWideP2 ||
           kind == kKindGnWideS1;
}
__host__ __device__ constexpr bool is_gn(int kind) { return kind == CONV_EPI_GN_SCALE_POOL_CLAMP || is_gnx(kind); }
// the fused GroupNorm kernel for a problem: the page's 64 stacked channels (rows of up to 64 or of
// 96..126 outputs), or one of the generalised instantiations (tc_gn_fused decides whether it runs)
inline int tc_gn_kind(const conv_epi_desc &d, int pool_k) {
    if (pool_k == 2 && d.Cout <= 64 && d.W <= 128 && d.W != 65) return kKindGnPool2;
    if (pool_k == 2 && d.Cout <= 64 && d.W >= 130 && d.W <= 256) return kKindGnWideP2;  // (where its plan fits)
    if (pool_k == 2 && d.Cout <= 128 && d.W <= 128 && d.W != 65) return kKindGnPool2S1;
    if (d.Cout > 64 && d.Cout <= 128 && d.W >= 130 && d.W <= 256) return kKindGnWideS1;
    if (d.Cout > 128) return kKindGnTiles;
    // (rows of 127 outputs too: one tile, its first pass masked)
    if ((d.W > 256 || d.W == 129) && d.Cout <= 64) return kKindGnColTiles;
    if (d.W > 128) return kKindGnWide;
    if (d.W > 64 && d.W - 2 < 96) return kKindGnXNarrow;
    return d.Cout == 64 ? CONV_EPI_GN_SCALE_POOL_CLAMP : kKindGnX;
}
constexpr int kMaxQ = 8;            // min chains: quadrant partials of a column loaded together

// Scalar kernel configuration.  The kernel copies it out of the parameter
// space into a local at entry, so the roles keep the fields in registers
// (reads through the parameter would be repeated after every asm statement
// that clobbers memory, on the critical path of every loop).
// (Measured: on the GroupNorm kernel, one more 8-byte field in this struct cost
// about 5 us of 88, with the same registers and no spills; so mode flags are
// derived from fields already here, and the conv-with-sums kind passes its
// buffer in gn.pmax, which only the GroupNorm kind otherwise uses.)
struct Cfg {
    const float *x, *b, *wpack;
    float *out;
    unsigned *err;
    int N, Cin, H, W, Cout, Ho, Wo;  // Cout: the GEMM's per channel tile (64 or 128)
    int Co;                          // the problem's output channels (<= Cout * MT)
    int S, P, U, RU, Rin, PL, ucol;
    int chunks, units_per_img, total_units;
    int CT, CW, BW;    // column tiles per row block, output columns per tile, staged tile width (NCHW)
    int MT;            // output-channel tiles of 128 (Cout > 128), each its own unit
    int resident;      // 1: the whole packed filter stays in shared memory
    int na, nb, nr;    // ring depths: filter stages (streaming), B planes, staged tiles
    uint32_t a_bytes, b_bytes, raw_bytes, raw_tx;  // raw_tx: exact bytes of one staged tile
    uint32_t a_off, b_off, raw_off, bar_off, scratch_off;
    uint32_t a_kw_stride, a_lbo, a_plane_bytes;
    uint32_t idesc;
    float scalar;
    const float *chan_scale, *gamma;
    float slope;
    int groups, Hp, Wp;
    GnWork gn;
    int drop_tile;  // test hook: per-CTA staged-tile index the producer never issues (-1: none)
    int nhwc;       // channels-last input: tiles go straight into the B planes (no staging, no converters)
    // GroupNorm chain finalized inside this kernel (cooperative launch)
    int gn_fin;
    const float *beta;
    float eps, lo, hi;
    float cnt;            // C/groups * Ho * Wo
    uint32_t per_magic;   // ceil(2^32 / (Hp * Wp))
    uint32_t f4_magic;    // ceil(2^32 / F4), F4 = float4 per (image, group) block
};

struct TcArgs {        // 64-byte aligned through CUtensorMap
    CUtensorMap xmap;  // x as a 4-D tensor: (W, H, Cin, N) with box (BW, Rin, 8, 1), or channels last
    Cfg c;
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
// as above, but a thread whose phase is not complete sleeps until it
// completes or `ns` nanoseconds pass, instead of returning at once: waiting
// warps then issue nothing (a polling loop of plain try_waits competes with
// the converters' shared-memory traffic in the same pipe)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
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
// shared -> global bulk copy (both addresses 16-byte aligned, size a multiple
// of 16), tracked by bulk groups of the issuing thread
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the issuing thread's bulk stores have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// 4-D tiled TMA load; coordinates innermost first
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Programmatic dependent launch: the conv kernel is launched while the
// small kernel before it (filter pack, row padding, output fill) still runs,
// so its launch and prologue overlap that kernel; every thread of it waits
// here for the preceding grid's completion and memory before its roles touch
// global memory.  (A no-op when launched without the attribute.)
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// fp32 -> tf32 (10 explicit mantissa bits), round to nearest with ties away
// from zero (the conversion instruction; measured cheaper here than the same
// rounding done with integer operations on the bit pattern)
__device__ __forceinline__ uint32_t f32_to_tf32(float f) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
    return r;
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }
// barrier over the epilogue warps that also ORs a flag across them, so they
// all take the same branch after it
__device__ __forceinline__ bool epi_bar_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kEpiThreads)
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
// two fp32 values as one 64-bit register pair, and the packed fp32x2 FMA
// d = a * b + c on such pairs (both halves rounded to nearest)
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma2u(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2u(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float2 fma2(uint64_t a, uint64_t b, uint64_t c) { return unpack2(fma2u(a, b, c)); }
__device__ __forceinline__ uint64_t mul2u(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t pack2f(float lo, float hi) { return pack2(__float_as_uint(lo), __float_as_uint(hi)); }
__device__ __forceinline__ uint64_t neg2(uint64_t a) { return a ^ 0x8000000080000000ull; }  // exact
// atomic minimum of a float in global memory: non-negative floats order like
// their bit patterns as signed integers, negative ones in reverse as unsigned
__device__ __forceinline__ void atomic_min_f32(float *p, float v) {
    if (v >= 0.0f) atomicMin(reinterpret_cast<int *>(p), __float_as_int(v));
    else atomicMax(reinterpret_cast<unsigned *>(p), __float_as_uint(v));
}
// minimum / maximum of three (NaN operands are ignored, as by fminf / fmaxf)
__device__ __forceinline__ float fmin3(float x, float y, float z) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
    return r;
}
__device__ __forceinline__ float fmax3(float x, float y, float z) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
    return r;
}
// arrive on `bar` once every MMA this thread issued before has completed
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.  Issue and wait are split so
// that the next load overlaps work on the current registers; the wait names
// the destination registers so no use can be scheduled before it.
struct Frag16 {
    uint32_t r[16];
};
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, Frag16 &f) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(f.r[0]), "=r"(f.r[1]), "=r"(f.r[2]), "=r"(f.r[3]), "=r"(f.r[4]), "=r"(f.r[5]), "=r"(f.r[6]),
          "=r"(f.r[7]), "=r"(f.r[8]), "=r"(f.r[9]), "=r"(f.r[10]), "=r"(f.r[11]), "=r"(f.r[12]), "=r"(f.r[13]),
          "=r"(f.r[14]), "=r"(f.r[15])
        : "r"(taddr)
        : "memory");
}
// The same 16 columns of a warp's 32 lanes as two 16x256b loads (lanes 0-15
// into r[0..7], lanes 16-31 into r[8..15]).  In that shape thread t holds, of
// its 16-lane half, lane t/4 at columns 2(t%4), 2(t%4)+1 (r0, r1) and +8
// (r4, r5), and lane t/4 + 8 at the same columns (r2, r3, r6, r7): four
// channels of four columns per thread, so a reduction over channels starts
// inside the thread.
__device__ __forceinline__ void tmem_ld16_rows4_issue(uint32_t taddr, Frag16 &f) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(f.r[0]), "=r"(f.r[1]), "=r"(f.r[2]), "=r"(f.r[3]), "=r"(f.r[4]), "=r"(f.r[5]), "=r"(f.r[6]),
                   "=r"(f.r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(f.r[8]), "=r"(f.r[9]), "=r"(f.r[10]), "=r"(f.r[11]), "=r"(f.r[12]), "=r"(f.r[13]),
                   "=r"(f.r[14]), "=r"(f.r[15])
                 : "r"(taddr + (16u << 16))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(Frag16 &f) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(f.r[0]), "+r"(f.r[1]), "+r"(f.r[2]), "+r"(f.r[3]), "+r"(f.r[4]), "+r"(f.r[5]),
                   "+r"(f.r[6]), "+r"(f.r[7]), "+r"(f.r[8]), "+r"(f.r[9]), "+r"(f.r[10]), "+r"(f.r[11]),
                   "+r"(f.r[12]), "+r"(f.r[13]), "+r"(f.r[14]), "+r"(f.r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait2(Frag16 &f, Frag16 &g) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(f.r[0]), "+r"(f.r[1]), "+r"(f.r[2]), "+r"(f.r[3]), "+r"(f.r[4]), "+r"(f.r[5]),
                   "+r"(f.r[6]), "+r"(f.r[7]), "+r"(f.r[8]), "+r"(f.r[9]), "+r"(f.r[10]), "+r"(f.r[11]),
                   "+r"(f.r[12]), "+r"(f.r[13]), "+r"(f.r[14]), "+r"(f.r[15]), "+r"(g.r[0]), "+r"(g.r[1]),
                   "+r"(g.r[2]), "+r"(g.r[3]), "+r"(g.r[4]), "+r"(g.r[5]), "+r"(g.r[6]), "+r"(g.r[7]),
                   "+r"(g.r[8]), "+r"(g.r[9]), "+r"(g.r[10]), "+r"(g.r[11]), "+r"(g.r[12]), "+r"(g.r[13]),
                   "+r"(g.r[14]), "+r"(g.r[15])
                 :
                 : "memory");
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
// honor_abort) once another role has given up.  Sleeps in the try_wait
// between checks of the abort flag and of the time limit.
__device__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err,
                         bool honor_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (honor_abort && *abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(err, ERRBIT_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// (image, unit within the image) of unit blockIdx.x + k * gridDim.x, stepped
// without divisions: the index advances by the grid size and wraps into the
// image index (units_per_img >= 1).  A unit within the image is a row block
// and, for rows wider than one tile, a column tile, and for more than 128
// output channels a channel tile (the fastest index, so the units that share
// an input tile run side by side and find it in L2).
struct UnitPos {
    int n, ru;
    __device__ void init(int unit, int upi) { n = unit / upi, ru = unit % upi; }
    __device__ void step(int stride, int upi) {
        ru += stride;
        while (ru >= upi) ru -= upi, ++n;
    }
    // ru = (rb * CT + ct) * MT + mt: row block, column tile and channel tile
    // (no division when CT = MT = 1, the compile-time case of the fast path)
    __device__ __forceinline__ int mt(int MT) const { return MT == 1 ? 0 : ru % MT; }
    __device__ __forceinline__ int ct(int CT, int MT) const { return CT == 1 ? 0 : (MT == 1 ? ru : ru / MT) % CT; }
    __device__ __forceinline__ int rb(int CT, int MT) const { return (MT == 1 ? ru : ru / MT) / CT; }
};

// ---------------------------------------------------------- barriers ----
struct Bars {
    uint32_t base;
    __device__ uint32_t a_full(int s) const { return base + 8u * s; }
    __device__ uint32_t a_empty(int s) const { return base + 8u * (kMaxRing + s); }
    __device__ uint32_t b_full(int s) const { return base + 8u * (2 * kMaxRing + s); }
    __device__ uint32_t b_empty(int s) const { return base + 8u * (3 * kMaxRing + s); }
    __device__ uint32_t r_full(int s) const { return base + 8u * (4 * kMaxRing + s); }
    __device__ uint32_t r_empty(int s) const { return base + 8u * (5 * kMaxRing + s); }
    __device__ uint32_t acc_full(int ab) const { return base + 8u * (6 * kMaxRing + ab); }
    __device__ uint32_t acc_empty(int ab) const { return base + 8u * (6 * kMaxRing + 2 + ab); }
    __device__ uint32_t final_bar() const { return base + 8u * (6 * kMaxRing + 4); }
    __device__ uint32_t wres() const { return base + 8u * (6 * kMaxRing + 5); }
    static constexpr int kCount = 6 * kMaxRing + 6;
};

// ------------------------------------------------------------- roles ----
// One thread issues every MMA, so the work between two issues is on the
// critical path of the tensor pipe: a descriptor rebuilt from scratch per MMA
// (multiplies, shifts, masks) costs more than a 128-cycle M128 x N256 x K8
// MMA.  The descriptors are therefore built once per chunk and stepped with
// plain adds: the start-address field sits in the low bits in 16-byte units,
// so adding (bytes >> 4) moves the start (no carry leaves the field: shared
// addresses stay below 2^18).  Ring slots and phases advance by counters.
// The (S + 2) x 3 MMAs of one accumulator slot set and one chunk, unrolled:
// shift sk reads input row sk of the B plane with the A planes for kh = sk - s
// of each row slot s; tap kw moves both operands by kw.  `poll` runs after the
// second-to-last shift, while the last MMAs are still queued ahead of the
// tensor pipe, so the latency of what it does is hidden behind them.
template <int S, typename Poll>
__device__ __forceinline__ void mma_taps(uint32_t d, uint64_t ad0, uint64_t bd0, uint32_t a_pl16, uint32_t a_kw16,
                                         uint32_t P16, uint32_t idesc, bool acc0, Poll &&poll) {
#pragma unroll
    for (int sk = 0; sk <= S + 1; ++sk) {
        const uint64_t ad = ad0 - (uint64_t)(sk * a_pl16), bd = bd0 + (uint64_t)(sk * P16);
        mma_tf32(d, ad, bd, idesc, (acc0 || sk != 0) ? 1u : 0u);
        mma_tf32(d, ad + a_kw16, bd + 1, idesc, 1u);
        mma_tf32(d, ad + 2 * a_kw16, bd + 2, idesc, 1u);
        if (sk == S) poll();
    }
}

// The MMA issuer (one thread).  The tensor pipe queues only about one MMA
// ahead of the one it executes, so every cycle this thread spends between two
// MMAs beyond that is idle tensor time.  Chunk and unit boundaries therefore
// carry as little as possible: the next chunk's stage barriers (and, at the
// last chunk of a unit, the next accumulator's barrier) are tested inside the
// current chunk's MMA sequence, and a boundary waits only when that early
// test found the stage not ready yet.
__device__ __forceinline__ void mma_role(const Cfg &a, uint32_t sbase, const Bars &bars, uint32_t tmem, volatile int *abort_flag) {
    const uint64_t a_desc0 = smem_desc(0, a.a_lbo, 128);      // LBO, SBO, version; start 0
    const uint64_t b_desc0 = smem_desc(0, 16u * a.PL, 128);
    const uint32_t a_kw16 = a.a_kw_stride >> 4, a_pl16 = a.a_plane_bytes >> 4;
    const uint32_t P16 = (uint32_t)a.P;                        // one position row = 16 bytes
    const uint32_t idesc = a.idesc;
    int sa = 0, sb = 0;
    uint32_t pa = 0, pb = 0;
    bool a_ready = false, b_ready = false, acc_ready = false;  // found complete by an early test
    int j = 0;
    bool ok = true;
    if (a.resident) ok = wait_bar(bars.wres(), 0, abort_flag, a.err);
    for (int unit = blockIdx.x; ok && unit < a.total_units; unit += gridDim.x, ++j) {
        const int ab = j & 1;
        if (!acc_ready && !wait_bar(bars.acc_empty(ab), ((j >> 1) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
        }
        acc_ready = false;
        tc_fence_after();
        const uint32_t dcol = tmem + ab * kAccStride;
        const bool more_units = unit + (int)gridDim.x < a.total_units;
        for (int c = 0; c < a.chunks; ++c) {
            if ((!a.resident && !a_ready && !wait_bar(bars.a_full(sa), pa, abort_flag, a.err)) ||
                (!b_ready && !wait_bar(bars.b_full(sb), pb, abort_flag, a.err))) {
                ok = false;
                break;
            }
            a_ready = b_ready = false;
            tc_fence_after();
            // A for shift sk starts at plane S+1-sk; tap kw adds kw planes-blocks
            const uint64_t ad0 = a_desc0 + ((sbase + a.a_off + (a.resident ? c : sa) * a.a_bytes) >> 4) +
                                 (uint64_t)((a.S + 1) * a_pl16);
            uint64_t bdu = b_desc0 + ((sbase + a.b_off + sb * a.b_bytes) >> 4);
            // stage slots of the next chunk, and the next unit's accumulator
            const int sb2 = sb + 1 == a.nb ? 0 : sb + 1, sa2 = sa + 1 == a.na ? 0 : sa + 1;
            const uint32_t pb2 = sb + 1 == a.nb ? pb ^ 1u : pb, pa2 = sa + 1 == a.na ? pa ^ 1u : pa;
            const bool test_acc = c + 1 == a.chunks && more_units;
            auto poll = [&]() {
                b_ready = mbar_try_wait(bars.b_full(sb2), pb2);
                if (!a.resident) a_ready = mbar_try_wait(bars.a_full(sa2), pa2);
                if (test_acc) acc_ready = mbar_try_wait(bars.acc_empty(ab ^ 1), (((j + 1) >> 1) & 1) ^ 1);
            };
            auto none = []() {};
            uint32_t dcu = dcol;
            for (int u = 0; u < a.U; ++u, dcu += a.ucol, bdu += a.S * P16) {
                const bool last_u = u + 1 == a.U;
                if (a.S == 2) {
                    if (last_u) mma_taps<2>(dcu, ad0, bdu, a_pl16, a_kw16, P16, idesc, c != 0, poll);
                    else mma_taps<2>(dcu, ad0, bdu, a_pl16, a_kw16, P16, idesc, c != 0, none);
                } else {
                    if (last_u) mma_taps<1>(dcu, ad0, bdu, a_pl16, a_kw16, P16, idesc, c != 0, poll);
                    else mma_taps<1>(dcu, ad0, bdu, a_pl16, a_kw16, P16, idesc, c != 0, none);
                }
            }
            // the stages may be refilled once these MMAs are done
            mma_commit(bars.b_empty(sb));
            if (!a.resident) mma_commit(bars.a_empty(sa));
            sb = sb2, pb = pb2, sa = sa2, pa = pa2;
        }
        if (!ok) break;
        mma_commit(bars.acc_full(ab));  // accumulator ab is complete
    }
    // drain: every MMA issued above completes before the CTA releases tensor memory
    mma_commit(bars.final_bar());
    wait_bar(bars.final_bar(), 0, abort_flag, a.err, false);
}

// Producer (one thread): per chunk (unit, c), in order, the raw input tile
// x[n][8c .. 8c+7][r0 .. r0+Rin-1][0 .. W-1] into the next staging slot (laid
// out [8][Rin][W]; rows >= H arrive as zeros) -- for channels-last input the
// tile's two 4-channel halves straight into the next B plane, each laid out
// [Rin][P][4] -- and, when the filter streams,
// chunk c of the packed filter into the next filter slot.  The two sequences
// advance independently: while both run, the thread tests both rings without
// blocking and issues whichever copy has a free slot, so a full filter ring
// (freed only as MMAs complete) does not hold back the input tiles, which have
// the longer latency; it sleeps briefly when neither can move, and gives up
// like every other wait after kWaitLimitNs without progress.  Once only the
// tiles are left (always, with a resident filter) it blocks in wait_bar.
// TILES: channel or column tiles outside the general instantiation (the
// generalised GroupNorm kinds).
template <bool GENERAL, bool TILES>
__device__ __forceinline__ void producer_role(const Cfg &a, const CUtensorMap *xmap, uint32_t sbase, const Bars &bars,
                                              volatile int *abort_flag) {
    const char *wsrc = reinterpret_cast<const char *>(a.wpack);
    const int CT = GENERAL || TILES ? a.CT : 1, MT = GENERAL || TILES ? a.MT : 1;  // (constants 1 on the fast path)
    prefetch_tensormap(xmap);
    if (a.resident) {
        const uint32_t total = a.chunks * a.a_bytes;
        mbar_arrive_expect_tx(bars.wres(), total);
        for (uint32_t off = 0; off < total; off += 16384u)
            bulk_g2s(sbase + a.a_off + off, wsrc + off, min(16384u, total - off), bars.wres());
    }
    // this CTA's chunk sequence: units blockIdx.x, + gridDim.x, ..., chunks 0..chunks-1
    const int my_units = a.total_units > (int)blockIdx.x ? (a.total_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_units * a.chunks;
    // ring slots and phases by counters; per slot, whether a copy was issued
    // into it and that copy's phase (bit s of the masks)
    // the tile ring: staging buffers (NCHW, read by the converters) or, for
    // channels-last input, the B planes themselves (two 4-channel boxes per
    // chunk, one per K-group plane, read by the MMAs)
    const int tn = a.nhwc ? a.nb : a.nr;
    const uint32_t t_off = a.nhwc ? a.b_off : a.raw_off, t_bytes = a.nhwc ? a.b_bytes : a.raw_bytes;
    auto t_empty = [&](int s) { return a.nhwc ? bars.b_empty(s) : bars.r_empty(s); };
    auto t_full = [&](int s) { return a.nhwc ? bars.b_full(s) : bars.r_full(s); };
    int sr = 0, sa = 0;
    uint32_t pr = 0, pa = 0;
    uint32_t r_iss = 0, r_par = 0, a_iss = 0, a_par = 0;
    int ir = 0, ia = a.resident ? total : 0;  // next raw tile / next filter chunk
    int cr = 0, ca = 0;                       // chunk of tile ir / of filter chunk ia
    UnitPos pos;                              // (image, unit) of tile ir
    pos.init(blockIdx.x, a.units_per_img);
    UnitPos fpos;                             // (image, unit) of filter chunk ia (channel tile)
    fpos.init(blockIdx.x, a.units_per_img);
    uint64_t t_idle = 0;
    while (ir < total || ia < total) {
        bool moved = false;
        // with the filter sequence done (or resident), the tile sequence
        // blocks in the ordinary bounded wait
        const bool tiles_only = ia >= total;
        if (tiles_only && !wait_bar(t_empty(sr), pr ^ 1, abort_flag, a.err)) break;
        if (ir < total && (tiles_only || mbar_try_wait(t_empty(sr), pr ^ 1))) {
            if (ir != a.drop_tile) {
                const uint32_t dst = sbase + t_off + sr * t_bytes;
                mbar_arrive_expect_tx(t_full(sr), a.raw_tx);
                if (a.nhwc) {
                    // x as (C, W, H, N): channels 8c..8c+3 and 8c+4..8c+7 of
                    // rows r0.., columns 0..P-1 (past W and H: zeros)
                    const int c0 = pos.ct(CT, MT) * a.CW, r0 = pos.rb(CT, MT) * a.RU;
                    tma_load_4d(dst, xmap, 8 * cr, c0, r0, pos.n, t_full(sr));
                    tma_load_4d(dst + 16u * a.PL, xmap, 8 * cr + 4, c0, r0, pos.n, t_full(sr));
                } else {
                    // the tile's first column (a multiple of 4: 16-byte aligned)
                    tma_load_4d(dst, xmap, pos.ct(CT, MT) * a.CW, pos.rb(CT, MT) * a.RU, 8 * cr, pos.n, t_full(sr));
                }
                r_iss |= 1u << sr, r_par = (r_par & ~(1u << sr)) | (pr << sr);
            } else {
                // test hook: this slot's phase never completes, so its
                // consumers' bounded waits run out; nothing is in flight here
                r_iss &= ~(1u << sr);
            }
            if (++sr == tn) sr = 0, pr ^= 1u;
            if (++cr == a.chunks) cr = 0, pos.step(gridDim.x, a.units_per_img);
            ++ir;
            moved = true;
        }
        if (ia < total && mbar_try_wait(bars.a_empty(sa), pa ^ 1)) {
            const uint32_t dst = sbase + a.a_off + sa * a.a_bytes;
            const char *src = wsrc + ((size_t)fpos.mt(MT) * a.chunks + ca) * a.a_bytes;
            if (++ca == a.chunks) {
                ca = 0;
                if (GENERAL) fpos.step(gridDim.x, a.units_per_img);
            }
            mbar_arrive_expect_tx(bars.a_full(sa), a.a_bytes);
            for (uint32_t off = 0; off < a.a_bytes; off += 16384u)
                bulk_g2s(dst + off, src + off, min(16384u, a.a_bytes - off), bars.a_full(sa));
            a_iss |= 1u << sa, a_par = (a_par & ~(1u << sa)) | (pa << sa);
            if (++sa == a.na) sa = 0, pa ^= 1u;
            ++ia;
            moved = true;
        }
        if (moved) {
            t_idle = 0;
            continue;
        }
        if (*abort_flag) break;
        const uint64_t now = globaltimer();
        if (t_idle == 0) t_idle = now;
        else if (now - t_idle > kWaitLimitNs) {
            atomicOr(a.err, ERRBIT_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        __nanosleep(64);
    }
    // copies still in flight land before the CTA exits
    if (a.resident) wait_bar(bars.wres(), 0, abort_flag, a.err, false);
    for (int s = 0; s < tn; ++s)
        if ((r_iss >> s) & 1u) wait_bar(t_full(s), (r_par >> s) & 1u, abort_flag, a.err, false);
    for (int s = 0; s < a.na; ++s)
        if ((a_iss >> s) & 1u) wait_bar(bars.a_full(s), (a_par >> s) & 1u, abort_flag, a.err, false);
}

// Converter warps: staged tile [8][Rin][W] -> B plane [ci4][q][4].  Work
// item = 32 consecutive positions of one (ci4 group, input row): each lane
// reads its position from the 4 channel rows (consecutive lanes, consecutive
// words: no bank conflict), rounds to tf32 and writes one 16-byte plane row
// (consecutive lanes, consecutive rows: no bank conflict).  Positions with
// w >= W are zero; plane rows past the staged rows are never written (they
// only feed output columns >= Wo, which are discarded).
// A warp's items are the same in every chunk, so their shared-memory
// offsets are computed once; per chunk a thread issues all its loads before
// its first convert/store (kConvItems items in flight, no latency chain).
constexpr int kConvItems = 12;  // items per converter warp per chunk (2*Rin*ceil(P/32) <= 72, checked on host)

__device__ __forceinline__ void converter_role(const Cfg &a, uint8_t *smem, const Bars &bars, volatile int *abort_flag) {
    if (a.nhwc) return;  // channels-last tiles arrive in the B layout
    const int cw = conv_index(threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int P = a.P, W = a.BW, Rin = a.Rin, PL = a.PL;  // W: the staged tile's row length
    const int ps = Rin * W;             // floats between channels of a staged tile
    const int mP = (P + 31) >> 5;       // 32-position groups per input row
    const int nrc = 2 * Rin * mP;       // items per chunk
    // Every position of every item inside the row ("dense"): items go in pairs
    // 32 positions apart in the same row and channel group, so the second item
    // reuses the first one's four channel addresses with fixed offsets (+32
    // floats to load, +32 plane rows to store).  Otherwise one item at a time,
    // with per-lane tests.  Per item (pair): float offset into the staged tile
    // (-1: position past W, a zero row; -2: no row for this lane) and float4
    // offset of the plane row.
    const bool dense = P == W && (P & 63) == 0 && (2 * Rin * (P >> 6)) % kConvWarps <= kConvWarps / 2;
    int so[kConvItems], dof[kConvItems];
    int nk = 0;                         // items (pairs) of this warp, the same for all its lanes
    // dense: pairs beyond a whole number per warp are split into single items,
    // one each for the first warps, so no warp converts more than one item
    // above the average
    bool xone = false;                  // this warp also converts one single item
    int xso = 0, xdof = 0;
    if (dense) {
        const int mP2 = P >> 6;         // 64-position pairs per input row
        const int nrp = 2 * Rin * mP2;  // pairs per chunk (at most kConvItems / 2 per warp, checked on host)
        const int npw = nrp / kConvWarps;  // whole pairs per warp
        auto pair_at = [&](int rc, int &o_s, int &o_d, int half) {
            const int m2 = rc % mP2, t2 = rc / mP2;
            const int rr = t2 % Rin, jg = t2 / Rin;
            const int w = m2 * 64 + half * 32 + lane;
            o_s = 4 * jg * ps + rr * W + w;
            o_d = jg * PL + rr * P + w;
        };
#pragma unroll
        for (int k = 0; k < kConvItems / 2; ++k) {
            so[k] = 0, dof[k] = 0;
            if (k < npw) {
                nk = k + 1;
                pair_at(cw + k * kConvWarps, so[k], dof[k], 0);
            }
        }
        const int left = 2 * (nrp - npw * kConvWarps);  // single items left over (<= kConvWarps by the test above)
        if (cw < left) {
            xone = true;
            pair_at(npw * kConvWarps + (cw >> 1), xso, xdof, cw & 1);
        }
    } else {
#pragma unroll
        for (int k = 0; k < kConvItems; ++k) {
            const int rc = cw + k * kConvWarps;
            so[k] = -2, dof[k] = 0;
            if (rc < nrc) {
                nk = k + 1;
                const int m = rc % mP, t2 = rc / mP;
                const int rr = t2 % Rin, jg = t2 / Rin;
                const int w = m * 32 + lane;
                if (w < P) {
                    so[k] = w < W ? 4 * jg * ps + rr * W + w : -1;
                    dof[k] = jg * PL + rr * P + w;
                }
            }
        }
    }
    int sr = 0, sb = 0;
    uint32_t pr = 0, pb = 0;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < a.total_units; unit += gridDim.x) {
        for (int c = 0; c < a.chunks; ++c) {
            if (!wait_bar(bars.r_full(sr), pr, abort_flag, a.err) || !wait_bar(bars.b_empty(sb), pb ^ 1, abort_flag, a.err)) {
                ok = false;
                break;
            }
            const float *raw = reinterpret_cast<const float *>(smem + a.raw_off + sr * a.raw_bytes);
            uint4 *plane = reinterpret_cast<uint4 *>(smem + a.b_off + sb * a.b_bytes);
            float4 v[kConvItems];
            if (dense) {
#pragma unroll
                for (int k = 0; k < kConvItems / 2; ++k)
                    if (k < nk) {
                        const float *s0 = raw + so[k], *s1 = s0 + ps, *s2 = s1 + ps, *s3 = s2 + ps;
                        v[2 * k] = make_float4(s0[0], s1[0], s2[0], s3[0]);
                        v[2 * k + 1] = make_float4(s0[32], s1[32], s2[32], s3[32]);
                    }
#pragma unroll
                for (int k = 0; k < kConvItems / 2; ++k)
                    if (k < nk) {
                        uint4 *d = plane + dof[k];
                        d[0] = make_uint4(f32_to_tf32(v[2 * k].x), f32_to_tf32(v[2 * k].y), f32_to_tf32(v[2 * k].z),
                                          f32_to_tf32(v[2 * k].w));
                        d[32] = make_uint4(f32_to_tf32(v[2 * k + 1].x), f32_to_tf32(v[2 * k + 1].y),
                                           f32_to_tf32(v[2 * k + 1].z), f32_to_tf32(v[2 * k + 1].w));
                    }
                if (xone) {
                    const float *s0 = raw + xso;
                    const float4 x = make_float4(s0[0], s0[ps], s0[2 * ps], s0[3 * ps]);
                    plane[xdof] = make_uint4(f32_to_tf32(x.x), f32_to_tf32(x.y), f32_to_tf32(x.z), f32_to_tf32(x.w));
                }
            } else {
#pragma unroll
                for (int k = 0; k < kConvItems; ++k) {
                    v[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (so[k] >= 0) {
                        const float *src = raw + so[k];
                        v[k] = make_float4(src[0], src[ps], src[2 * ps], src[3 * ps]);
                    }
                }
#pragma unroll
                for (int k = 0; k < kConvItems; ++k)
                    if (so[k] >= -1)
                        plane[dof[k]] = make_uint4(f32_to_tf32(v[k].x), f32_to_tf32(v[k].y), f32_to_tf32(v[k].z),
                                                   f32_to_tf32(v[k].w));
            }
            // each thread makes its own generic-proxy stores visible to the
            // tensor core, then one arrive per warp on each barrier
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bars.r_empty(sr));  // staged tile read
                mbar_arrive(bars.b_full(sb));
            }
            if (++sr == a.nr) sr = 0, pr ^= 1u;
            if (++sb == a.nb) sb = 0, pb ^= 1u;
        }
    }
}

// Column-wise minimum of scalar * (acc + bias) over the 32 channels (lanes)
// of a warp for 16 columns, from a tmem_ld16_rows4_issue fragment.  Each
// thread first takes the min over its four channels for its four columns
// 2m, 2m+1, 8+2m, 9+2m (m = lane & 3); the eight lanes that share m then
// finish with a transposing butterfly over lane bits 4 and 3 (each level a
// lane keeps half of its columns and trades the other half with the partner
// that keeps the opposite half) and a plain exchange over bit 2: four
// shuffles for 16 columns.  Lane l ends with column
// 8*bit4(l) + 2*(l & 3) + bit3(l), which lanes l and l ^ 4 share.
// in-register step: this thread's four channels, columns 2m, 2m+1, 8+2m, 9+2m.
// A channel's two adjacent columns sit in an even/odd register pair, so the
// scale and bias go in with one packed fp32x2 FMA per pair (ss = (s, s),
// sb2[k] = (sb[k], sb[k])).
__device__ __forceinline__ float4 colmin16_own(const Frag16 &f, uint64_t ss, const uint64_t (&sb2)[4]) {
    float c[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {              // columns 2m, 2m+1 (h = 0) and 8+2m, 9+2m (h = 1)
        const int b = 4 * h;                   // registers of channel 0
        const float2 x0 = fma2(pack2(f.r[b], f.r[b + 1]), ss, sb2[0]);
        const float2 x1 = fma2(pack2(f.r[b + 2], f.r[b + 3]), ss, sb2[1]);
        const float2 x2 = fma2(pack2(f.r[b + 8], f.r[b + 9]), ss, sb2[2]);
        const float2 x3 = fma2(pack2(f.r[b + 10], f.r[b + 11]), ss, sb2[3]);
        c[2 * h] = fminf(fmin3(x0.x, x1.x, x2.x), x3.x);
        c[2 * h + 1] = fminf(fmin3(x0.y, x1.y, x2.y), x3.y);
    }
    return make_float4(c[0], c[1], c[2], c[3]);
}
// butterfly step across the eight lanes that share m
__device__ __forceinline__ float colmin16_lanes(float4 c4, int lane) {
    float c[4] = {c4.x, c4.y, c4.z, c4.w};
    const bool up16 = (lane & 16) != 0;  // keeps columns 8+2m, 9+2m
    {
        const float s0 = up16 ? c[0] : c[2], s1 = up16 ? c[1] : c[3];
        const float k0 = up16 ? c[2] : c[0], k1 = up16 ? c[3] : c[1];
        c[0] = fminf(k0, __shfl_xor_sync(0xffffffffu, s0, 16));
        c[1] = fminf(k1, __shfl_xor_sync(0xffffffffu, s1, 16));
    }
    const bool up8 = (lane & 8) != 0;    // keeps the odd column of the pair
    const float sd = up8 ? c[0] : c[1], kp = up8 ? c[1] : c[0];
    const float m = fminf(kp, __shfl_xor_sync(0xffffffffu, sd, 8));
    return fminf(m, __shfl_xor_sync(0xffffffffu, m, 4));
}
// scratch slot of the column a lane ends with, for the 16 columns at col0
__device__ __forceinline__ int colmin16_col(int col0, int lane) {
    return col0 + 8 * ((lane >> 4) & 1) + 2 * (lane & 3) + ((lane >> 3) & 1);
}

// tanh from its exponential form: tanh|x| = (1 - e) / (1 + e), e = exp(-2|x|),
// odd in x; about 1e-7 absolute error (no cancellation problem in absolute
// terms for small |x|, e -> 0 saturates to 1 for large |x|)
__device__ __forceinline__ float tanh_exp(float x) {
    const float e = __expf(-2.0f * fabsf(x));
    return copysignf(__fdividef(1.0f - e, 1.0f + e), x);
}
// GELU with the exact-erf form 0.5 t (1 + erf(t / sqrt 2)), on a pair of
// values.  erf by Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26: for x >= 0, erf(x) = 1 - (a1 u + a2 u^2 + a3 u^3 + a4 u^4 +
// a5 u^5) exp(-x^2) with u = 1 / (1 + p x), |error| <= 1.5e-7, and
// erf(-x) = -erf(x): branch-free (one reciprocal, one exponential, five FMAs
// per value), which matters in the per-channel epilogue; the strict fp32 mode
// keeps the library erff.  The arithmetic runs in packed fp32x2 operations,
// the reciprocal, exponential, absolute value and sign per value; each value
// takes the same operations and roundings as the scalar form
// 0.5 t (1 + copysign(1 - poly(u) u exp(-x^2), x)), x = t / sqrt 2, with
// 1 - poly*e as one fused multiply-add.
__device__ __forceinline__ float2 gelu_erf2(float t0, float t1) {
    const uint64_t t = pack2f(t0, t1);
    const float2 xv = unpack2(mul2u(t, pack2f(0.70710678118654752f, 0.70710678118654752f)));
    const uint64_t ax = pack2f(fabsf(xv.x), fabsf(xv.y));
    const float2 dv = unpack2(fma2u(pack2f(0.3275911f, 0.3275911f), ax, pack2f(1.0f, 1.0f)));
    const uint64_t u = pack2f(__fdividef(1.0f, dv.x), __fdividef(1.0f, dv.y));
    uint64_t poly = fma2u(pack2f(1.061405429f, 1.061405429f), u, pack2f(-1.453152027f, -1.453152027f));
    poly = fma2u(poly, u, pack2f(1.421413741f, 1.421413741f));
    poly = fma2u(poly, u, pack2f(-0.284496736f, -0.284496736f));
    poly = fma2u(poly, u, pack2f(0.254829592f, 0.254829592f));
    poly = mul2u(poly, u);
    const float2 nv = unpack2(mul2u(neg2(ax), ax));  // -x^2
    const uint64_t e = pack2f(__expf(nv.x), __expf(nv.y));
    const float2 rv = unpack2(fma2u(neg2(poly), e, pack2f(1.0f, 1.0f)));
    const uint64_t erfv = pack2f(copysignf(rv.x, xv.x), copysignf(rv.y, xv.y));
    const uint64_t half_t = mul2u(pack2f(0.5f, 0.5f), t);
    return unpack2(mul2u(half_t, add2u(pack2f(1.0f, 1.0f), erfv)));
}

// Per-chunk work of the per-channel chains (MUL_LRELU_GELU, NONE) on 16
// accumulator columns: f is a 32x32b fragment (one channel per lane, 16
// columns).  The 32 channels x 16 columns go through a per-warp staging tile
// in shared memory, [32 rows][16 floats] with the 4-float groups of row r
// XOR-swizzled by (r / 2) & 3, which keeps both sides free of bank
// conflicts: lane r writes its row as four 16-byte groups, and the stores
// read it transposed.  Where every lane's row start is 16-byte aligned (v4:
// even rows of the 254-wide maps, whose 64516-float planes keep channel
// starts aligned) lane l stores 16 bytes, columns 4 (l & 3) .. +3 of
// channels l/4 + 8 rp (rp = 0..3): each store instruction writes 8 channel
// rows of 64 contiguous bytes.  Otherwise (rows starting 8 bytes past a
// 16-byte boundary) lane l stores 8 bytes, columns 2 (l & 7), +1 of
// channels l/8 + 4 rp (rp = 0..7), or single floats for odd row widths.
// o4 / o2: this lane's first output column of its first channel in the
// current row, in the two store layouts; cstride: floats between channels.
__device__ __forceinline__ int stg_at(int r, int c) { return r * 16 + 4 * ((c >> 2) ^ ((r >> 1) & 3)) + (c & 3); }

template <int KIND>
__device__ __forceinline__ void epi_chunk_chan(const Cfg &a, const Frag16 &f, float bias, float mult, int lane, int qd,
                                               int ew, bool row_ok, bool v4, int col0, float *o4, float *o2,
                                               size_t cstride, int wv, int co_left, float *scratch, float &ys,
                                               float &yss) {
    float *stg = scratch + ew * 32 * 16;
    {
        const uint64_t bias2 = pack2f(bias, bias), mult2 = pack2f(mult, mult), slope2 = pack2f(a.slope, a.slope);
        auto tv2 = [](float2 v) { return pack2f(v.x, v.y); };
        float2 v[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            if constexpr (KIND == CONV_EPI_NONE || KIND == kKindConvStats) {
                // the conv output itself: acc + bias
                v[i / 2] = unpack2(add2u(pack2(f.r[i], f.r[i + 1]), bias2));
            } else {
                // (acc + bias) * mult for two columns, then LeakyReLU per value
                const float2 tv = unpack2(mul2u(add2u(pack2(f.r[i], f.r[i + 1]), bias2), mult2));
                const float2 sv = unpack2(mul2u(tv2(tv), slope2));
                const float t0 = tv.x > 0.0f ? tv.x : sv.x, t1 = tv.y > 0.0f ? tv.y : sv.y;
                v[i / 2] = gelu_erf2(t0, t1);
            }
        }
#pragma unroll
        for (int g = 0; g < 4; ++g)
            *reinterpret_cast<float4 *>(stg + stg_at(lane, 4 * g)) =
                make_float4(v[2 * g].x, v[2 * g].y, v[2 * g + 1].x, v[2 * g + 1].y);
        if constexpr (KIND == kKindConvStats) {
            // this channel's sums over the chunk's valid outputs
            if (row_ok) {
                if (col0 + 16 <= wv) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) ys += v[i].x + v[i].y, yss = fmaf(v[i].x, v[i].x, fmaf(v[i].y, v[i].y, yss));
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (col0 + 2 * i < wv) ys += v[i].x, yss = fmaf(v[i].x, v[i].x, yss);
                        if (col0 + 2 * i + 1 < wv) ys += v[i].y, yss = fmaf(v[i].y, v[i].y, yss);
                    }
                }
            }
        }
    }
    __syncwarp();
    if (row_ok) {
        const int cq = (qd * 32) % a.Cout;  // the quadrant's first channel in the tile
        if (v4) {
            const int k = lane & 3, col = col0 + 4 * k;
            const int cb0 = cq + (lane >> 2);
            // rp < nrp: this lane's channels cb0 + 8 rp below the tile's real
            // channels co_left (all 4 unless the GEMM is padded)
            const int nrp = co_left >= a.Cout ? 4 : max(0, min(4, (co_left - cb0 + 7) >> 3));
            const float *src = stg + stg_at(lane >> 2, 4 * k);
            float *dst = o4 + col0;
            if (col + 4 <= wv) {
#pragma unroll
                for (int rp = 0; rp < 4; ++rp)
                    if (rp < nrp)
                        *reinterpret_cast<float4 *>(dst + rp * 8 * cstride) =
                            *reinterpret_cast<const float4 *>(src + rp * 8 * 16);
            } else if (col < wv) {  // the row's ragged end
#pragma unroll
                for (int rp = 0; rp < 4; ++rp)
                    if (rp < nrp)
                        for (int e = 0; e < 4 && col + e < wv; ++e) dst[rp * 8 * cstride + e] = src[rp * 8 * 16 + e];
            }
        } else {
            const int c2 = 2 * (lane & 7), r0 = lane >> 3;
            const int cb0 = cq + r0;
            const int nrp = co_left >= a.Cout ? 8 : max(0, min(8, (co_left - cb0 + 3) >> 2));
            float *dst = o2 + col0;
            if ((a.Wo & 1) == 0) {
                if (col0 + c2 < wv) {
#pragma unroll
                    for (int rp = 0; rp < 8; ++rp)
                        if (rp < nrp)
                            *reinterpret_cast<float2 *>(dst + rp * 4 * cstride) =
                                *reinterpret_cast<const float2 *>(stg + stg_at(r0 + 4 * rp, c2));
                }
            } else {
#pragma unroll
                for (int rp = 0; rp < 8; ++rp) {
                    if (rp >= nrp) break;
                    const float *src = stg + stg_at(r0 + 4 * rp, c2);
                    if (col0 + c2 < wv) dst[rp * 4 * cstride] = src[0];
                    if (col0 + c2 + 1 < wv) dst[rp * 4 * cstride + 1] = src[1];
                }
            }
        }
    }
    __syncwarp();
}

template <int KIND, bool GENERAL>
__device__ __forceinline__ void epilogue_role(const Cfg &a, float *scratch, const Bars &bars, uint32_t tmem,
                              volatile int *abort_flag) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ew = warp - kEpiWarp0;  // 0..7
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const int qd = warp & 3;          // tensor-memory lane quadrant
    const int hc = ew >> 2;           // column group: chunks cc = hc, hc + 2, ...
    const int L = qd * 32 + lane;     // accumulator row
    const int slot = L / a.Cout, co = L % a.Cout;
    constexpr bool kMin = KIND == CONV_EPI_MIN_TANH2 || KIND == CONV_EPI_SCALE_MIN;
    constexpr bool kGnX = is_gnx(KIND);  // the generalised GroupNorm chain
    // rows of 130..256 columns, or column tiles of wider rows: two passes per unit
    constexpr bool kWide = KIND == kKindGnWide || KIND == kKindGnColTiles || KIND == kKindGnWideS1;
    constexpr bool kWideS1 = KIND == kKindGnWideS1;  // ... one row (a quarter band) per unit
    constexpr bool kColT = KIND == kKindGnColTiles;
    constexpr bool kPool2 = KIND == kKindGnPool2 || KIND == kKindGnPool2S1;  // 2 x 2 windows: a band per u
    constexpr bool kP2S1 = KIND == kKindGnPool2S1;  // ... without row stacking: a band per unit
    constexpr bool kWideP2 = KIND == kKindGnWideP2;  // 2 x 2 windows on rows of 130..256 columns
    // pooled tile pitch: up to 63 windows, (rows of up to 64 columns) 31, or
    // (2 x 2 windows on wide rows) 127
    constexpr int kPitch = kWideP2 ? 129 : kWide || (kPool2 && !GENERAL) ? 65 : kPoolPitch;
    constexpr bool kGN = KIND == CONV_EPI_GN_SCALE_POOL_CLAMP || kGnX;
    // more than 128 channels: channel tiles of 128, each unit one tile
    constexpr bool kTiles = KIND == kKindGnTiles;
    // this lane's channel parameters; with more than 128 output channels they
    // belong to the unit's channel tile and are reloaded when it changes
    // (channels Co.. pad the GEMM with zero filters)
    int cbase = 0;                    // first channel of the current channel tile
    float bias = co < a.Co ? __ldg(&a.b[co]) : 0.0f;
    float mult = KIND == CONV_EPI_MUL_LRELU_GELU && co < a.Co ? __ldg(&a.chan_scale[co]) : 0.0f;
    // GroupNorm chain: the sign of the channel's affine slope gamma * scale
    // (rstd > 0), folded into the packed filter: the accumulator is gsg * (y - b)
    auto sign_of = [&](int ch) {
        return kGN && (!kGnX || ch < a.Co) && (signbit(__ldg(&a.gamma[ch])) != signbit(__ldg(&a.chan_scale[ch]))) ? -1.0f
                                                                                                          : 1.0f;
    };
    float gsg = sign_of(co);
    // min chains: scalar * bias of the four channels this thread holds in a
    // rows4 fragment (lanes g, g+8, g+16, g+24 of the quadrant, g = lane/4),
    // each duplicated into a register pair, and the scalar likewise.  The
    // chain's minimum over channels is of scalar * y: the scalar goes in
    // first, so a negative scalar needs no separate max.
    uint64_t sb2[4];
    auto load_sb2 = [&](int cb0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int ch = cb0 + (qd * 32 + (lane >> 2) + 8 * k) % a.Cout;
            // a padding channel never wins the minimum
            const float v = !kMin ? 0.0f : ch < a.Co ? a.scalar * __ldg(&a.b[ch]) : INFINITY;
            sb2[k] = pack2(__float_as_uint(v), __float_as_uint(v));
        }
    };
    load_sb2(0);
    const uint64_t ss = pack2(__float_as_uint(a.scalar), __float_as_uint(a.scalar));
    // per-channel chains: this lane's stores go to channels cb4 + 8 rp
    // (16-byte stores) or cb2 + 4 rp (8-byte stores)
    const int cb4 = (qd * 32) % a.Cout + (lane >> 2), cb2 = (qd * 32) % a.Cout + (lane >> 3);
    const size_t plane = (size_t)a.Ho * a.Wo;
    const int nchunks = a.P / 16;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    // GroupNorm chain: group size, lanes per group inside a warp, and the sign
    // and bias tables of the pooled extremes (after the tiles, written here
    // and first read after the first combine barrier; with channel tiles,
    // rewritten per unit)
    // (groups of the problem's Co channels; the GEMM's channels from Co up
    // to its 64 or 128 are zero filters whose sums and extremes are never
    // read)
    const int gn_cpg = kGN ? (kGnX ? a.Co : a.Cout) / a.groups : 1, gn_cw = gn_cpg < 32 ? gn_cpg : 32;
    // pooling bands of 4 rows per unit: one (rows of 80..128 columns: two u
    // of two row slots) or, in the general instantiation, two (rows of up to
    // 64 columns: four u); 16-column chunks per warp and u: 4 or 2
    // (2 x 2 windows: one band per u, two per unit, 8 windows per chunk
    // written to the tiles as they are found)
    constexpr int kNB = kPool2 && GENERAL ? 4 : (kGN && (GENERAL || kPool2)) ? 2 : 1;
    constexpr int kKC = (kGN && GENERAL) ? 2 : 4;
    constexpr int kWin = 4 * kKC;  // pooling windows per band and thread (4 x 4 windows)
    float *gn_sgn = scratch + kNB * 2 * 64 * kPitch + 2 * kEpiThreads, *gn_bias = gn_sgn + (kGnX ? 128 : 64);
    if (kGN && slot == 0) gn_sgn[co] = gsg, gn_bias[co] = bias;
    // GroupNorm: this thread's chunks are cc = hc + 2 kc.  In the one-band
    // form (kKC = 4) chunks kc < kMask0 are whole: below column 96 in the
    // page-shape kernel and the generalised one (their rows have Wo >= 96),
    // below column 64 in the others (Wo >= 64); the others may hold columns >= Wo (or lie
    // past P), which the sums skip: bit 16 (kc - kMask0) + i of gn_rag is set
    // when column 16 cc + i < Wo.  (A select per value costs as much as the
    // sums, so only the chunks that can be ragged take it.)  gn_ncol counts
    // this thread's valid columns.
    constexpr int kMask0 = kWide || kWideP2 ? 4 : kKC == 4 ? (KIND == kKindGnXNarrow || kPool2 || kTiles ? 2 : 3) : 0;
    uint32_t gn_rag = 0;
    int gn_ncol = 0;
    if constexpr (kGN) {
        for (int kc = 0; kc < kKC; ++kc) {
            const int lim = a.Wo - 16 * (hc + 2 * kc);  // valid columns in the chunk
            const int nv = lim < 0 ? 0 : lim > 16 ? 16 : lim;
            gn_ncol += nv;
            if (kc >= kMask0) gn_rag |= ((1u << nv) - 1u) << (16 * (kc - kMask0));
        }
    }
    // wide rows: the second pass's chunks cc = hc + 8 + 2 kc, bit 16 kc + i
    // set when column 16 cc + i < Wo (the first pass's lie below 128 <= Wo)
    uint64_t gn_ragw = 0;
    if constexpr (kWide || kWideP2) {
        for (int kc = 0; kc < 4; ++kc) {
            const int lim = a.Wo - 16 * (hc + 8 + 2 * kc), nv = lim < 0 ? 0 : lim > 16 ? 16 : lim;
            gn_ncol += nv;
            gn_ragw |= (uint64_t)((1u << nv) - 1u) << (16 * kc);
        }
    }
    // Min chains: the cross-quadrant combine of a unit's partial minima, the
    // chain's tail and the row stores.  Every partial of a column (each row of
    // the unit, each quadrant) is loaded before any is used: under the tensor
    // core's operand traffic a shared-memory load waits long, so the loads go
    // out together instead of one row after another.  Scratch row k of the
    // unit (k = u * 4 + quadrant) holds quadrant partials; row slot s of u
    // uses quadrants s * qps .. s * qps + qps - 1.
    // with several channel tiles each one's minimum (tanh∘tanh is increasing,
    // so it commutes with the minimum) goes in by an atomic minimum on the
    // output, which starts at +inf
    auto store_min = [&](float *dst, float v) {
        if (GENERAL && a.MT > 1) atomic_min_f32(dst, v);
        else *dst = v;
    };
    auto combine_min = [&](int pn, int pr0, int pc0) {
        const int qps = 4 / a.S;  // quadrants per slot
        const int nq = a.U * 4;   // scratch rows of the unit (<= 32)
        const int wv = GENERAL ? min(a.CW, a.Wo - pc0) : a.Wo;  // the column tile's output columns
        float *orow0 = a.out + ((size_t)pn * a.Ho + pr0) * a.Wo + (GENERAL ? pc0 : 0);
        for (int col = et; col < wv; col += kEpiThreads)
            for (int kb = 0; kb < nq; kb += kMaxQ) {  // two u at a time (nq is a multiple of 4)
                float pv[kMaxQ];
#pragma unroll
                for (int k = 0; k < kMaxQ; ++k)
                    if (kb + k < nq) pv[k] = scratch[(kb + k) * a.P + col];
#pragma unroll
                for (int k = 0; k < kMaxQ; k += 4) {
                    if (kb + k >= nq) break;
                    // the 4 quadrants of u = (kb + k) / 4: one row (qps = 4) or two (qps = 2)
                    const int u = (kb + k) >> 2;
                    if (qps == 4) {
                        const int row = pr0 + u;
                        float o = fmin3(pv[k], pv[k + 1], pv[k + 2]);
                        o = fminf(o, pv[k + 3]);
                        if (KIND == CONV_EPI_MIN_TANH2) o = tanh_exp(tanh_exp(o));
                        if (row < a.Ho) store_min(orow0 + (size_t)(u) * a.Wo + col, o);
                    } else {
                        const int row = pr0 + 2 * u;
                        float o0 = fminf(pv[k], pv[k + 1]), o1 = fminf(pv[k + 2], pv[k + 3]);
                        if (KIND == CONV_EPI_MIN_TANH2) o0 = tanh_exp(tanh_exp(o0)), o1 = tanh_exp(tanh_exp(o1));
                        if (row < a.Ho) store_min(orow0 + (size_t)(2 * u) * a.Wo + col, o0);
                        if (row + 1 < a.Ho) store_min(orow0 + (size_t)(2 * u + 1) * a.Wo + col, o1);
                    }
                }
            }
    };
    int prev_n = -1, prev_r0 = 0, prev_c0 = 0;  // min chains: the unit whose combine is still due
    int j = 0;
    UnitPos pos;
    pos.init(blockIdx.x, a.units_per_img);
    for (int unit = blockIdx.x; unit < a.total_units; unit += gridDim.x, ++j, pos.step(gridDim.x, a.units_per_img)) {
        const int n = pos.n;
        const int ru = pos.ru;                  // (GroupNorm: one column tile; one channel tile but in the tiles kind)
        const int CT = GENERAL || kColT ? a.CT : 1, MT = GENERAL || kTiles ? a.MT : 1;  // constants 1 on the fast path
        const int rb = pos.rb(CT, MT);          // row block of the unit
        const int r0 = rb * a.RU;               // first output row of the unit
        const int c0 = pos.ct(CT, MT) * a.CW;   // first output column of the unit
        if ((GENERAL || kTiles) && MT > 1) {
            const int cb_unit = pos.mt(MT) * a.Cout;  // the unit's channel tile
            if (cb_unit != cbase) {
                cbase = cb_unit;
                const int ch = cbase + co;
                bias = ch < a.Co ? __ldg(&a.b[ch]) : 0.0f;
                mult = KIND == CONV_EPI_MUL_LRELU_GELU && ch < a.Co ? __ldg(&a.chan_scale[ch]) : 0.0f;
                if (kMin) load_sb2(cbase);
                if (kTiles) gsg = sign_of(ch);
            }
        }
        const int ab = j & 1;
        float ys = 0.0f, yss = 0.0f;  // kKindConvStats: this thread's sums over the unit
        const bool ok = wait_bar(bars.acc_full(ab), (j >> 1) & 1, abort_flag, a.err);
        if constexpr (kGN) {
            // the GroupNorm chain votes at the end of the unit's sums (below),
            // so a warp that finished the previous unit's stores early starts
            // this unit's loads without waiting for the others; a warp whose
            // wait failed joins that vote here and leaves with the rest
            if (!ok) {
                epi_bar_any(true);
                break;
            }
        } else if (epi_bar_any(!ok)) {  // all epilogue warps leave together
            prev_n = -1;
            break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem + lane_off + ab * kAccStride;

        // GN per-thread state: the pooled extreme of this thread's 4-column
        // windows (4 per 16-column chunk) in each band, and sums of y, y^2.
        // The extreme is the max of gsg * y: gsg = -1 turns it into the min
        // for channels whose affine slope gamma * scale * rstd is negative
        // (rstd > 0, so the sign is known before the statistics).  One array
        // per band, so every index is a compile-time constant.
        float pext0[kWin], pext1[kNB == 2 && !kPool2 ? kWin : 1];
        // sums of w and w^2 in four chains each (two packed pairs)
        uint64_t ls2[2] = {0ull, 0ull}, lss2[2] = {0ull, 0ull};
        if constexpr (kGN) {
#pragma unroll
            for (int k = 0; k < kWin; ++k) pext0[k] = -INFINITY;
            if constexpr (kNB == 2 && !kPool2) {
#pragma unroll
                for (int k = 0; k < kWin; ++k) pext1[k] = -INFINITY;
            }
        }

        int gn_rows = 0;  // this thread's rows below Ho in the unit
        bool gn_quit = false;  // wide rows: the mid-unit vote said to leave
        if constexpr (kGN) {
            // Per u: the warp's kKC chunks loaded together, then per chunk the
            // window maxima of the accumulator (sgn * (y - b)) and, over the
            // valid columns, sums of it and of its square.  The code is
            // straight-line: only chunks kc >= kMask0 select their valid
            // columns, and a row at or past Ho is skipped whole (its band is
            // never stored).
            auto gn_step = [&](const Frag16 (&f)[kKC], float (&pext)[kWin]) {
#pragma unroll
                for (int kc = 0; kc < kKC; ++kc) {
                    uint64_t v2[8];
#pragma unroll
                    for (int p = 0; p < 8; ++p) v2[p] = pack2(f[kc].r[2 * p], f[kc].r[2 * p + 1]);
                    // window extremes (windows past Wp are never stored)
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const float2 a01 = unpack2(v2[2 * wi]), a23 = unpack2(v2[2 * wi + 1]);
                        pext[4 * kc + wi] = fmax3(fmax3(a01.x, a01.y, a23.x), a23.y, pext[4 * kc + wi]);
                    }
                    if (kc >= kMask0) {  // columns >= Wo add nothing to the sums
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            const uint32_t b0 = 1u << (16 * (kc - kMask0) + 2 * p);
                            const float2 w = unpack2(v2[p]);
                            v2[p] = pack2(__float_as_uint((gn_rag & b0) ? w.x : 0.0f),
                                          __float_as_uint((gn_rag & (b0 << 1)) ? w.y : 0.0f));
                        }
                    }
                    // column i feeds chain i & 3: pair p's halves go to
                    // chains 2 (p & 1) and 2 (p & 1) + 1
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        ls2[p & 1] = add2u(ls2[p & 1], v2[p]);
                        lss2[p & 1] = fma2u(v2[p], v2[p], lss2[p & 1]);
                    }
                }
            };
            if constexpr (kWideP2) {
                // one u (rows r0, r0 + 1 in the two slots: one 2 x 2 band),
                // 8 or fewer chunks per warp in two passes of 4 (the first,
                // columns below 128, whole; the second masked); a chunk's 8
                // window maxima go to the tile at once, after the vote that
                // every warp is past the previous unit's tile reads
                if (epi_bar_any(false)) {
                    gn_quit = true;
                } else {
                    const bool row_ok = r0 + slot < a.Ho;  // the same for the whole warp
                    gn_rows += row_ok ? 1 : 0;
                    float *pt = scratch + slot * 64 * kPitch + ((qd & 1) * 32 + lane) * kPitch;
#pragma unroll
                    for (int pass = 0; pass < 2; ++pass) {
                        Frag16 f[kKC];
#pragma unroll
                        for (int kc = 0; kc < kKC; ++kc)
                            if (hc + 8 * pass + 2 * kc < nchunks)
                                tmem_ld16_issue(tbase + (hc + 8 * pass + 2 * kc) * 16, f[kc]);
                        tmem_ld_wait2(f[0], f[1]);
                        tmem_ld_wait2(f[2], f[3]);
                        if (!row_ok) continue;
#pragma unroll
                        for (int kc = 0; kc < kKC; ++kc) {
                            uint64_t v2[8];
#pragma unroll
                            for (int p = 0; p < 8; ++p) v2[p] = pack2(f[kc].r[2 * p], f[kc].r[2 * p + 1]);
                            const int pw0 = (hc + 8 * pass + 2 * kc) * 8;  // this chunk's first window
#pragma unroll
                            for (int wi = 0; wi < 8; ++wi) {
                                const float2 a01 = unpack2(v2[wi]);
                                if (pw0 + wi < kPitch - 1) pt[pw0 + wi] = fmaxf(a01.x, a01.y);
                            }
                            if (pass == 1) {  // columns >= Wo add nothing to the sums
#pragma unroll
                                for (int p = 0; p < 8; ++p) {
                                    const uint64_t b0 = 1ull << (16 * kc + 2 * p);
                                    const float2 w = unpack2(v2[p]);
                                    v2[p] = pack2(__float_as_uint((gn_ragw & b0) ? w.x : 0.0f),
                                                  __float_as_uint((gn_ragw & (b0 << 1)) ? w.y : 0.0f));
                                }
                            }
#pragma unroll
                            for (int p = 0; p < 8; ++p) {
                                ls2[p & 1] = add2u(ls2[p & 1], v2[p]);
                                lss2[p & 1] = fma2u(v2[p], v2[p], lss2[p & 1]);
                            }
                        }
                    }
                }
            } else if constexpr (kWide) {
                // one u (rows r0, r0 + 1 in the two slots), 8 or fewer chunks
                // per warp in two passes of 4: the first (columns below 128)
                // whole, the second masked; each pass's window extremes go to
                // the tile at once (windows 0..31, then 32..63)
                auto gn_step_w = [&](const Frag16 (&f)[kKC], float (&pext)[kWin], uint64_t rag) {
#pragma unroll
                    for (int kc = 0; kc < kKC; ++kc) {
                        uint64_t v2[8];
#pragma unroll
                        for (int p = 0; p < 8; ++p) v2[p] = pack2(f[kc].r[2 * p], f[kc].r[2 * p + 1]);
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            const float2 a01 = unpack2(v2[2 * wi]), a23 = unpack2(v2[2 * wi + 1]);
                            pext[4 * kc + wi] = fmax3(fmax3(a01.x, a01.y, a23.x), a23.y, pext[4 * kc + wi]);
                        }
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            const uint64_t b0 = 1ull << (16 * kc + 2 * p);
                            const float2 w = unpack2(v2[p]);
                            v2[p] = pack2(__float_as_uint((rag & b0) ? w.x : 0.0f),
                                          __float_as_uint((rag & (b0 << 1)) ? w.y : 0.0f));
                        }
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            ls2[p & 1] = add2u(ls2[p & 1], v2[p]);
                            lss2[p & 1] = fma2u(v2[p], v2[p], lss2[p & 1]);
                        }
                    }
                };
                auto put_w = [&](int pass) {
                    // (no stacking: channel row L of a 128-channel tile)
                    float *pt = scratch + (kWideS1 ? L * kPitch : slot * 64 * kPitch + ((qd & 1) * 32 + lane) * kPitch);
#pragma unroll
                    for (int k = 0; k < kWin; ++k) {
                        const int pw = (hc + 8 * pass + 2 * (k / 4)) * 4 + (k % 4);
                        if (pw < 64) pt[pw] = pext0[k];
                    }
                };
                const bool row_ok = r0 + slot < a.Ho;  // the same for the whole warp
                gn_rows += row_ok ? 1 : 0;
                // column tiles: this unit's valid columns (the last tile may
                // end below column 128), bit 16 kc + i of pass p's mask set
                // when column 16 (hc + 8 p + 2 kc) + i of the tile is an output
                uint64_t rag0 = 0, rag1 = gn_ragw;
                if constexpr (kColT) {
                    const int wv = min(a.CW, a.Wo - c0);
                    rag1 = 0;
#pragma unroll
                    for (int kc = 0; kc < kKC; ++kc) {
                        const int l0 = wv - 16 * (hc + 2 * kc), l1 = l0 - 128;
                        const int n0 = l0 < 0 ? 0 : l0 > 16 ? 16 : l0, n1 = l1 < 0 ? 0 : l1 > 16 ? 16 : l1;
                        rag0 |= (uint64_t)((1u << n0) - 1u) << (16 * kc);
                        rag1 |= (uint64_t)((1u << n1) - 1u) << (16 * kc);
                    }
                    gn_ncol = __popcll(rag0) + __popcll(rag1);
                }
                Frag16 f[kKC];
#pragma unroll
                for (int kc = 0; kc < kKC; ++kc) tmem_ld16_issue(tbase + (hc + 2 * kc) * 16, f[kc]);
                tmem_ld_wait2(f[0], f[1]);
                tmem_ld_wait2(f[2], f[3]);
                if (row_ok) {
                    if constexpr (kColT) gn_step_w(f, pext0, rag0);
                    else gn_step(f, pext0);
                }
                // every warp is past the previous unit's tile and statistics
                // reads (and none has given up) before the tile is rewritten
                if (epi_bar_any(false)) {
                    gn_quit = true;
                } else {
                    put_w(0);
#pragma unroll
                    for (int k = 0; k < kWin; ++k) pext0[k] = -INFINITY;
#pragma unroll
                    for (int kc = 0; kc < kKC; ++kc)
                        if (hc + 8 + 2 * kc < nchunks) tmem_ld16_issue(tbase + (hc + 8 + 2 * kc) * 16, f[kc]);
                    tmem_ld_wait2(f[0], f[1]);
                    tmem_ld_wait2(f[2], f[3]);
                    if (row_ok) gn_step_w(f, pext0, rag1);
                    put_w(1);
                }
            } else if constexpr (kPool2) {
                // two u (rows r0 + 2u, r0 + 2u + 1 in the two row slots), each
                // one pooling band, so a chunk's 8 window maxima are final
                // once it is processed: they go to the band's tile at once
                // (a band with a row at or past Ho is never stored, so such
                // a row writes nothing).  Every warp is past the previous
                // unit's tile and statistics reads (and none has given up)
                // before the first tile write.
                // Without row stacking (65..128 channels) the two u are the
                // rows r0, r0 + 1 of the one band, both in this thread's
                // channel row of a 128-channel tile: the first u writes its
                // maxima, the second folds its own into them in place.
                if (epi_bar_any(false)) {
                    gn_quit = true;
                } else {
#pragma unroll
                    for (int u = 0; u < (GENERAL ? 4 : 2); ++u) {  // (rows of up to 64 columns: four u, four bands)
                        const bool row_ok = r0 + (kP2S1 ? 1 : 2) * u + slot < a.Ho;  // the same for the whole warp
                        gn_rows += row_ok ? 1 : 0;
                        Frag16 f[kKC];
#pragma unroll
                        for (int kc = 0; kc < kKC; ++kc)
                            if (hc + 2 * kc < nchunks) tmem_ld16_issue(tbase + u * a.ucol + (hc + 2 * kc) * 16, f[kc]);
                        tmem_ld_wait2(f[0], f[1]);
                        tmem_ld_wait2(f[2], f[3]);
                        if (!row_ok) continue;
                        // (no stacking: band u / 2's region of 128 channel rows)
                        constexpr bool s1 = kP2S1;
                        float *pt = scratch + (s1 ? ((u >> 1) * 128 + L) * kPitch
                                                  : (u * 2 + slot) * 64 * kPitch + ((qd & 1) * 32 + lane) * kPitch);
#pragma unroll
                        for (int kc = 0; kc < kKC; ++kc) {
                            uint64_t v2[8];
#pragma unroll
                            for (int p = 0; p < 8; ++p) v2[p] = pack2(f[kc].r[2 * p], f[kc].r[2 * p + 1]);
                            const int pw0 = (hc + 2 * kc) * 8;  // this chunk's first window
#pragma unroll
                            for (int wi = 0; wi < 8; ++wi) {
                                const float2 a01 = unpack2(v2[wi]);
                                const float m = fmaxf(a01.x, a01.y);
                                if (pw0 + wi < kPitch - 1) pt[pw0 + wi] = s1 && (u & 1) ? fmaxf(pt[pw0 + wi], m) : m;
                            }
                            if (kc >= kMask0) {  // columns >= Wo add nothing to the sums
#pragma unroll
                                for (int p = 0; p < 8; ++p) {
                                    const uint32_t b0 = 1u << (16 * (kc - kMask0) + 2 * p);
                                    const float2 w = unpack2(v2[p]);
                                    v2[p] = pack2(__float_as_uint((gn_rag & b0) ? w.x : 0.0f),
                                                  __float_as_uint((gn_rag & (b0 << 1)) ? w.y : 0.0f));
                                }
                            }
#pragma unroll
                            for (int p = 0; p < 8; ++p) {
                                ls2[p & 1] = add2u(ls2[p & 1], v2[p]);
                                lss2[p & 1] = fma2u(v2[p], v2[p], lss2[p & 1]);
                            }
                        }
                    }
                }
            } else
            for (int u = 0; u < a.U; ++u) {
                const bool row_ok = r0 + u * a.S + slot < a.Ho;  // the same for the whole warp
                gn_rows += row_ok ? 1 : 0;
                Frag16 f[kKC];
#pragma unroll
                for (int kc = 0; kc < kKC; ++kc)
                    if (hc + 2 * kc < nchunks) tmem_ld16_issue(tbase + u * a.ucol + (hc + 2 * kc) * 16, f[kc]);
                tmem_ld_wait2(f[0], f[1]);
                if constexpr (kKC == 4) tmem_ld_wait2(f[2], f[3]);
                if (row_ok) {
                    // this u's rows belong to band u / 2 (two row slots per
                    // u; without stacking, the four u are the one band)
                    if constexpr (kNB == 2) {
                        if (u >= 2 && (!kGnX || a.S == 2)) gn_step(f, pext1);
                        else gn_step(f, pext0);
                    } else {
                        gn_step(f, pext0);
                    }
                }
            }
        } else {
        for (int u = 0; u < a.U; ++u) {
            const int row = r0 + u * a.S + slot;  // the same for the whole warp
            if constexpr (kMin) {
                // 64-column batches: the warp takes batches hc, hc + 2, ...,
                // loads a batch's four 16-column fragments with one wait and
                // reduces each fragment's own four channels in registers;
                // then the next batch's loads go out, and the butterflies and
                // stores of this batch run while they are in flight
                const uint32_t tb = tbase + u * a.ucol;
                const int nbt = (nchunks + 3) >> 2;
                float *srow = scratch + (u * 4 + qd) * a.P;
                auto load = [&](int q, Frag16 &f0, Frag16 &f1, Frag16 &f2, Frag16 &f3) {
                    const int c0 = 4 * q;
                    tmem_ld16_rows4_issue(tb + c0 * 16, f0);
                    if (c0 + 1 < nchunks) tmem_ld16_rows4_issue(tb + (c0 + 1) * 16, f1);
                    if (c0 + 2 < nchunks) tmem_ld16_rows4_issue(tb + (c0 + 2) * 16, f2);
                    if (c0 + 3 < nchunks) tmem_ld16_rows4_issue(tb + (c0 + 3) * 16, f3);
                };
                int q = hc;
                Frag16 f0, f1, f2, f3;
                if (q < nbt) load(q, f0, f1, f2, f3);
                if (u == 0) {
                    // the previous unit's combine runs while these loads are
                    // in flight (its partials were made visible by the barrier
                    // at the top of this unit); the barrier after it keeps this
                    // unit's partial stores behind every thread's reads
                    if (prev_n >= 0) combine_min(prev_n, prev_r0, prev_c0);
                    epi_bar();
                }
                if (q < nbt) {
                    tmem_ld_wait2(f0, f1);
                    tmem_ld_wait2(f2, f3);
                    float4 c0 = colmin16_own(f0, ss, sb2), c1 = colmin16_own(f1, ss, sb2);
                    float4 c2 = colmin16_own(f2, ss, sb2), c3 = colmin16_own(f3, ss, sb2);
                    for (;;) {
                        const bool more = q + 2 < nbt;
                        if (more) load(q + 2, f0, f1, f2, f3);
                        const int col = 64 * q;
                        const float m0 = colmin16_lanes(c0, lane), m1 = colmin16_lanes(c1, lane);
                        const float m2 = colmin16_lanes(c2, lane), m3 = colmin16_lanes(c3, lane);
                        if ((lane & 4) == 0) {
                            srow[colmin16_col(col, lane)] = m0;
                            if (4 * q + 1 < nchunks) srow[colmin16_col(col + 16, lane)] = m1;
                            if (4 * q + 2 < nchunks) srow[colmin16_col(col + 32, lane)] = m2;
                            if (4 * q + 3 < nchunks) srow[colmin16_col(col + 48, lane)] = m3;
                        }
                        if (!more) break;
                        q += 2;
                        tmem_ld_wait2(f0, f1);
                        tmem_ld_wait2(f2, f3);
                        c0 = colmin16_own(f0, ss, sb2), c1 = colmin16_own(f1, ss, sb2);
                        c2 = colmin16_own(f2, ss, sb2), c3 = colmin16_own(f3, ss, sb2);
                    }
                }
            } else {
                // 16-column chunks cc = hc, hc + 2, ...: the load of the next
                // chunk is in flight while this one is processed
                const bool row_ok = row < a.Ho;
                const size_t rowoff = (size_t)(row_ok ? row : 0) * a.Wo + c0;
                float *o4 = a.out + ((size_t)n * a.Co + cbase + cb4) * plane + rowoff + 4 * (lane & 3);
                float *o2 = a.out + ((size_t)n * a.Co + cbase + cb2) * plane + rowoff + 2 * (lane & 7);
                // 16-byte stores when every lane's row start is 16-byte aligned
                const bool v4 = __all_sync(0xffffffffu, (reinterpret_cast<uintptr_t>(o4) & 15u) == 0);
                const int wv = GENERAL ? min(a.CW, a.Wo - c0) : a.Wo;  // the column tile's output columns
                const uint32_t tb = tbase + u * a.ucol;
                int cc = hc;
                Frag16 cur, nxt;
                if (cc < nchunks) {
                    tmem_ld16_issue(tb + cc * 16, cur);
                    tmem_ld_wait(cur);
                }
                for (; cc < nchunks; cc += 2) {
                    const bool more = cc + 2 < nchunks;
                    if (more) tmem_ld16_issue(tb + (cc + 2) * 16, nxt);
                    epi_chunk_chan<KIND>(a, cur, bias, mult, lane, qd, ew, row_ok, v4, cc * 16, o4, o2, plane, wv,
                                         a.Co - cbase, scratch, ys, yss);
                    if (more) {
                        tmem_ld_wait(nxt);
                        cur = nxt;
                    }
                }
            }
        }
        }
        if (gn_quit) break;
        // tensor memory of this unit is no longer needed
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.acc_empty(ab));
        if constexpr (KIND == kKindConvStats) {
            // (image, unit, column group hc, accumulator row L): coalesced float pairs
            // (the buffer comes in gn.pmax: [n][unit][hc][L] float pairs)
            reinterpret_cast<float2 *>(a.gn.pmax)[(((size_t)n * a.units_per_img + ru) * 2 + hc) * 128 + L] =
                make_float2(ys, yss);
        }

        if constexpr (kMin) {
            // this unit's partial minima are in scratch; they are combined
            // during the next unit's first tensor-memory loads (or after the
            // loop, for the last unit)
            prev_n = n, prev_r0 = r0, prev_c0 = c0;
        } else if constexpr (kGN) {
            // group partial sums: lanes of one group (cw = min(cpg, 32) adjacent
            // channels) add by shuffles, the rest folds below in a fixed order
            // the sums are of v = gsg * (y - b) over cnt values: back to y,
            // sum y = gsg sum v + cnt b, sum y^2 = sum v^2 + 2 b gsg sum v + cnt b^2
            const float2 l0 = unpack2(ls2[0]), l1 = unpack2(ls2[1]), q0 = unpack2(lss2[0]), q1 = unpack2(lss2[1]);
            const float sv = gsg * ((l0.x + l0.y) + (l1.x + l1.y)), svv = (q0.x + q0.y) + (q1.x + q1.y);
            const float cnt = (float)(gn_ncol * gn_rows);
            float gs = fmaf(cnt, bias, sv), gss = fmaf(2.0f * bias, sv, fmaf(cnt * bias, bias, svv));
            for (int o = 1; o < gn_cw; o <<= 1) {
                gs += __shfl_xor_sync(0xffffffffu, gs, o);
                gss += __shfl_xor_sync(0xffffffffu, gss, o);
            }
            // pooled tiles [band][2 row slots][64 channels][kPoolPitch] (window
            // extremes in gsg space); both slots write, one barrier, and the
            // stores fold the two slots
            // every warp is past the previous unit's tile and statistics reads
            // (and none has given up) before they are rewritten
            if (!kWide && !kPool2 && !kWideP2 && epi_bar_any(false)) break;  // (wide rows, 2 x 2 windows: voted before their first tile)
            // channel tiles: the sign and bias tables of this unit's tile (the
            // vote above ends the previous unit's reads of them)
            if (kTiles && MT > 1) gn_sgn[co] = gsg, gn_bias[co] = bias;
            float *st = scratch + kNB * 2 * 64 * kPitch;  // [2 stats][8 warps][32 lanes]
            st[ew * 32 + lane] = gs;
            st[kEpiThreads + ew * 32 + lane] = gss;
            // channel within the tile: two row slots of 64 channels, or (no
            // stacking) one slot of 128 spanning both slots' space
            const int cl = kGnX && a.S == 1 ? L : (qd & 1) * 32 + lane;
            auto put_tile = [&](int band, const float (&pext)[kWin]) {
                float *pt = scratch + (band * 2 + slot) * 64 * kPoolPitch;
#pragma unroll
                for (int k = 0; k < kWin; ++k) {
                    const int pw = (hc + 2 * (k / 4)) * 4 + (k % 4);
                    if (pw < 32) pt[cl * kPoolPitch + pw] = pext[k];
                }
            };
            if constexpr (!kWide && !kPool2 && !kWideP2) {
                put_tile(0, pext0);
                if constexpr (kNB == 2) {
                    if (!kGnX || a.S == 2) put_tile(1, pext1);
                }
            }
            epi_bar();
            if (ew == 2) {
                // one warp (the others go on to the band stores): per group,
                // the shuffled sums from both row slots, both column groups
                // and (cpg = 64: two lane groups) both halves, loaded together
                // and added in a fixed order, stored as a float pair.  (Spread
                // over all eight warps this fold measured slower: every
                // warp's tail then waits on it.)
                const int nci = gn_cpg / gn_cw;  // 1, or 2 when a group spans two warps' lanes
                float *fpart = reinterpret_cast<float *>(a.gn.part);
                for (int g = lane; g < a.groups; g += 32) {
                    // (channel tiles: the groups of other tiles get zero sums from this unit)
                    const int lc = g * gn_cpg - cbase;
                    const bool in_tile = !kTiles || (lc >= 0 && lc < a.Cout);
                    float v0[8], v1[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {  // k = (row slot, column group, half)
                        const int sl = k >> 2, h2 = (k >> 1) & 1, ci = k & 1;
                        v0[k] = v1[k] = 0.0f;
                        if (in_tile && ci < nci && (!kGnX || sl < a.S)) {
                            const int LL = sl * a.Cout + lc + ci * gn_cw;
                            const int e2 = h2 * 4 + (LL >> 5);
                            v0[k] = st[e2 * 32 + (LL & 31)];
                            v1[k] = st[kEpiThreads + e2 * 32 + (LL & 31)];
                        }
                    }
                    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if ((k & 1) < nci && (!kGnX || (k >> 2) < a.S)) s0 += v0[k], s1 += v1[k];
                    *reinterpret_cast<float2 *>(fpart + (((size_t)n * a.units_per_img + ru) * a.groups + g) * 2) =
                        make_float2(s0, s1);
                }
            }
            if constexpr (kPool2) {
                // the unit's bands: one (no stacking: rb, its channels' rows
                // of the tile already both rows' maxima) or two (2 ru and
                // 2 ru + 1, each the two row slots folded); sign and bias
                // restored; windows lane and lane + 32, channels ew + 8 i
                constexpr bool s1 = kP2S1;
                // (no stacking: one band per unit, or two in the four-u form)
                constexpr int nbnd = s1 ? (GENERAL ? 2 : 1) : kNB, nch = s1 ? 128 / kEpiWarps : 64 / kEpiWarps;
#pragma unroll
                for (int band = 0; band < nbnd; ++band) {
                    const int prow = (s1 ? rb : ru) * nbnd + band;
                    if (prow < a.Hp) {
                        const float *pt0 = scratch + band * 2 * 64 * kPitch, *pt1 = pt0 + 64 * kPitch;
                        float *dst = a.gn.pmax + (((size_t)n * a.Co + ew) * a.Hp + prow) * a.Wp;
                        const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
#pragma unroll
                        for (int hw = 0; hw < 2; ++hw) {
                            const int w = lane + 32 * hw;
                            if (w >= a.Wp) continue;
                            // (8 channels at a time: all their tile reads before the stores)
#pragma unroll
                            for (int i0 = 0; i0 < nch; i0 += 8) {
                                float m[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int c2 = ew + kEpiWarps * (i0 + i);
                                    const float v =
                                        s1 ? pt0[c2 * kPitch + w] : fmaxf(pt0[c2 * kPitch + w], pt1[c2 * kPitch + w]);
                                    m[i] = fmaf(gn_sgn[c2], v, gn_bias[c2]);
                                }
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    if (ew + kEpiWarps * (i0 + i) < a.Co) dst[(i0 + i) * cstep + w] = m[i];
                            }
                        }
                    }
                }
            } else if constexpr (kWideP2) {
                // the unit's one band rb, the two row slots folded, sign and
                // bias restored; windows lane + 32 hw (up to 127)
                const int prow = rb;
                if (prow < a.Hp) {
                    const float *pt0 = scratch, *pt1 = scratch + 64 * kPitch;
                    float *dst = a.gn.pmax + (((size_t)n * a.Co + ew) * a.Hp + prow) * a.Wp;
                    const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
#pragma unroll
                    for (int hw = 0; hw < 4; ++hw) {
                        const int w = lane + 32 * hw;
                        if (w >= a.Wp) continue;
                        float m[64 / kEpiWarps];
#pragma unroll
                        for (int i = 0; i < 64 / kEpiWarps; ++i) {
                            const int c2 = ew + kEpiWarps * i;
                            m[i] = fmaf(gn_sgn[c2], fmaxf(pt0[c2 * kPitch + w], pt1[c2 * kPitch + w]), gn_bias[c2]);
                        }
#pragma unroll
                        for (int i = 0; i < 64 / kEpiWarps; ++i)
                            if (ew + kEpiWarps * i < a.Co) dst[i * cstep + w] = m[i];
                    }
                }
            } else if constexpr (kWideS1) {
                // quarter rb & 3 of band rb / 4 (sign and bias restored) into
                // slot rb & 3; windows lane and lane + 32, channels ew + 8 i
                const int prow = rb >> 2, q = rb & 3;
                if (prow < a.Hp) {
                    float *slot_base = q == 0   ? a.gn.pmax
                                       : q == 1 ? a.gn.pmin
                                       : q == 2 ? reinterpret_cast<float *>(a.gn.amax)
                                                : reinterpret_cast<float *>(a.gn.amin);
                    float *dst = slot_base + (((size_t)n * a.Co + ew) * a.Hp + prow) * a.Wp;
                    const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
#pragma unroll
                    for (int hw = 0; hw < 2; ++hw) {
                        const int w = lane + 32 * hw;
                        if (w >= a.Wp) continue;
#pragma unroll
                        for (int i0 = 0; i0 < 128 / kEpiWarps; i0 += 8) {
                            float m[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int c2 = ew + kEpiWarps * (i0 + i);
                                m[i] = fmaf(gn_sgn[c2], scratch[c2 * kPitch + w], gn_bias[c2]);
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                if (ew + kEpiWarps * (i0 + i) < a.Co) dst[(i0 + i) * cstep + w] = m[i];
                        }
                    }
                }
            } else if constexpr (kWide) {
                // half band rb / 2, two row slots folded, sign and bias
                // restored, into slot rb & 1; windows lane and lane + 32 (of
                // the column tile's, which start at window c0 / 4)
                const int prow = rb >> 1;
                const int w0 = kColT ? c0 / 4 : 0, nw = kColT ? min(a.CW / 4, a.Wp - w0) : a.Wp;
                if (prow < a.Hp) {
                    const float *pt0 = scratch, *pt1 = scratch + 64 * kPitch;
                    float *dst = ((rb & 1) ? a.gn.pmin : a.gn.pmax) + (((size_t)n * a.Co + ew) * a.Hp + prow) * a.Wp + w0;
                    const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
#pragma unroll
                    for (int hw = 0; hw < 2; ++hw) {
                        const int w = lane + 32 * hw;
                        if (w >= nw) continue;
                        float m[64 / kEpiWarps];
#pragma unroll
                        for (int i = 0; i < 64 / kEpiWarps; ++i) {
                            const int c2 = ew + kEpiWarps * i;
                            m[i] = fmaf(gn_sgn[c2], fmaxf(pt0[c2 * kPitch + w], pt1[c2 * kPitch + w]), gn_bias[c2]);
                        }
#pragma unroll
                        for (int i = 0; i < 64 / kEpiWarps; ++i)
                            if (ew + kEpiWarps * i < a.Co) dst[i * cstep + w] = m[i];
                    }
                }
            } else
            if (kGnX && !GENERAL && a.S == 1) {
                // no stacking: this unit's 2 rows are half of band rb / 2; its
                // extremes (sign and bias restored: the half's selected y) go
                // to slot rb & 1, and the finalize folds the two halves
                // (channels cbase + ...: the unit's channel tile)
                const int prow = rb >> 1;
                if (prow < a.Hp && lane < a.Wp) {
                    float *dst = ((rb & 1) ? a.gn.pmin : a.gn.pmax) +
                                 (((size_t)n * a.Co + cbase + ew) * a.Hp + prow) * a.Wp + lane;
                    const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
                    float m[128 / kEpiWarps];
#pragma unroll
                    for (int i = 0; i < 128 / kEpiWarps; ++i) {
                        const int c2 = ew + kEpiWarps * i;
                        m[i] = fmaf(gn_sgn[c2], scratch[c2 * kPoolPitch + lane], gn_bias[c2]);
                    }
#pragma unroll
                    for (int i = 0; i < 128 / kEpiWarps; ++i)
                        if (cbase + ew + kEpiWarps * i < a.Co) dst[i * cstep] = m[i];
                }
            } else if (kGnX && GENERAL && a.S == 1) {
                // no stacking, rows of up to 64 columns: the unit's four u
                // are one whole band, each thread's extremes over all four
                // rows in the one tile of 128 channels; warp ew stores
                // channels cbase + ew, cbase + ew + 8, ..., sign and bias
                // restored
                const int prow = rb;
                if (prow < a.Hp && lane < a.Wp) {
                    float *dst = a.gn.pmax + (((size_t)n * a.Co + cbase + ew) * a.Hp + prow) * a.Wp + lane;
                    const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
                    float m[128 / kEpiWarps];
#pragma unroll
                    for (int i = 0; i < 128 / kEpiWarps; ++i) {
                        const int c2 = ew + kEpiWarps * i;
                        m[i] = fmaf(gn_sgn[c2], scratch[c2 * kPoolPitch + lane], gn_bias[c2]);
                    }
#pragma unroll
                    for (int i = 0; i < 128 / kEpiWarps; ++i)
                        if (cbase + ew + kEpiWarps * i < a.Co) dst[i * cstep] = m[i];
                }
            } else
#pragma unroll
            for (int band = 0; band < kNB; ++band) {
                const int prow = ru * kNB + band;  // pooled row of this band
                if (prow < a.Hp && lane < a.Wp) {
                    // warp ew stores channels ew, ew + 8, ..., ew + 56: one
                    // pooled row each (Wp <= 32), the two row slots folded and
                    // the sign restored; all sixteen tile reads go out before
                    // the stores
                    const float *pt0 = scratch + band * 2 * 64 * kPoolPitch, *pt1 = pt0 + 64 * kPoolPitch;
                    float *dst = a.gn.pmax + (((size_t)n * (kGnX ? a.Co : a.Cout) + ew) * a.Hp + prow) * a.Wp + lane;
                    const size_t cstep = (size_t)kEpiWarps * a.Hp * a.Wp;
                    float m[64 / kEpiWarps];
#pragma unroll
                    for (int i = 0; i < 64 / kEpiWarps; ++i) {
                        const int c2 = ew + kEpiWarps * i;
                        m[i] = fmaf(gn_sgn[c2], fmaxf(pt0[c2 * kPoolPitch + lane], pt1[c2 * kPoolPitch + lane]),
                                    gn_bias[c2]);
                    }
#pragma unroll
                    for (int i = 0; i < 64 / kEpiWarps; ++i)
                        if (!kGnX || ew + kEpiWarps * i < a.Co) dst[i * cstep] = m[i];
                }
            }
            // (the vote of the next unit keeps the tile until all stores have read it)
        }
    }
    if constexpr (kMin) {
        if (prev_n >= 0) {  // the last unit's combine
            epi_bar();
            combine_min(prev_n, prev_r0, prev_c0);
        }
    }
}

// In-kernel GroupNorm finalize (launched cooperatively, so every CTA is
// resident and a grid-wide arrival count is safe to wait on).  After every
// CTA has stored its units' partial sums and pooled extremes and released
// tensor memory, CTA b takes the (image, group) pairs b, b + gridDim.x, ...
// Thread 0 bulk-copies their pooled blocks (contiguous, F4 float4 each) into
// the (now free) shared memory, while one warp per pair folds its
// statistics and its channels' coefficients; every thread then applies
// z = clamp(A y + B) in place, and thread 0 bulk-copies the blocks out to
// the output.  The blocks take the shared memory from kFinBufOff up to the
// main loop's barriers and flags, which sit at the end of the layout (a
// variant whose blocks lay over them lost 8 bytes of a block between the
// apply and the copy out).  The copies keep whole blocks in flight, where
// per-thread loads left the pass latency-bound.  The page-shape kernel takes the pairs
// in batches of up to one per warp, as many as shared memory holds (for its
// 15 KB blocks, nearly all of a CTA's pairs at once).  The generalised
// kinds, whose blocks are up to four times larger, run a ring of pair slots
// instead: the copy of pair k + cap goes out as soon as pair k's block has
// been copied out, so later pairs' loads overlap earlier pairs' apply and
// stores (x[128,8,128,128] with 2x2 windows 235 -> 203 us, Cout 128
// 236 -> 222; the ring measured 5 us slower for the page shape's small
// blocks, and rounds of several pairs slower for both).
constexpr int kFinPairs = kThreads / 32;
constexpr uint32_t kFinFlagOff = kFinPairs * 64 * 2 * 4;  // after the coefficient tables
constexpr uint32_t kFinBarOff = kFinFlagOff + 8;         // an mbarrier per batch (or per ring slot)
constexpr uint32_t kFinBufOff = 8448;                     // the pooled blocks (128-byte aligned)
static_assert(kFinBarOff + 8u * kFinPairs <= kFinBufOff, "finalize barriers overlap the pooled blocks");
// kSl: the parts a band's pooled blocks may come in: 2 where a unit of 2
// rows holds half a 4-row band (65..128 channels, or rows of 127 or more
// columns), 4 where a unit of 1 row holds a quarter (65..128 channels on
// rows of 130..256 columns), else 1
template <bool kGnX, int kSl>
__device__ __forceinline__ void gn_finalize_tail(const Cfg &a, uint8_t *smem, volatile int *abort_flag) {
    float *sA = reinterpret_cast<float *>(smem), *sB = sA + kFinPairs * 64;
    int &s_go = *reinterpret_cast<int *>(smem + kFinFlagOff);
    const uint32_t fbar = smem_u32(smem + kFinBarOff);
    float4 *buf = reinterpret_cast<float4 *>(smem + kFinBufOff);
    __threadfence();  // this CTA's partials and pooled extremes, device-wide
    fence_proxy_async_smem();  // this thread's earlier shared-memory accesses before the copies' writes
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_init(fbar, 1);
        fence_mbar_init();
        atomicAdd(a.gn.arrive, 1u);
        int go = 1;
        const uint64_t t0 = globaltimer();
        for (;;) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.gn.arrive) : "memory");
            if (v >= gridDim.x) break;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicOr(a.err, ERRBIT_TIMEOUT);
                go = 0;
                break;
            }
            __nanosleep(256);
        }
        __threadfence();
        // the other CTAs' pooled extremes (generic stores, acquired above)
        // are read below by bulk copies: order them for the async proxy too
        asm volatile("fence.proxy.async.global;" ::: "memory");
        s_go = go && !*abort_flag;
    }
    __syncthreads();
    if (!s_go) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cpg = (kGnX ? a.Co : a.Cout) / a.groups;
    const uint32_t F4 = (uint32_t)cpg * (uint32_t)(a.Hp * a.Wp) / 4u, pbytes = F4 * 16u;
    const int npairs = a.N * a.groups;
    // (with half bands, a pair's two slots side by side: [pair][slot][F4])
    // (a unit of 2 rows holds half a band: 65..128 channels, or rows of 130..256 columns)
    const uint32_t nsl = kSl == 4 ? 4u : kGnX && kSl == 2 && a.RU == 2 ? 2u : 1u, sbytes = nsl * pbytes;
    // slot h of a pair's pooled block: pmax, pmin and the index buffers
    auto slot_src = [&](uint32_t h) -> const char * {
        return reinterpret_cast<const char *>(h == 0   ? a.gn.pmax
                                              : h == 1 ? a.gn.pmin
                                              : h == 2 ? reinterpret_cast<const float *>(a.gn.amax)
                                                       : reinterpret_cast<const float *>(a.gn.amin));
    };
    if constexpr (kGnX) {
        // this CTA's pairs p = blockIdx.x + k * gridDim.x (k < K) through a ring
        // of cap slots: pair k lands in slot k % cap, and the copy of pair
        // k + cap goes out as soon as pair k's block has been copied out of it.
        const int cap = min(kFinPairs, (int)((a.bar_off - kFinBufOff) / sbytes));  // >= 1: checked on the host
        const int K = npairs > (int)blockIdx.x ? (npairs - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
        auto issue = [&](int k) {
            const int sl = k % cap;
            const size_t p = (size_t)blockIdx.x + (size_t)k * gridDim.x;
            mbar_arrive_expect_tx(fbar + 8u * (uint32_t)sl, sbytes);
            for (uint32_t h = 0; h < nsl; ++h) {
                const char *src = slot_src(h) + p * pbytes;
                const uint32_t dsm = smem_u32(buf) + (uint32_t)sl * sbytes + h * pbytes;
                for (uint32_t off = 0; off < pbytes; off += 16384u)
                    bulk_g2s(dsm + off, src + off, min(16384u, pbytes - off), fbar + 8u * (uint32_t)sl);
            }
        };
        if (threadIdx.x == 0) {
            for (int sl = 1; sl < cap; ++sl) mbar_init(fbar + 8u * (uint32_t)sl, 1);  // (slot 0's is set up above)
            fence_mbar_init();
            for (int k = 0; k < min(cap, K); ++k) issue(k);
        }
        uint32_t phases = 0;  // bit sl: the parity of slot sl's next completion
        for (int k = 0; k < K; ++k) {
            if (k % kFinPairs == 0) {
                // the coefficients of pairs k .. k + kFinPairs - 1, one warp per
                // pair, while their copies are in flight
                __syncthreads();  // (the barriers are set up; the tables' previous readers are done)
                const int kk = k + warp;
                if (kk < K) {
                    const int p = (int)blockIdx.x + kk * (int)gridDim.x;
                    const int n = p / a.groups, g = p % a.groups;
                    float mean, rstd;
                    gn_group_stats_f(reinterpret_cast<const float *>(a.gn.part), a.units_per_img, a.groups, n, g, a.cnt,
                                     a.eps, mean, rstd);
                    for (int cl = lane; cl < cpg; cl += 32) {
                        const int c = g * cpg + cl;
                        gn_coeffs(__ldg(&a.gamma[c]), __ldg(&a.beta[c]), __ldg(&a.chan_scale[c]), mean, rstd,
                                  sA[warp * 64 + cl], sB[warp * 64 + cl]);
                    }
                }
            }
            const int sl = k % cap;
            const bool landed = wait_bar(fbar + 8u * (uint32_t)sl, (phases >> sl) & 1u, abort_flag, a.err, false);
            phases ^= 1u << sl;
            if (__syncthreads_or(!landed)) return;  // (also publishes the coefficients)
            const float *cA = sA + (k % kFinPairs) * 64, *cB = sB + (k % kFinPairs) * 64;
            float4 *bp0 = buf + (uint32_t)sl * nsl * F4;
            for (uint32_t t = threadIdx.x; t < F4; t += kThreads) {
                const uint32_t e = 4u * t;
                float4 *bp = bp0 + t;
                const float4 v = bp[0];
                float r[4] = {v.x, v.y, v.z, v.w};
                for (uint32_t h = 1; h < nsl; ++h) {
                    // the band's extreme from its parts: the larger y where
                    // the slope A is >= 0, else the smaller
                    const float4 w = bp[h * F4];
                    const float h2[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t cl = __umulhi(e + q, a.per_magic);
                        r[q] = cA[cl] >= 0.0f ? fmaxf(r[q], h2[q]) : fminf(r[q], h2[q]);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t cl = __umulhi(e + q, a.per_magic);  // channel within the group
                    r[q] = fminf(fmaxf(fmaf(cA[cl], r[q], cB[cl]), a.lo), a.hi);
                }
                bp[0] = make_float4(r[0], r[1], r[2], r[3]);
            }
            fence_proxy_async_smem();  // these writes before the copy's reads
            __syncthreads();
            if (threadIdx.x == 0) {
                char *dst = reinterpret_cast<char *>(a.out) + ((size_t)blockIdx.x + (size_t)k * gridDim.x) * pbytes;
                for (uint32_t off = 0; off < pbytes; off += 16384u)
                    bulk_s2g(dst + off, smem_u32(buf) + (uint32_t)sl * sbytes + off, min(16384u, pbytes - off));
                bulk_commit();
                bulk_wait_read();  // slot sl is copied out: pair k + cap (or the exit) may reuse it
                if (k + cap < K) issue(k + cap);
            }
        }
    } else {
        const int cap = min(kFinPairs, (int)((a.bar_off - kFinBufOff) / sbytes));  // >= 1: checked on the host
        uint32_t phase = 0;
        for (int p0 = blockIdx.x; p0 < npairs; p0 += (int)gridDim.x * cap) {
            const int nbp = min(cap, (npairs - p0 + (int)gridDim.x - 1) / (int)gridDim.x);  // pairs in this batch
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(fbar, (uint32_t)nbp * sbytes);
                for (int j = 0; j < nbp; ++j)
                    for (uint32_t sl = 0; sl < nsl; ++sl) {
                        const char *src = reinterpret_cast<const char *>(sl ? a.gn.pmin : a.gn.pmax) +
                                          (size_t)(p0 + j * (int)gridDim.x) * pbytes;
                        const uint32_t dsm = smem_u32(buf) + (uint32_t)j * sbytes + sl * pbytes;
                        for (uint32_t off = 0; off < pbytes; off += 16384u)
                            bulk_g2s(dsm + off, src + off, min(16384u, pbytes - off), fbar);
                    }
            }
            const int p = p0 + warp * (int)gridDim.x;
            if (warp < nbp) {
                const int n = p / a.groups, g = p % a.groups;
                float mean, rstd;
                gn_group_stats_f(reinterpret_cast<const float *>(a.gn.part), a.units_per_img, a.groups, n, g, a.cnt,
                                 a.eps, mean, rstd);
                for (int cl = lane; cl < cpg; cl += 32) {
                    const int c = g * cpg + cl;
                    gn_coeffs(__ldg(&a.gamma[c]), __ldg(&a.beta[c]), __ldg(&a.chan_scale[c]), mean, rstd,
                              sA[warp * 64 + cl], sB[warp * 64 + cl]);
                }
            }
            const bool landed = wait_bar(fbar, phase, abort_flag, a.err, false);
            phase ^= 1u;
            if (__syncthreads_or(!landed)) return;  // (also publishes the coefficients)
            const uint32_t total = (uint32_t)nbp * F4;
            for (uint32_t t = threadIdx.x; t < total; t += kThreads) {
                const uint32_t jb = __umulhi(t, a.f4_magic);  // t / F4: the pair within the batch
                const float *cA = sA + jb * 64, *cB = sB + jb * 64;
                const uint32_t fo = t - jb * F4, e = 4u * fo;
                float4 *bp = buf + jb * nsl * F4 + fo;
                const float4 v = bp[0];
                float r[4] = {v.x, v.y, v.z, v.w};
                if (kGnX && nsl == 2) {
                    // the band's extreme from its two halves: the larger y where
                    // the slope A is >= 0, else the smaller
                    const float4 w = bp[F4];
                    const float h2[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t cl = __umulhi(e + q, a.per_magic);
                        r[q] = cA[cl] >= 0.0f ? fmaxf(r[q], h2[q]) : fminf(r[q], h2[q]);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t cl = __umulhi(e + q, a.per_magic);  // channel within the group
                    r[q] = fminf(fmaxf(fmaf(cA[cl], r[q], cB[cl]), a.lo), a.hi);
                }
                bp[0] = make_float4(r[0], r[1], r[2], r[3]);
            }
            fence_proxy_async_smem();  // these writes before the copies' reads
            __syncthreads();
            if (threadIdx.x == 0) {
                for (int j = 0; j < nbp; ++j) {
                    char *dst = reinterpret_cast<char *>(a.out) + (size_t)(p0 + j * (int)gridDim.x) * pbytes;
                    for (uint32_t off = 0; off < pbytes; off += 16384u)
                        bulk_s2g(dst + off, smem_u32(buf) + (uint32_t)j * sbytes + off, min(16384u, pbytes - off));
                }
                bulk_commit();
                bulk_wait_read();  // the buffer is read: the next batch (or the exit) may reuse it
            }
            __syncthreads();  // (and the next batch rewrites the coefficients)
        }
    }
}

template <int KIND, bool GENERAL>
__global__ void __launch_bounds__(kThreads, 1) tc_conv_epi(const __grid_constant__ TcArgs args) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Cfg a = args.c;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    Bars bars;
    bars.base = sbase + a.bar_off;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + a.bar_off + 8 * Bars::kCount);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *scratch = reinterpret_cast<float *>(smem + a.scratch_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxRing; ++s) {
            mbar_init(bars.a_full(s), 1);
            mbar_init(bars.a_empty(s), 1);
            mbar_init(bars.b_full(s), a.nhwc ? 1 : kConvWarps);  // NHWC: the producer's transaction arrive
            mbar_init(bars.b_empty(s), 1);
            mbar_init(bars.r_full(s), 1);
            mbar_init(bars.r_empty(s), kConvWarps);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(bars.acc_full(ab), 1);
            mbar_init(bars.acc_empty(ab), kEpiWarps);
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
    // A CTA that allocates all 512 columns owns the whole tensor memory, so the
    // allocation starts at lane 0, column 0: the roles use that constant base
    // (uniform, no per-thread copy of the loaded address).  Any other answer
    // is reported and the CTA does no work.
    constexpr uint32_t tmem = 0;
    const bool tmem_ok = *tmem_slot == tmem;
    if (!tmem_ok && threadIdx.x == 0) atomicOr(a.err, ERRBIT_TMEM);
    grid_dep_wait();

    if (!tmem_ok) {
        // nothing issued, nothing to drain
    } else if (warp == 0) {
        if (lane == 0) mma_role(a, sbase, bars, tmem, abort_flag);
        __syncwarp();
    } else if (warp == kProducerWarp) {
        if (lane == 0)
            producer_role<GENERAL, KIND == kKindGnTiles || KIND == kKindGnColTiles>(a, &args.xmap, sbase, bars,
                                                                                   abort_flag);
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        converter_role(a, smem, bars, abort_flag);
    } else {
        epilogue_role<KIND, GENERAL>(a, scratch, bars, tmem, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, kTmemCols);
    }
    if constexpr (is_gn(KIND)) {
        if (a.gn_fin)
            gn_finalize_tail<is_gnx(KIND), KIND == kKindGnWideS1 ? 4 : KIND != kKindGnPool2S1 && KIND != kKindGnWideP2 ? 2 : 1>(
                a, smem, abort_flag);
    }
}

// ------------------------------------------------------ filter packing ----
// wpack[c][kw][jg][p][co][e] = tf32(w[co][8c + 4jg + e][kh][kw]) with
// kh = S+1-p when 0 <= kh <= 2, else 0 (the zero planes that pad the
// stacked row slots), 0 for output channels co >= Co (a problem Cout below the
// GEMM's 64 or 128, or the last channel tile's remainder, is padded with zero
// filters; one launch per channel tile), and 0 for input channels
// 8c + 4jg + e >= Cin (the last
// chunk of a Cin that is not a multiple of 8; the input tile's matching
// channels arrive as zeros too, from the tensor load's out-of-range fill).
// For the fused GroupNorm chain (gamma, scale given) filter co is negated
// where gamma[co] and scale[co] differ in sign, so the accumulator holds
// sgn * (y - b) with sgn the sign of the channel's affine slope (negation is
// exact, and tf32 rounding to nearest is symmetric).
__global__ void pack_weights(const float *__restrict__ w, float *__restrict__ wp, int Cin, int Cout, int Co, int S,
                             const float *__restrict__ gamma, const float *__restrict__ scale,
                             unsigned *__restrict__ reset) {
    grid_dep_launch();
    if (reset && blockIdx.x == 0 && threadIdx.x == 0) *reset = 0u;  // the conv kernel's grid-wide arrival count
    const int planes = 2 * S + 1;
    const int Cpad = (Cin + 7) / 8 * 8;
    const size_t total = (size_t)Cpad * 3 * planes * Cout;  // = chunks*3*2*planes*Cout*4
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
        const int ci = 8 * c + 4 * jg + e;
        if (kh >= 0 && kh <= 2 && ci < Cin && co < Co) {
            v = w[(((size_t)co * Cin + ci) * 3 + kh) * 3 + kw];
            if (gamma && signbit(__ldg(&gamma[co])) != signbit(__ldg(&scale[co]))) v = -v;
        }
        wp[i] = __uint_as_float(f32_to_tf32(v));
    }
}

// the min chains' output before channel tiles take their atomic minima
__global__ void fill_f32(float *__restrict__ p, size_t n, float v) {
    grid_dep_launch();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = v;
}

// x viewed as rows [rows][W] -> xp [rows][Wp] (Wp = W rounded up to 4): one
// warp per row at a time, consecutive lanes on consecutive floats.  The pad
// columns are left unwritten: the tensor map's row extent stays W, so the
// tensor load never reads them (it fills zeros past W).
__global__ void pad_rows(const float *__restrict__ x, float *__restrict__ xp, size_t rows, int W, int Wp) {
    grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const size_t warps = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t r = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const float *src = x + r * W;
        float *dst = xp + r * Wp;
        for (int c = lane; c < W; c += 32) dst[c] = __ldg(src + c);
    }
}

// ----------------------------------------------------------- planning ----
struct Plan {
    int S, P, U, RU, Rin, PL, chunks, ucol;
    int CT, CW, BW;  // column tiles, output columns per tile, staged tile width
    int MT;          // channel tiles
    int Cg;          // the GEMM's output channels per channel tile
    int resident, na, nb, nr;
    uint32_t a_bytes, b_bytes, raw_bytes, scratch_bytes;
    uint32_t a_off, b_off, raw_off, bar_off, scratch_off;
    size_t smem;
    // filter operand layout [chunk][kw][ci4][plane][co][4]: one plane, the
    // K-group (ci4) stride, the tap (kw) stride
    uint32_t a_plane_bytes, a_lbo, a_kw_stride;
    int xpitch;         // floats between input rows as the tensor load reads them
    uint32_t box[4];    // tensor-load box: NCHW (BW, Rin, 8, 1), NHWC (4, P, Rin, 1)
};

uint32_t scratch_bytes_for(int kind, int U, int P) {
    switch (kind) {
    case CONV_EPI_MIN_TANH2:
    case CONV_EPI_SCALE_MIN:
        return (uint32_t)(U * 4 * P * sizeof(float));
    case CONV_EPI_MUL_LRELU_GELU:
    case CONV_EPI_NONE:
    case kKindConvStats:
        return (uint32_t)(kEpiWarps * 32 * 16 * sizeof(float));  // a 32 x 16 staging tile per warp
    case CONV_EPI_GN_SCALE_POOL_CLAMP:  // U / 2 bands of pooled tiles, the statistics, the sign and bias tables
        return (uint32_t)(((U / 2) * 2 * 64 * kPoolPitch + 2 * kEpiThreads + 2 * 64) * sizeof(float));
    case kKindGnWideP2:  // one band region of pitch 129, the statistics, the tables
        return (uint32_t)((2 * 64 * 129 + 2 * kEpiThreads + 2 * 128) * sizeof(float));
    case kKindGnWide:  // one band region of pitch 65, the statistics, the tables
    case kKindGnColTiles:
    case kKindGnWideS1:
        return (uint32_t)((2 * 64 * 65 + 2 * kEpiThreads + 2 * 128) * sizeof(float));
    case kKindGnPool2:  // two band regions of pitch 65 (rows of up to 64 columns: four of pitch 33), the
    case kKindGnPool2S1:  // statistics, the tables
        return (uint32_t)(((U == 4 ? 4 * 2 * 64 * kPoolPitch : 2 * 2 * 64 * 65) + 2 * kEpiThreads + 2 * 128) *
                          sizeof(float));
    case kKindGnX:  // (the tables for up to 128 channels)
    case kKindGnXNarrow:
    case kKindGnTiles:
        return (uint32_t)(((U / 2) * 2 * 64 * kPoolPitch + 2 * kEpiThreads + 2 * 128) * sizeof(float));
    }
    return 0;
}

uint32_t up1k(uint32_t v) { return (v + 1023u) & ~1023u; }

// Shared memory: [filter: resident or ring][B ring][staged-tile ring][epilogue
// scratch][mbarriers, tmem slot, abort flag]
// the GEMM's output-channel count per channel tile: a problem Cout up to 64
// runs as 64 (two stacked row slots), larger ones as tiles of 128, with zero
// filters for the rest
int gemm_cout(int Cout) { return Cout <= 64 ? 64 : 128; }
// floats per row of the input the tensor load reads: W rounded up to whole
// 16-byte units (row strides of a tensor map are multiples of 16 bytes)
int row_pitch(int W) { return (W + 3) / 4 * 4; }
// NCHW input whose rows are not whole 16-byte units is first copied into
// rows of row_pitch(W) floats
bool needs_xpad(const conv_epi_desc &d) { return d.layout == CONV_EPI_LAYOUT_NCHW && d.W % 4 != 0; }
int channel_tiles(int Cout) { return Cout <= 128 ? 1 : (Cout + 127) / 128; }

bool make_plan(const conv_epi_desc &d, int kind, Plan &pl) {
    if (d.Cout < 1) return false;
    if (d.Cin < 1 || d.W < 3 || d.H < 3) return false;
    pl.MT = channel_tiles(d.Cout);
    // (channel tiles of the GroupNorm chain: the generalised kinds' half bands)
    if (pl.MT > 1 && is_gn(kind) && kind != kKindGnTiles) return false;
    const bool nhwc = d.layout == CONV_EPI_LAYOUT_NHWC;
    if (nhwc && d.Cin % 4 != 0) return false;  // 16-byte position stride
    const int Cg = gemm_cout(d.Cout);
    pl.S = 128 / Cg;
    if (d.W <= 256) {
        // one tile spans the row; the GroupNorm chain runs rows of up to 64
        // columns at P = 64 (four u per unit: two pooling bands)
        pl.P = (d.W + 15) / 16 * 16;
        if (is_gn(kind) && pl.P < 64) pl.P = 64;
        // (staged rows are whole 16-byte units: columns W..BW-1 arrive as zeros)
        pl.CT = 1, pl.CW = d.W - 2, pl.BW = row_pitch(d.W);
    } else {
        // column tiles of 252 outputs from 256 staged columns (the last two
        // unused; tiles start on multiples of 4 columns, 16-byte aligned);
        // past the image's right edge the tensor load fills zeros
        if (is_gn(kind) && kind != kKindGnColTiles) return false;
        pl.P = 256;
        pl.CW = 252, pl.BW = 256;
        pl.CT = (d.W - 2 + pl.CW - 1) / pl.CW;
    }
    pl.ucol = (pl.P + 31) / 32 * 32;
    pl.U = kAccStride / pl.ucol;
    pl.RU = pl.U * pl.S;
    pl.Rin = pl.RU + 2;
    if (pl.Rin > 256) return false;  // TMA box height
    pl.PL = (pl.Rin * pl.P + 4 + 7) / 8 * 8;
    pl.chunks = (d.Cin + 7) / 8;  // the last chunk of a Cin not a multiple of 8 is zero-padded
    if (pl.PL >= (1 << 16)) return false;
    if (!nhwc && 2 * pl.Rin * ((pl.P + 31) / 32) > kConvItems * kConvWarps) return false;  // converter items per chunk
    pl.a_bytes = up1k(3u * 2u * (2 * pl.S + 1) * Cg * 16u);
    pl.b_bytes = up1k(2u * pl.PL * 16u);
    pl.raw_bytes = nhwc ? 0u : up1k(8u * pl.Rin * pl.BW * 4u);  // channels last: no staging ring
    pl.scratch_bytes = scratch_bytes_for(kind, pl.U, pl.P);
    const uint32_t tail = 8u * Bars::kCount + 32u + pl.scratch_bytes;  // (scratch, barriers, slot, flag, alignment)
    auto total = [&](int na, int nb, int nr) {
        return (size_t)na * pl.a_bytes + (size_t)nb * pl.b_bytes + (size_t)nr * pl.raw_bytes + tail;
    };
    // resident filter when it still leaves 2 B planes and 2 staged tiles
    const int nr0 = nhwc ? 0 : 2;
    // (with several channel tiles the units alternate between their filters,
    // so the filter streams)
    pl.resident = pl.MT == 1 && total(pl.chunks, 2, nr0) <= (size_t)kSmemLimit;
    const int na_min = pl.resident ? pl.chunks : 2;
    pl.na = na_min, pl.nb = 2, pl.nr = nr0;
    if (total(pl.na, pl.nb, pl.nr) > (size_t)kSmemLimit) return false;
    // grow the rings while they fit: staged tiles first (they hide DRAM
    // latency), then B planes, then filter stages
    for (bool grew = true; grew;) {
        grew = false;
        if (!nhwc && pl.nr < kMaxRing && total(pl.na, pl.nb, pl.nr + 1) <= (size_t)kSmemLimit) ++pl.nr, grew = true;
        // channels last, the B planes are also the input prefetch ring
        if (pl.nb < (nhwc ? kMaxRing : 3) && total(pl.na, pl.nb + 1, pl.nr) <= (size_t)kSmemLimit) ++pl.nb, grew = true;
        if (!pl.resident && pl.na < 3 && total(pl.na + 1, pl.nb, pl.nr) <= (size_t)kSmemLimit) ++pl.na, grew = true;
    }
    pl.a_off = 0;
    pl.b_off = pl.na * pl.a_bytes;
    pl.raw_off = pl.b_off + pl.nb * pl.b_bytes;
    // (the barriers, the tensor-memory slot and the abort flag last: the
    // GroupNorm finalize reuses everything below them once the roles end)
    pl.scratch_off = (pl.raw_off + pl.nr * pl.raw_bytes + 15u) & ~15u;
    pl.bar_off = (pl.scratch_off + pl.scratch_bytes + 7u) & ~7u;
    pl.smem = pl.bar_off + 8u * Bars::kCount + 8u;
    if (pl.resident) pl.na = 1;  // no filter ring: the resident block is read per chunk
    pl.Cg = Cg;
    pl.a_plane_bytes = (uint32_t)Cg * 16u;
    pl.a_lbo = (uint32_t)(2 * pl.S + 1) * pl.a_plane_bytes;
    pl.a_kw_stride = 2u * pl.a_lbo;
    pl.xpitch = needs_xpad(d) ? row_pitch(d.W) : d.W;
    if (nhwc) pl.box[0] = 4u, pl.box[1] = (uint32_t)pl.P, pl.box[2] = (uint32_t)pl.Rin, pl.box[3] = 1u;
    else pl.box[0] = (uint32_t)pl.BW, pl.box[1] = (uint32_t)pl.Rin, pl.box[2] = 8u, pl.box[3] = 1u;
    return pl.smem <= (size_t)kSmemLimit;
}

uint32_t make_idesc(int M, int N) {
    // kind::tf32 instruction descriptor: D fp32 (bits 4-5 = 1), A tf32 (bits 7-9 = 2),
    // B tf32 (bits 10-12 = 2), both K-major (bits 15, 16 = 0), N>>3 at bits 17-22,
    // M>>4 at bits 24-28; dense, no negation, no saturation.
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the CUDA driver API's tensor-map encoder, looked up once (a function-local static:
// initialised exactly once even when several host threads call first)
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return nullptr;
    }();
    return fn;
}

// rows of one tile with at most 128 output channels, and everything else
// (column tiles, channel tiles) run separate instantiations, so the common
// case carries none of the tiling arithmetic (the GroupNorm chain's column
// tiles never occur, its channel tiles only in their own instantiation)
template <int KIND>
conv_epi_status launch_tc(const TcArgs &args, const Plan &pl, int grid, cudaStream_t s) {
    // (the GroupNorm chain's general instantiation pools two bands per unit)
    const bool general = is_gn(KIND) ? args.c.U == 4 : (args.c.CT > 1 || args.c.MT > 1);
    auto k = general ? tc_conv_epi<KIND, true> : tc_conv_epi<KIND, false>;
    CE_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem));
    // The in-kernel finalize waits for every CTA: a cooperative launch
    // guarantees they are all resident (one per SM, grid <= SM count).  Where
    // the device refuses it (fewer SMs granted to this context), the caller
    // runs the separate finalize kernel instead.  Every launch also allows
    // programmatic dependent launch on the kernel before it (see
    // grid_dep_wait); a launch refused with both attributes is retried
    // without that one.  (Measured per chain: C4 -3 us, C5 -2 us, the 32x32
    // case -4 us; the per-channel chains ran slower with it, C3 581 -> 587 us,
    // so they launch without it.)
    cudaLaunchAttribute attr[2];
    int na = 0;
    constexpr bool kPdl = KIND != CONV_EPI_MUL_LRELU_GELU && KIND != CONV_EPI_NONE && KIND != kKindConvStats;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na++].val.programmaticStreamSerializationAllowed = kPdl ? 1 : 0;
    if (args.c.gn_fin) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na++].val.cooperative = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid), cfg.blockDim = dim3(kThreads), cfg.dynamicSmemBytes = pl.smem, cfg.stream = s;
    cfg.attrs = attr, cfg.numAttrs = (unsigned)na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, args);
    if (e != cudaSuccess && e != cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();
        cfg.attrs = attr + 1, cfg.numAttrs = (unsigned)(na - 1);
        e = cudaLaunchKernelEx(&cfg, k, args);
    }
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();
        return CONV_EPI_ERR_UNSUPPORTED;
    }
    CE_CUDA(e);
    CE_CUDA(cudaGetLastError());
    return CONV_EPI_OK;
}

}  // namespace

// The GroupNorm chain fused into the conv kernel: its epilogue pools 4x4
// windows over bands of 4 rows.  Up to 64 channels (two 64-channel row slots
// per u): one band per unit with P in 80..128 (4 sixteen-column chunks per
// warp; Wo >= 96 in the page-shape kernel, Wo >= 64 in the generalised one,
// which masks one chunk more), two with P = 64 (2 chunks).  65..128 channels
// (one slot of 128, P in 80..128, Wo >= 64): half a band per unit, folded by
// the finalize.  Rows of 128..254 outputs (up to 64 channels): one row pair
// per unit, half a band.  2x2 windows (up to 64 channels, Wo 64..126): two
// bands of 2 rows per unit.  Other GroupNorm shapes run as two passes
// (tc_forward).
bool tc_gn_fused(const conv_epi_desc &d, const conv_epi_epilogue_desc &e) {
    Plan pl;
    const int kind = tc_gn_kind(d, e.pool_k);
    if (!make_plan(d, kind, pl)) return false;
    // one-band rows: the unmasked chunks must be whole (see the epilogue)
    const bool wide = pl.P > 64 && pl.P <= 128 && d.W - 2 >= (kind == kKindGnXNarrow || kind == kKindGnTiles ? 64 : 96);
    const bool one_band = pl.S == 2 && pl.RU == 4 && wide;
    const bool two_bands = pl.S == 2 && pl.RU == 8 && pl.P == 64;
    // more than 64 channels in rows of up to 64 columns: no stacking, the
    // unit's four rows one whole band (more than 128: per channel tile)
    const bool one_band_s1 = pl.S == 1 && pl.RU == 4 && pl.P == 64;
    // 65..128 channels fill M without stacking: a unit holds 2 rows, half a
    // band, and the finalize folds the halves
    // (more than 128 channels: channel tiles of 128, each unit one tile; a
    // group's channels, a power of two up to 64, never straddle two tiles)
    const bool half_band = pl.S == 1 && pl.RU == 2 && wide;
    // rows of 130..256 columns (Cout <= 64): one row pair per unit (U = 1),
    // the first 128 output columns whole
    const bool wide_rows = kind == kKindGnWide && pl.S == 2 && pl.U == 1 && pl.CT == 1 && pl.P > 128 &&
                           d.W - 2 >= 128;
    // (Cout below 64 or 128 runs as a 64- or 128-channel GEMM with zero
    // filters; a group's channels must be a power-of-two run of lanes, at
    // most 64, for the shuffle sums and the fold)
    // 2 x 2 windows (Cout <= 64): the one-band layout, two bands per unit,
    // the first 64 output columns whole
    // (65..128 channels: no stacking, a unit's two rows the one band)
    const bool pool2 = ((kind == kKindGnPool2 || kind == kKindGnPool2S1) && pl.U == 2 && pl.P > 64 && pl.P <= 128 &&
                        d.W - 2 >= 64) ||
                       ((kind == kKindGnPool2 || kind == kKindGnPool2S1) && pl.U == 4 && pl.P == 64);  // (four u per unit)
    // rows wider than 256 columns (Cout <= 64): column tiles of 252 outputs,
    // each unit one row pair of one tile (rows of 127 outputs: one tile)
    const bool col_tiles = kind == kKindGnColTiles && pl.S == 2 && pl.U == 1 && pl.P > 128;
    const int cpg = d.Cout / e.groups;
    // 65..128 channels on rows of 130..256 columns: one row, a quarter band, per unit
    const bool wide_s1 = kind == kKindGnWideS1 && pl.S == 1 && pl.U == 1 && pl.CT == 1 && pl.P > 128 && d.W - 2 >= 128;
    // 2 x 2 windows on rows of 130..240 columns (Cout <= 64): a row pair, one band, per unit (the plan
    // above fails for wider rows: shared memory)
    const bool wide_p2 = kind == kKindGnWideP2 && pl.S == 2 && pl.U == 1 && pl.CT == 1 && pl.P > 128 && d.W - 2 >= 128;
    const bool shape =
        e.pool_k == 4 ? (one_band || two_bands || one_band_s1 || half_band || wide_rows || wide_s1 || col_tiles)
                      : e.pool_k == 2 && (pool2 || wide_p2);
    return shape && (cpg & (cpg - 1)) == 0 && cpg <= 64;
}

// the workspace slots of a fused GroupNorm band's pooled extremes, folded by
// the finalize: a unit of 2 rows holds half a 4-row band (2; 2 x 2 windows
// make such a unit a whole band), a unit of 1 row a quarter (4)
int tc_gn_slots(const Plan &pl, int kind) {
    if (kind == kKindGnWideS1) return 4;  // a unit of 1 row: a quarter band
    return pl.RU == 2 && kind != kKindGnPool2S1 && kind != kKindGnWideP2 ? 2 : 1;
}

conv_epi_status tc_supported(const conv_epi_desc &d, const conv_epi_epilogue_desc *e) {
    Plan pl;
    int kind = e ? e->kind : CONV_EPI_MIN_TANH2;
    // a GroupNorm shape the fused epilogue does not take needs the plain conv
    if (kind == CONV_EPI_GN_SCALE_POOL_CLAMP) kind = tc_gn_fused(d, *e) ? tc_gn_kind(d, e->pool_k) : CONV_EPI_NONE;
    if (!make_plan(d, kind, pl)) return CONV_EPI_ERR_UNSUPPORTED;
    return CONV_EPI_OK;
}

// The two-pass form's buffer: the conv output y [N][Cout][Ho][Wo], then (from
// a 256-byte boundary) the conv kernel's per-unit sums
// [N][units per image][2 column groups][128 accumulator rows] float pairs.
size_t tc_y_bytes(const conv_epi_desc &d) {
    return ((size_t)d.N * d.Cout * (d.H - 2) * (d.W - 2) * sizeof(float) + 255) & ~(size_t)255;
}
int tc_stat_units(const conv_epi_desc &d) {
    Plan pl;
    if (!make_plan(d, kKindConvStats, pl)) return 0;
    return (d.H - 2 + pl.RU - 1) / pl.RU * pl.CT * pl.MT;
}
size_t tc_ybuf_bytes(const conv_epi_desc &d) {
    return tc_y_bytes(d) + (size_t)d.N * tc_stat_units(d) * 2 * 128 * sizeof(float2);
}

size_t tc_xpad_bytes(const conv_epi_desc &d) {
    if (d.mode != CONV_EPI_MODE_TF32 || !needs_xpad(d)) return 0;
    return (size_t)d.N * d.Cin * d.H * row_pitch(d.W) * sizeof(float);
}

conv_epi_status tc_plan_query(const conv_epi_desc &d, const conv_epi_epilogue_desc &e, conv_epi_plan &q) {
    q = conv_epi_plan{};
    q.struct_bytes = (int64_t)sizeof(conv_epi_plan);
    Plan pl;
    // a GroupNorm shape the fused epilogue does not take: the plain conv's
    // plan (its first pass)
    const bool two_pass = e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP && !tc_gn_fused(d, e);
    const int kind = two_pass ? CONV_EPI_NONE : e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP ? tc_gn_kind(d, e.pool_k) : e.kind;
    q.gn_two_pass = two_pass ? 1 : 0;
    if (!make_plan(d, kind, pl)) return CONV_EPI_ERR_UNSUPPORTED;
    q.gemm_cout = pl.Cg, q.S = pl.S, q.P = pl.P, q.U = pl.U, q.RU = pl.RU, q.Rin = pl.Rin, q.PL = pl.PL;
    q.ucol = pl.ucol, q.chunks = pl.chunks, q.CT = pl.CT, q.CW = pl.CW, q.BW = pl.BW, q.MT = pl.MT;
    q.units_per_image = (int64_t)((d.H - 2 + pl.RU - 1) / pl.RU) * pl.CT * pl.MT;
    q.resident = pl.resident, q.na = pl.na, q.nb = pl.nb, q.nr = pl.nr;
    q.a_bytes = pl.a_bytes, q.b_bytes = pl.b_bytes, q.raw_bytes = pl.raw_bytes, q.scratch_bytes = pl.scratch_bytes;
    q.a_off = pl.a_off, q.b_off = pl.b_off, q.raw_off = pl.raw_off, q.bar_off = pl.bar_off;
    q.scratch_off = pl.scratch_off;
    q.bar_bytes = 8 * Bars::kCount;
    q.smem = (int64_t)pl.smem, q.smem_limit = kSmemLimit;
    q.a_plane_bytes = pl.a_plane_bytes, q.a_lbo = pl.a_lbo, q.a_kw_stride = pl.a_kw_stride;
    q.x_pitch = pl.xpitch;
    for (int i = 0; i < 4; ++i) q.box[i] = pl.box[i];
    q.acc_cols = kAccStride, q.tmem_cols = kTmemCols;
    q.conv_items = kConvItems * kConvWarps;
    conv_epi_desc dt = d;
    dt.mode = CONV_EPI_MODE_TF32;
    q.wpack_bytes = (int64_t)tc_wpack_bytes(dt);
    q.xpad_bytes = (int64_t)tc_xpad_bytes(dt);
    q.ybuf_bytes = two_pass ? (int64_t)tc_ybuf_bytes(dt) : 0;
    return tc_supported(d, &e);
}

size_t tc_wpack_bytes(const conv_epi_desc &d) {
    const int Cg = gemm_cout(d.Cout), S = 128 / Cg;
    const size_t chunk = ((size_t)3 * 2 * (2 * S + 1) * Cg * 16 + 1023) & ~(size_t)1023;
    return ((size_t)channel_tiles(d.Cout) * ((d.Cin + 7) / 8) + 1) * chunk + 256;
}

int tc_gn_units(const conv_epi_desc &d, int Ho, int pool_k) {
    Plan pl;
    if (!make_plan(d, tc_gn_kind(d, pool_k), pl)) return (Ho + pool_k - 1) / pool_k;
    return (Ho + pl.RU - 1) / pl.RU * pl.CT * pl.MT;  // (channel tiles: a unit per tile)
}

conv_epi_status tc_reserve(conv_epi_handle h, const conv_epi_epilogue_desc &e) {
    if (e.kind != CONV_EPI_GN_SCALE_POOL_CLAMP) return CONV_EPI_OK;
    if (tc_gn_fused(h->d, e)) return ensure_gn_workspace(h, e.pool_k, e.groups, tc_gn_units(h->d, h->Ho, e.pool_k));
    const size_t need = tc_ybuf_bytes(h->d);  // the two-pass form: the conv output
    if (need > h->ybuf_bytes) {
        if (h->ybuf) {
            CE_CUDA(cudaDeviceSynchronize());
            CE_CUDA(cudaFree(h->ybuf));
            h->ybuf = nullptr, h->ybuf_bytes = 0;
        }
        CE_CUDA(cudaMalloc(&h->ybuf, need));
        h->ybuf_bytes = need;
    }
    return ensure_post_stats(h, e.groups);
}

conv_epi_status tc_forward(conv_epi_handle h, const float *x, const float *w, const float *b,
                           const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    if (e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP && !tc_gn_fused(d, e)) {
        // GroupNorm shapes the fused epilogue does not take, in two passes:
        // the tensor-core conv writes y + b to the handle's buffer, then the
        // chain's post-pass (statistics, then normalise-scale-pool-clamp)
        if (!h->ybuf || h->ybuf_bytes < tc_ybuf_bytes(d) || h->post_bytes < (size_t)d.N * e.groups * 2 * sizeof(float))
            return CONV_EPI_ERR_INVALID_ARG;  // conv_epi_reserve sizes both
        conv_epi_epilogue_desc plain = e;
        plain.kind = kKindConvStats;  // y, and each unit's sums of y and y^2 per channel
        plain.index_out = nullptr;
        conv_epi_status st = tc_forward(h, x, w, b, plain, h->ybuf, s);
        if (st) return st;
        const int conv_launches = h->last_launches;
        Plan pl;
        if (!make_plan(d, kKindConvStats, pl)) return CONV_EPI_ERR_UNSUPPORTED;
        const float2 *ystat = reinterpret_cast<const float2 *>(reinterpret_cast<const char *>(h->ybuf) + tc_y_bytes(d));
        if ((st = postpass_gn_units(h, h->ybuf, ystat, tc_stat_units(d), pl.S, pl.MT, gemm_cout(d.Cout), e, out, s)))
            return st;
        h->last_launches += conv_launches;
        return CONV_EPI_OK;
    }
    // the kernel: the GroupNorm chain's page-shape or generalised instantiation
    const int kkind = e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP ? tc_gn_kind(d, e.pool_k) : e.kind;
    Plan pl;
    if (!make_plan(d, kkind, pl)) return CONV_EPI_ERR_UNSUPPORTED;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return CONV_EPI_ERR_CUDA;
    TcArgs args{};  // value-initialised: zeros, and the workspace pointers' defaults
    Cfg &a = args.c;
    const bool nhwc = d.layout == CONV_EPI_LAYOUT_NHWC;
    // NCHW rows that are not whole 16-byte units: the tensor map describes the
    // padded copy (filled by pad_rows below, before the conv kernel)
    const bool padded = needs_xpad(d);
    const size_t nrows = (size_t)d.N * d.Cin * d.H;
    if (padded && (!h->xpad || h->xpad_bytes < nrows * row_pitch(d.W) * sizeof(float))) return CONV_EPI_ERR_UNSUPPORTED;
    {
        // NCHW: x as (W, H, C, N), box (BW, Rin, 8, 1) -> staging [8][Rin][BW]
        // (BW = W rounded up to 4, or 256 per column tile of a wider row); the
        // row stride is the padded copy's when W is not a multiple of 4.
        // NHWC: x as (C, W, H, N), box (4, P, Rin, 1) -> a B plane [Rin][P][4]
        // (columns W..P-1, rows past H and channels past Cin read as zeros).
        cuuint64_t dims[4], strides[3];
        cuuint32_t box[4];
        if (nhwc) {
            dims[0] = (cuuint64_t)d.Cin, dims[1] = (cuuint64_t)d.W, dims[2] = (cuuint64_t)d.H, dims[3] = (cuuint64_t)d.N;
            strides[0] = (cuuint64_t)d.Cin * 4, strides[1] = (cuuint64_t)d.Cin * d.W * 4,
            strides[2] = (cuuint64_t)d.Cin * d.W * d.H * 4;
        } else {
            const cuuint64_t pitch = (cuuint64_t)pl.xpitch;
            dims[0] = (cuuint64_t)d.W, dims[1] = (cuuint64_t)d.H, dims[2] = (cuuint64_t)d.Cin, dims[3] = (cuuint64_t)d.N;
            strides[0] = pitch * 4, strides[1] = pitch * d.H * 4, strides[2] = pitch * d.H * d.Cin * 4;
        }
        for (int i = 0; i < 4; ++i) box[i] = (cuuint32_t)pl.box[i];
        const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
        void *base = padded ? static_cast<void *>(h->xpad) : const_cast<float *>(x);
        const CUresult r = enc(&args.xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return CONV_EPI_ERR_UNSUPPORTED;
    }
    // 1) pack the filter for this call: chunk c at byte offset c * a_bytes
    {
        const size_t per_chunk = (size_t)3 * 2 * (2 * pl.S + 1) * gemm_cout(d.Cout) * 4;  // floats
        const size_t total = (size_t)pl.chunks * per_chunk;
        const int threads = 256;
        const int blocks = (int)((total + threads - 1) / threads);
        if (pl.a_bytes != per_chunk * 4) return CONV_EPI_ERR_UNSUPPORTED;  // chunks must pack back to back
        // channel tile m: filters 128m .. 128m + 127, after the previous tiles' chunks
        for (int m = 0; m < pl.MT; ++m) {
            const int Cg = gemm_cout(d.Cout);
            const bool gn_sign = e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP;  // (the fused form: the slope's sign)
            pack_weights<<<blocks, threads, 0, s>>>(w + (size_t)m * Cg * d.Cin * 9, h->wpack + (size_t)m * total,
                                                    d.Cin, Cg, min(Cg, d.Cout - m * Cg), pl.S,
                                                    gn_sign ? e.gamma + (size_t)m * Cg : nullptr,
                                                    gn_sign ? e.chan_scale + (size_t)m * Cg : nullptr,
                                                    m == 0 && gn_sign ? h->gn.arrive : nullptr);
            CE_CUDA(cudaGetLastError());
        }
    }
    if (padded) {
        const size_t blocks = (nrows + 7) / 8;  // 8 warps (rows) per block
        pad_rows<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(x, h->xpad, nrows, d.W, row_pitch(d.W));
        CE_CUDA(cudaGetLastError());
    }
    a.x = x, a.b = b, a.wpack = h->wpack, a.out = out, a.err = h->dev_err;
    a.N = d.N, a.Cin = d.Cin, a.H = d.H, a.W = d.W, a.Cout = gemm_cout(d.Cout), a.Co = d.Cout, a.Ho = h->Ho, a.Wo = h->Wo;
    a.S = pl.S, a.P = pl.P, a.U = pl.U, a.RU = pl.RU, a.Rin = pl.Rin, a.PL = pl.PL, a.ucol = pl.ucol;
    a.chunks = pl.chunks;
    a.CT = pl.CT, a.CW = pl.CW, a.BW = pl.BW, a.MT = pl.MT;
    a.units_per_img = (h->Ho + pl.RU - 1) / pl.RU * pl.CT * pl.MT;
    a.total_units = d.N * a.units_per_img;
    a.resident = pl.resident, a.na = pl.na, a.nb = pl.nb, a.nr = pl.nr;
    a.a_bytes = pl.a_bytes, a.b_bytes = pl.b_bytes, a.raw_bytes = pl.raw_bytes;
    a.raw_tx = nhwc ? 2u * 4u * pl.P * pl.Rin * 4u : 8u * pl.Rin * pl.BW * 4u;  // bytes one tile delivers
    a.nhwc = nhwc ? 1 : 0;
    a.a_off = pl.a_off, a.b_off = pl.b_off, a.raw_off = pl.raw_off, a.bar_off = pl.bar_off;
    a.scratch_off = pl.scratch_off;
    a.a_plane_bytes = pl.a_plane_bytes, a.a_lbo = pl.a_lbo, a.a_kw_stride = pl.a_kw_stride;
    a.idesc = make_idesc(128, pl.P);
    a.scalar = e.scalar, a.chan_scale = e.chan_scale, a.gamma = e.gamma, a.slope = e.lrelu_slope;
    a.groups = e.groups;
    if (e.kind == kKindConvStats)  // the per-unit sums, after y in the two-pass buffer
        a.gn.pmax = reinterpret_cast<float *>(reinterpret_cast<char *>(h->ybuf) + tc_y_bytes(d));
    a.drop_tile = h->test_drop_tile;
    h->test_drop_tile = -1;  // one forward only
    if (e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP) {
        a.gn = h->gn;
        a.Hp = h->gn.Hp, a.Wp = h->gn.Wp;
        // (a unit's windows: up to 32 or, for the two-pass rows, 64; column tiles any number)
        const int max_wp = kkind == kKindGnColTiles                                                  ? a.Wp
                           : kkind == kKindGnWideP2                                                   ? 128
                           : kkind == kKindGnWide || kkind == kKindGnWideS1 || kkind == kKindGnPool2 ||
                                     kkind == kKindGnPool2S1
                               ? 64
                                                                                                      : 32;
        if (h->gn.units != a.units_per_img || a.Wp > max_wp) return CONV_EPI_ERR_INVALID_ARG;
        // finalize inside the kernel when each (image, group) block of pooled
        // values is whole float4s (16-byte aligned blocks) and small enough
        // for the multiply-high divisions (t < 2^18 pooled float4 per batch,
        // channel offsets < 2^16); otherwise the separate finalize kernel
        const uint32_t per = (uint32_t)(a.Hp * a.Wp), F = (uint32_t)(d.Cout / e.groups) * per;
        a.gn_fin = (F % 4 == 0 && F <= 65536u && d.Cout / e.groups <= 64 && h->coop &&
                    // one pair's blocks (two slots each for half bands) fit the buffer
                    F * 4u * (uint32_t)tc_gn_slots(pl, kkind) <= pl.bar_off - kFinBufOff &&
                    (reinterpret_cast<uintptr_t>(out) & 15u) == 0 && (reinterpret_cast<uintptr_t>(h->gn.pmax) & 15u) == 0)
                       ? 1 : 0;
        a.beta = e.beta, a.eps = e.eps, a.lo = e.clamp_lo, a.hi = e.clamp_hi;
        a.cnt = (float)((double)(d.Cout / e.groups) * h->Ho * h->Wo);
        a.per_magic = (uint32_t)((((uint64_t)1 << 32) + per - 1) / per);
        const uint32_t F4 = F / 4 ? F / 4 : 1;
        a.f4_magic = (uint32_t)((((uint64_t)1 << 32) + F4 - 1) / F4);
    }
    const int grid = a.total_units < h->sm_count ? a.total_units : h->sm_count;
    int fills = 0;
    if (pl.MT > 1 && (e.kind == CONV_EPI_MIN_TANH2 || e.kind == CONV_EPI_SCALE_MIN)) {
        const size_t n_out = (size_t)d.N * h->Ho * h->Wo;
        const size_t fb = (n_out + 255) / 256;
        fill_f32<<<(unsigned)(fb < 4096 ? fb : 4096), 256, 0, s>>>(out, n_out, INFINITY);
        CE_CUDA(cudaGetLastError());
        fills = 1;
    }
    conv_epi_status st;
    switch (e.kind) {
    case CONV_EPI_MIN_TANH2: st = launch_tc<CONV_EPI_MIN_TANH2>(args, pl, grid, s); break;
    case CONV_EPI_SCALE_MIN: st = launch_tc<CONV_EPI_SCALE_MIN>(args, pl, grid, s); break;
    case CONV_EPI_MUL_LRELU_GELU: st = launch_tc<CONV_EPI_MUL_LRELU_GELU>(args, pl, grid, s); break;
    case CONV_EPI_NONE: st = launch_tc<CONV_EPI_NONE>(args, pl, grid, s); break;
    case kKindConvStats: st = launch_tc<kKindConvStats>(args, pl, grid, s); break;
    case CONV_EPI_GN_SCALE_POOL_CLAMP: {
        auto launch_gn = [&]() {
            return kkind == kKindGnX         ? launch_tc<kKindGnX>(args, pl, grid, s)
                   : kkind == kKindGnXNarrow ? launch_tc<kKindGnXNarrow>(args, pl, grid, s)
                   : kkind == kKindGnWide    ? launch_tc<kKindGnWide>(args, pl, grid, s)
                   : kkind == kKindGnPool2   ? launch_tc<kKindGnPool2>(args, pl, grid, s)
                   : kkind == kKindGnPool2S1 ? launch_tc<kKindGnPool2S1>(args, pl, grid, s)
                   : kkind == kKindGnWideP2  ? launch_tc<kKindGnWideP2>(args, pl, grid, s)
                   : kkind == kKindGnWideS1  ? launch_tc<kKindGnWideS1>(args, pl, grid, s)
                   : kkind == kKindGnTiles   ? launch_tc<kKindGnTiles>(args, pl, grid, s)
                   : kkind == kKindGnColTiles ? launch_tc<kKindGnColTiles>(args, pl, grid, s)
                                             : launch_tc<CONV_EPI_GN_SCALE_POOL_CLAMP>(args, pl, grid, s);
        };
        st = launch_gn();
        if (st == CONV_EPI_ERR_UNSUPPORTED && a.gn_fin) {  // cooperative launch refused: finalize separately
            a.gn_fin = 0;
            st = launch_gn();
        }
        break;
    }
    default: return CONV_EPI_ERR_INVALID_ARG;
    }
    if (st) return st;
    h->last_launches = pl.MT + 1 + fills + (padded ? 1 : 0);  // packs, fill, conv, row padding
    if (e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP && !a.gn_fin) {
        if ((st = gn_finalize(h, e, out, s, true, tc_gn_slots(pl, kkind)))) return st;
        h->last_launches += 1;
    }
    return CONV_EPI_OK;
}

}  // namespace conv_epi
