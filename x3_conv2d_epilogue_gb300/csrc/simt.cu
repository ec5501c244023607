// simt.cu -- fp32 CUDA-core path (CONV_EPI_MODE_FP32, the strict-tolerance
// mode): a direct 3x3 convolution with the post-conv chain fused into the
// same kernel, so the full conv output is written only by the per-channel
// chain (MUL_LRELU_GELU) and by CONV_EPI_NONE, whose outputs are the full
// tensor anyway.
//
// Prior art: the p54 page (POPCORNBENCH Kimi-K2.6, level-2 problem 54), in
// its fused direct-conv design, stages a haloed input tile and a few output
// channels' filters in shared memory and has each thread accumulate outputs
// over (c_in, kh, kw).  Here a CTA owns one output row (or one pooling band
// of rows) of one image and every output channel, so the channel reductions
// of the min chains and the pooling of the GroupNorm chain finish on chip.
//
// Work decomposition (one CTA):
//   threads  = PG pixel groups x CS channel slots (<= 256)
//   a thread = 4 consecutive output pixels x 16 output channels per pass,
//              accumulated as 8 channel pairs by the paired fp32 FMA
//              (fma.rn.f32x2: two FMAs per issued instruction, each rounded
//              as fmaf, so the bits are those of scalar FMAs)
//   a pass   = CS*16 channels; passes loop until Cout is covered
//   staging  = 16 input channels x 3 input rows x (PG*4 + 4) columns of x,
//              and the matching 16 x 9 x (CS*16) filter taps, in shared memory,
//              by asynchronous copies (cp.async; 16-byte ones for x where its
//              rows are whole 16-byte groups)
#include <float.h>
#include <math.h>

#include "internal.h"

namespace conv_epi {
namespace {

constexpr int kCI = 16;  // input channels staged per step
constexpr int kCO = 16;  // output channels per thread per pass
constexpr int kPX = 4;   // consecutive output pixels per thread
constexpr int kRowsPerCta = 4;  // output rows per CTA for the min and per-channel chains
// dynamic shared memory per CTA: the 227 KB opt-in less the static group sums
// (5 KB) and a margin
constexpr size_t kSmemDynLimit = 227 * 1024 - 6 * 1024;
// a GroupNorm band staged at once, or the min and per-channel chains' ring
// of input rows, where the CTA's tiles keep two CTAs per SM
constexpr size_t kBandSmemLimit = 110 * 1024;

struct SimtArgs {
    const float *x, *w, *b;
    int N, Cin, H, W, Cout, Ho, Wo;
    int PG, CS;          // thread layout
    int units;           // CTAs per image
    int rpc;             // output rows per CTA (min and per-channel chains)
    int xrows;           // input rows staged at a time: 3 (one output row), or
                         // PK + 2 (a GroupNorm band's rows, staged once), or
                         // 4 (ring: a slot per input row, see below)
    int ring;            // min and per-channel chains: input rows in a ring of 4
    const float *wpk;    // the filter packed as [pass][Cin * 9][COP] (zeros past
                         // Cout), so a step's tile is one contiguous copy
    int ntiles;          // pixel tiles of PG*4 columns along a row
    float scalar;        // MIN kinds
    const float *chan_scale;
    float slope;
    int groups, Hp, Wp;  // GN
    float *out;
    int32_t *idx;
    GnWork gn;
};

__device__ __forceinline__ float gelu_erf(float t) { return 0.5f * t * (1.0f + erff(t * 0.70710678118654752f)); }

// two fp32 values as one 64-bit register pair, and the paired FMA on such
// pairs: each half is fmaf(a, b, c) of its own operands, rounded once, so a
// paired accumulation gives the same bits as two scalar ones
__device__ __forceinline__ uint64_t pair(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(__float_as_uint(lo)), "r"(__float_as_uint(hi)));
    return r;
}
__device__ __forceinline__ float2 unpair(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t add_pair(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma_pair(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// asynchronous global -> shared copies (cp.async): src_bytes below the copy
// size zero-fills the rest (0: nothing is read, src need only be a valid
// address); completed by cp_async_wait_all
__device__ __forceinline__ void cp_async16(float *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// KIND: conv_epi_kind; PK: pool kernel (GN only; 1, 2 or 4, dividing kPX);
// CO: output channels per thread per pass (16, or 8 for the GroupNorm chain
// where 16 would leave channel slots of the CTA empty: twice the threads, and
// its per-channel band state in half the registers, so two CTAs fit an SM;
// with 1 x 1 windows the state of four windows a channel does not fit 128
// registers, and that instantiation keeps one CTA per SM)
template <int KIND, int PK, int CO>
__global__ void __launch_bounds__(256, KIND == CONV_EPI_GN_SCALE_POOL_CLAMP && (CO == 16 || PK == 1) ? 1 : 2)
    simt_conv_epi(const SimtArgs a) {
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    const int tid = threadIdx.x;
    const int PG = a.PG, CS = a.CS;
    const int tx = tid % PG, ty = tid / PG;
    const int TW = PG * kPX, XW = TW + 4, COP = CS * CO;
    const int NR = a.xrows;          // staged input rows
    float *xs = sm;                  // [kCI][NR][XW]
    float *ws = sm + kCI * NR * XW;  // [kCI][9][COP]
    const int n = blockIdx.x / a.units;
    const int u = blockIdx.x % a.units;
    constexpr bool kGN = KIND == CONV_EPI_GN_SCALE_POOL_CLAMP;
    constexpr bool kMin = KIND == CONV_EPI_MIN_TANH2 || KIND == CONV_EPI_SCALE_MIN;
    // rows of this CTA: a pooling band (GroupNorm), else rpc output rows, one
    // after the other (r0 .. r1 - 1 is the current band or row)
    const int row_lo = kGN ? u * PK : u * a.rpc;
    const int row_hi = kGN ? row_lo + 1 : min(row_lo + a.rpc, a.Ho);
    // min kinds: +1 tracks the minimum of y (scalar > 0), -1 the maximum (scalar < 0)
    const int sgn = a.scalar > 0.0f ? 1 : (a.scalar < 0.0f ? -1 : 0);
    // one input-channel step and one output-channel pass: the filter tile is
    // the same for every row and column tile of the CTA and is staged once,
    // when the reductions' scratch (at the start of shared memory) stays
    // below it
    const bool w_once = a.Cin <= kCI && a.Cout <= COP && 2 * CS * TW <= kCI * NR * XW && 2 * COP * PG <= kCI * NR * XW;
    // a GroupNorm band staged at once (one input-channel step, one channel
    // pass, one pixel tile: the host sets xrows = PK + 2 only then): rows
    // r0 .. r0 + PK + 1 are staged before the band's first row and serve all
    // of its rows (rows at or past H, below a short last band, are zeros)
    const bool band_once = kGN && NR > 3;
    // min and per-channel chains with several rows per CTA, one input-channel
    // step, one channel pass and one pixel tile (the host sets ring then,
    // with xrows = 4): input row ir lives in slot ir & 3; the CTA's first row
    // stages three rows, and each row then prefetches the one input row the
    // next needs (into the slot of the row just finished) while it computes.
    // The min chain's scratch then lies past the filter tile.
    const bool ring = !kGN && a.ring && w_once;
    float *red = ring ? ws + kCI * 9 * COP : sm;
    // input rows of whole 16-byte groups (x itself is 16-byte aligned): the
    // staged rows then start on 16-byte boundaries too (XW and wo0 are
    // multiples of 4)
    const bool xv4 = (a.W & 3) == 0;
    // GroupNorm: window indices tracked and stored only when the caller asks
    // for them (the finalize reads them only then)
    const bool want_idx = a.idx != nullptr;

    // GroupNorm per-CTA group partial sums, in a fixed summation order
    __shared__ double gpart[2 * 64];
    __shared__ double gred[2 * 256];  // per-thread partials of the group sums
    if (kGN) {
        for (int i = tid; i < 2 * 64; i += blockDim.x) gpart[i] = 0.0;
    }

    for (int row = row_lo; row < row_hi; ++row) {
    const int r0 = kGN ? row_lo : row;
    const int r1 = kGN ? min(row_lo + PK, a.Ho) : row + 1;
    for (int t = 0; t < a.ntiles; ++t) {
        const int wo0 = t * TW;
        float best[kPX];
        int bidx[kPX];
#pragma unroll
        for (int p = 0; p < kPX; ++p) best[p] = 0.0f, bidx[p] = -1;

        for (int cobase = 0; cobase < a.Cout; cobase += COP) {
            const int co0 = cobase + ty * CO;
            constexpr int WPT = kGN ? kPX / PK : 1;  // pooling windows per thread
            // GroupNorm sums of y and y^2 for channels 2h, 2h + 1 as packed
            // pairs (each half added in the same order as a scalar sum)
            uint64_t gs2[CO / 2], gss2[CO / 2];
            float pmx[CO][WPT], pmn[CO][WPT];
            int amx[CO][WPT], amn[CO][WPT];
            if (kGN) {
#pragma unroll
                for (int h = 0; h < CO / 2; ++h) gs2[h] = gss2[h] = pair(0.0f, 0.0f);
#pragma unroll
                for (int c = 0; c < CO; ++c) {
#pragma unroll
                    for (int j = 0; j < WPT; ++j) pmx[c][j] = -FLT_MAX, pmn[c][j] = FLT_MAX, amx[c][j] = -1, amn[c][j] = -1;
                }
            }
            for (int r = r0; r < r1; ++r) {
                // accumulators of channels 2h and 2h + 1 at pixel p, as one
                // packed pair (acc2[h][p]) for the paired FMA
                uint64_t acc2[CO / 2][kPX];
#pragma unroll
                for (int h = 0; h < CO / 2; ++h) {
                    const int c = co0 + 2 * h;
                    const float b0 = c < a.Cout ? __ldg(&a.b[c]) : 0.0f, b1 = c + 1 < a.Cout ? __ldg(&a.b[c + 1]) : 0.0f;
#pragma unroll
                    for (int p = 0; p < kPX; ++p) acc2[h][p] = pair(b0, b1);
                }
                // first input row of the staged tile
                const int rs = band_once ? r0 : r;
                for (int ci0 = 0; ci0 < a.Cin; ci0 += kCI) {
                    // channels staged and used in this step (the tiles past
                    // them are never read)
                    const int nci = min(kCI, a.Cin - ci0);
                    // input rows ra .. ra + nrows - 1 of the step's channels
                    // into their tile rows (ir - rs, or slot ir & 3 in the
                    // ring), by asynchronous copies (every copy of a thread
                    // in flight at once, no register round trip), zero-filled
                    // past W and H; each copy's (channel, row, column) is
                    // stepped by the block size without divisions
                    auto stage_x = [&](int ra, int nrows) {
                        if (xv4) {  // rows of whole 16-byte groups: one copy per 4 columns
                            const int XW4 = XW >> 2, total = nci * nrows * XW4;
                            int col = tid % XW4, rr = (tid / XW4) % nrows, ci = tid / (nrows * XW4);
                            for (int i = tid; i < total; i += blockDim.x) {
                                const int gci = ci0 + ci, gw = wo0 + 4 * col, gr = ra + rr;
                                const int nv = gr < a.H ? max(0, min(4, a.W - gw)) : 0;
                                const float *src = nv ? a.x + (((size_t)n * a.Cin + gci) * a.H + gr) * a.W + gw : a.x;
                                const int srow = ring ? (gr & 3) : gr - rs;
                                cp_async16(xs + ((ci * NR + srow) * XW4 + col) * 4, src, 4 * nv);
                                col += blockDim.x;
                                while (col >= XW4) {
                                    col -= XW4;
                                    if (++rr == nrows) rr = 0, ++ci;
                                }
                            }
                        } else {
                            const int total = nci * nrows * XW;
                            int col = tid % XW, rr = (tid / XW) % nrows, ci = tid / (nrows * XW);
                            for (int i = tid; i < total; i += blockDim.x) {
                                const int gci = ci0 + ci, gw = wo0 + col, gr = ra + rr;
                                const bool ok = gr < a.H && gw < a.W;
                                const int srow = ring ? (gr & 3) : gr - rs;
                                cp_async4(xs + (ci * NR + srow) * XW + col,
                                          ok ? a.x + (((size_t)n * a.Cin + gci) * a.H + gr) * a.W + gw : a.x, ok ? 4 : 0);
                                col += blockDim.x;
                                while (col >= XW) {
                                    col -= XW;
                                    if (++rr == nrows) rr = 0, ++ci;
                                }
                            }
                        }
                    };
                    // ring, after the CTA's first row: the prefetched row has
                    // landed and every thread is past the previous row
                    if (ring && row > row_lo) {
                        cp_async_wait_all();
                        __syncthreads();
                    }
                    if (ring ? row == row_lo : (!band_once || r == r0)) {
                    __syncthreads();
                    stage_x(ring ? row : rs, ring ? 3 : NR);
                    if ((!w_once || (row == row_lo && t == 0 && r == r0)) && a.wpk) {
                        // the step's [nci * 9][COP] tile is contiguous in the
                        // packed filter (COP is a multiple of 8: whole
                        // 16-byte pieces, 16-byte aligned)
                        const int n4 = nci * 9 * COP / 4;
                        const float *src = a.wpk + ((size_t)(cobase / COP) * a.Cin * 9 + ci0 * 9) * COP;
                        for (int i = tid; i < n4; i += blockDim.x) cp_async16(ws + 4 * i, src + 4 * i, 16);
                    } else if ((!w_once || (row == row_lo && t == 0 && r == r0)) && (blockDim.x & 3) == 0) {
                        // the filter taps k = ci * 9 + tap of this step are
                        // contiguous per output channel in w: a warp copies 8
                        // channels x 4 consecutive taps (8 16-byte pieces of
                        // w), into ws[k][co]; a thread keeps its tap lane kk
                        const int KK = nci * 9, kk = tid & 3, step = blockDim.x >> 2;
                        int co = (tid >> 2) % COP, kb = (tid >> 2) / COP;
                        while (4 * kb < KK) {
                            const int k = 4 * kb + kk, gco = cobase + co;
                            if (k < KK) {
                                const bool ok = gco < a.Cout;
                                cp_async4(ws + k * COP + co, ok ? a.w + ((size_t)gco * a.Cin + ci0) * 9 + k : a.w,
                                          ok ? 4 : 0);
                            }
                            co += step;
                            while (co >= COP) co -= COP, ++kb;
                        }
                    } else if (!w_once || (row == row_lo && t == 0 && r == r0)) {
                        // (blocks of fewer or an odd number of threads, on the
                        // smallest shapes: one channel per thread, taps outer)
                        const int total = nci * 9 * COP;
                        int col = tid % COP, tap = (tid / COP) % 9, ci = tid / (9 * COP);
                        for (int i = tid; i < total; i += blockDim.x) {
                            const int gci = ci0 + ci, gco = cobase + col;
                            const bool ok = gco < a.Cout;
                            cp_async4(ws + i, ok ? a.w + ((size_t)gco * a.Cin + gci) * 9 + tap : a.w, ok ? 4 : 0);
                            col += blockDim.x;
                            while (col >= COP) {
                                col -= COP;
                                if (++tap == 9) tap = 0, ++ci;
                            }
                        }
                    }
                    cp_async_wait_all();
                    __syncthreads();
                    }
                    // ring: the next row's new input row, in flight during this row
                    if (ring && row + 1 < row_hi) stage_x(row + 3, 1);
                    for (int ci = 0; ci < nci; ++ci) {
#pragma unroll
                        for (int kh = 0; kh < 3; ++kh) {
                            const int srow = ring ? ((r + kh) & 3) : (r - rs) + kh;
                            const float *xr = xs + (ci * NR + srow) * XW + tx * kPX;
                            const float4 xa = *reinterpret_cast<const float4 *>(xr);
                            const float2 xb = *reinterpret_cast<const float2 *>(xr + 4);
                            // each input value twice, as the pair that meets two channels' taps
                            const uint64_t xd[6] = {pair(xa.x, xa.x), pair(xa.y, xa.y), pair(xa.z, xa.z),
                                                    pair(xa.w, xa.w), pair(xb.x, xb.x), pair(xb.y, xb.y)};
#pragma unroll
                            for (int kw = 0; kw < 3; ++kw) {
                                // the taps of channels 2h, 2h + 1: adjacent in the staged filter
                                const ulonglong2 *wr =
                                    reinterpret_cast<const ulonglong2 *>(ws + (ci * 9 + kh * 3 + kw) * COP + ty * CO);
                                uint64_t w2[CO / 2];
#pragma unroll
                                for (int q = 0; q < CO / 4; ++q) {
                                    const ulonglong2 f = wr[q];
                                    w2[2 * q] = f.x, w2[2 * q + 1] = f.y;
                                }
#pragma unroll
                                for (int h = 0; h < CO / 2; ++h)
#pragma unroll
                                    for (int p = 0; p < kPX; ++p) acc2[h][p] = fma_pair(w2[h], xd[p + kw], acc2[h][p]);
                            }
                        }
                    }
                }
                float acc[CO][kPX];
#pragma unroll
                for (int h = 0; h < CO / 2; ++h)
#pragma unroll
                    for (int p = 0; p < kPX; ++p) {
                        const float2 v = unpair(acc2[h][p]);
                        acc[2 * h][p] = v.x, acc[2 * h + 1][p] = v.y;
                    }

                // ---- fold this row into the chain ----
                const int wbase = wo0 + tx * kPX;
                if (kMin) {
#pragma unroll
                    for (int c = 0; c < CO; ++c) {
                        if (co0 + c >= a.Cout) break;
#pragma unroll
                        for (int p = 0; p < kPX; ++p) {
                            const float v = acc[c][p];
                            const bool better = sgn >= 0 ? v < best[p] : v > best[p];
                            if (bidx[p] < 0 || better) best[p] = v, bidx[p] = co0 + c;
                        }
                    }
                } else if (KIND == CONV_EPI_MUL_LRELU_GELU || KIND == CONV_EPI_NONE) {
                    if (wbase < a.Wo) {
#pragma unroll
                        for (int c = 0; c < CO; ++c) {
                            const int co = co0 + c;
                            if (co >= a.Cout) break;
                            float o[kPX];
                            if (KIND == CONV_EPI_NONE) {  // the conv output itself
#pragma unroll
                                for (int p = 0; p < kPX; ++p) o[p] = acc[c][p];
                            } else {
                                const float m = __ldg(&a.chan_scale[co]);
#pragma unroll
                                for (int p = 0; p < kPX; ++p) {
                                    float v = acc[c][p] * m;
                                    v = v > 0.0f ? v : a.slope * v;
                                    o[p] = gelu_erf(v);
                                }
                            }
                            float *dst = a.out + (((size_t)n * a.Cout + co) * a.Ho + r) * a.Wo + wbase;
                            if (wbase + kPX <= a.Wo && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
                                reinterpret_cast<float2 *>(dst)[0] = make_float2(o[0], o[1]);
                                reinterpret_cast<float2 *>(dst)[1] = make_float2(o[2], o[3]);
                            } else {
#pragma unroll
                                for (int p = 0; p < kPX; ++p)
                                    if (wbase + p < a.Wo) dst[p] = o[p];
                            }
                        }
                    }
                } else if (kGN) {
                    const bool prow = r < a.Hp * PK;
                    // the sums over this row's pixels inside the row (the
                    // channels past Cout have zero filters and bias: their
                    // sums stay 0 and are never read)
#pragma unroll
                    for (int p = 0; p < kPX; ++p)
                        if (wbase + p < a.Wo) {
#pragma unroll
                            for (int h = 0; h < CO / 2; ++h)
                                gs2[h] = add_pair(gs2[h], acc2[h][p]), gss2[h] = fma_pair(acc2[h][p], acc2[h][p], gss2[h]);
                        }
                    if (want_idx) {
#pragma unroll
                        for (int c = 0; c < CO; ++c) {
                            if (co0 + c >= a.Cout) break;
#pragma unroll
                            for (int p = 0; p < kPX; ++p) {
                                const int wo = wbase + p;
                                if (wo >= a.Wo) continue;
                                const float v = acc[c][p];
                                if (prow && wo < a.Wp * PK) {
                                    const int j = p / PK;
                                    const int off = (r - r0) * PK + (p % PK);
                                    if (amx[c][j] < 0 || v > pmx[c][j]) pmx[c][j] = v, amx[c][j] = off;
                                    if (amn[c][j] < 0 || v < pmn[c][j]) pmn[c][j] = v, amn[c][j] = off;
                                }
                            }
                        }
                    } else {
                        // no indices asked for: the window extremes as values
                        // only (the same values: conv outputs are finite)
#pragma unroll
                        for (int c = 0; c < CO; ++c) {
                            if (co0 + c >= a.Cout) break;
#pragma unroll
                            for (int p = 0; p < kPX; ++p) {
                                const int wo = wbase + p;
                                if (wo >= a.Wo) continue;
                                const float v = acc[c][p];
                                if (prow && wo < a.Wp * PK) {
                                    pmx[c][p / PK] = fmaxf(pmx[c][p / PK], v);
                                    pmn[c][p / PK] = fminf(pmn[c][p / PK], v);
                                }
                            }
                        }
                    }
                }
            }  // rows

            if (kGN) {
                // pooled max/min of this band (a full band only: u < Hp)
                if (u < a.Hp) {
#pragma unroll
                    for (int c = 0; c < CO; ++c) {
                        const int co = co0 + c;
                        if (co >= a.Cout) break;
#pragma unroll
                        for (int j = 0; j < WPT; ++j) {
                            const int pw = (wo0 + tx * kPX) / PK + j;
                            if (pw >= a.Wp) continue;
                            const size_t o = (((size_t)n * a.Cout + co) * a.Hp + u) * a.Wp + pw;
                            a.gn.pmax[o] = pmx[c][j];
                            a.gn.pmin[o] = pmn[c][j];
                            if (want_idx) a.gn.amax[o] = amx[c][j], a.gn.amin[o] = amn[c][j];
                        }
                    }
                }
                // statistics: per-thread channel sums -> shared memory -> fixed-order group sums
                __syncthreads();
                float *S = sm, *SS = sm + COP * PG;  // [COP][PG] each
#pragma unroll
                for (int h = 0; h < CO / 2; ++h) {
                    const float2 sv = unpair(gs2[h]), qv = unpair(gss2[h]);
                    S[(ty * CO + 2 * h) * PG + tx] = sv.x, S[(ty * CO + 2 * h + 1) * PG + tx] = sv.y;
                    SS[(ty * CO + 2 * h) * PG + tx] = qv.x, SS[(ty * CO + 2 * h + 1) * PG + tx] = qv.y;
                }
                __syncthreads();
                // groups g0 .. g1 - 1 have channels in this pass; T threads
                // a group each sum every T-th of its values (its channel rows
                // of S are contiguous), then one thread a group adds the T
                // partials in order: a fixed order with short fp64 chains
                const int cpg = a.Cout / a.groups;
                const int cend = min(cobase + COP, a.Cout);
                const int g0 = cobase / cpg, g1 = (cend + cpg - 1) / cpg, ng = g1 - g0;
                int T = 1;
                while (2 * T * ng <= (int)blockDim.x && T < 64) T *= 2;
                for (int i = tid; i < ng * T; i += blockDim.x) {
                    const int g = g0 + i / T, k = i % T;
                    const int c_lo = max(cobase, g * cpg), c_hi = min(cend, (g + 1) * cpg);
                    const float *s0 = S + (c_lo - cobase) * PG, *ss0 = SS + (c_lo - cobase) * PG;
                    const int nel = (c_hi - c_lo) * PG;
                    double sv = 0.0, ssv = 0.0;
                    for (int e = k; e < nel; e += T) sv += s0[e], ssv += ss0[e];
                    gred[2 * i] = sv, gred[2 * i + 1] = ssv;
                }
                __syncthreads();
                for (int gg = tid; gg < ng; gg += blockDim.x) {
                    double sv = 0.0, ssv = 0.0;
                    for (int k = 0; k < T; ++k) sv += gred[2 * (gg * T + k)], ssv += gred[2 * (gg * T + k) + 1];
                    gpart[2 * (g0 + gg)] += sv;
                    gpart[2 * (g0 + gg) + 1] += ssv;
                }
            }
        }  // channel passes

        if (kMin) {
            // combine the CS channel slots: lowest value, then lowest channel
            __syncthreads();
            float *rv = red;
            int *ri = reinterpret_cast<int *>(red + CS * TW);
#pragma unroll
            for (int p = 0; p < kPX; ++p) rv[ty * TW + tx * kPX + p] = best[p], ri[ty * TW + tx * kPX + p] = bidx[p];
            __syncthreads();
            for (int col = tid; col < TW; col += blockDim.x) {
                const int wo = wo0 + col;
                if (wo >= a.Wo) continue;
                float bv = 0.0f;
                int bi = -1;
                for (int s = 0; s < CS; ++s) {
                    const float v = rv[s * TW + col];
                    const int i = ri[s * TW + col];
                    if (i < 0) continue;
                    const bool better = sgn >= 0 ? v < bv : v > bv;
                    if (bi < 0 || better || (v == bv && i < bi)) bv = v, bi = i;
                }
                float o = sgn == 0 ? 0.0f * bv : a.scalar * bv;
                if (KIND == CONV_EPI_MIN_TANH2) o = tanhf(tanhf(o));
                const size_t oi = ((size_t)n * a.Ho + r0) * a.Wo + wo;
                a.out[oi] = o;
                if (a.idx) a.idx[oi] = sgn == 0 ? 0 : bi;
            }
        }
    }  // pixel tiles
    }  // rows of the CTA

    if (kGN) {
        __syncthreads();
        for (int g = tid; g < a.groups; g += blockDim.x) {
            double *dst = a.gn.part + (((size_t)n * a.units + u) * a.groups + g) * 2;
            dst[0] = gpart[2 * g];
            dst[1] = gpart[2 * g + 1];
        }
    }
}

int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

struct Layout {
    int PG, CS, TW, XW, COP, ntiles;
    size_t smem;
};

// co: output channels per thread per pass (kCO, or 8 for gn_co's shapes);
// nr: input rows staged at a time
Layout layout_for(const conv_epi_desc &d, int Wo, int co = kCO, int nr = 3) {
    Layout L;
    L.PG = pow2ceil((Wo + kPX - 1) / kPX);
    if (L.PG > 64) L.PG = 64;
    const int cg = (d.Cout + co - 1) / co;
    L.CS = 256 / L.PG;
    if (L.CS > cg) L.CS = cg;
    L.TW = L.PG * kPX, L.XW = L.TW + 4;
    L.ntiles = (Wo + L.TW - 1) / L.TW;
    // fewer channel slots where narrow rows would otherwise stage more filter
    // taps than a CTA's shared memory holds (many output channels, few pixel
    // groups); the channel passes then take the rest
    for (;;) {
        L.COP = L.CS * co;
        const size_t stage = (size_t)(kCI * nr * L.XW + kCI * 9 * L.COP) * sizeof(float);
        const size_t red_min = (size_t)2 * L.CS * L.TW * sizeof(float);
        const size_t red_gn = (size_t)2 * L.COP * L.PG * sizeof(float);
        L.smem = stage;
        if (red_min > L.smem) L.smem = red_min;
        if (red_gn > L.smem) L.smem = red_gn;
        if (L.smem <= kSmemDynLimit || L.CS == 1) break;
        --L.CS;
    }
    return L;
}

// the GroupNorm chain's channels per thread: 8 where 16 would leave the
// CTA's channel slots (256 / pixel groups of them) partly empty
int gn_co(const conv_epi_desc &d, int Wo) {
    const Layout L = layout_for(d, Wo);
    return L.PG * L.CS < 256 ? 8 : kCO;
}

// The filter in the order the conv kernel stages it: pass p (output
// channels p * COP ..), then channel-tap q = ci * 9 + tap, then the pass's
// COP channels (zeros past Cout), so one input-channel step of one pass is a
// contiguous [nci * 9][COP] block.
__global__ void __launch_bounds__(256) pack_filter(const float *__restrict__ w, float *__restrict__ wp, int Cout,
                                                   int Cin, int COP, size_t total) {
    const int K = Cin * 9;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int col = (int)(i % COP);
        const size_t rq = i / COP;
        const int q = (int)(rq % K), p = (int)(rq / K);
        const int co = p * COP + col;
        wp[i] = co < Cout ? w[(size_t)co * K + q] : 0.0f;
    }
}

// wpack (bytes wbytes): the handle's buffer for the packed filter; where it
// holds this layout's packing, the filter is packed first (one more launch,
// counted by the caller) and the kernel stages from it
template <int KIND, int PK, int CO = kCO>
conv_epi_status launch(SimtArgs a, const Layout &L, int grid, cudaStream_t s, float *wpack, size_t wbytes) {
    const size_t total = (size_t)((a.Cout + L.COP - 1) / L.COP) * L.COP * a.Cin * 9;
    a.wpk = nullptr;
    if (wpack && total * sizeof(float) <= wbytes) {
        const size_t blocks = (total + 255) / 256;
        pack_filter<<<(unsigned)(blocks < 1024 ? blocks : 1024), 256, 0, s>>>(a.w, wpack, a.Cout, a.Cin, L.COP, total);
        CE_CUDA(cudaGetLastError());
        a.wpk = wpack;
    }
    auto k = simt_conv_epi<KIND, PK, CO>;
    CE_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem));
    k<<<grid, L.PG * L.CS, L.smem, s>>>(a);
    CE_CUDA(cudaGetLastError());
    return CONV_EPI_OK;
}

}  // namespace

// The GroupNorm chain runs fused in the fp32 kernel for pool_k 1, 2 or 4 and
// at most 64 groups (the kernel's pooling windows divide its 4-pixel thread
// strip; its per-CTA group sums are a 64-entry table); other GroupNorm shapes
// run as two passes, the fp32 conv into a handle-owned buffer of y and the
// chain's post-pass, which gives no window indices.
bool simt_gn_two_pass(const conv_epi_epilogue_desc &e) {
    return e.kind == CONV_EPI_GN_SCALE_POOL_CLAMP && (!(e.pool_k == 1 || e.pool_k == 2 || e.pool_k == 4) || e.groups > 64);
}

conv_epi_status simt_supported(const conv_epi_desc &d, const conv_epi_epilogue_desc &e) {
    (void)d;
    if (simt_gn_two_pass(e) && e.index_out) return CONV_EPI_ERR_UNSUPPORTED;  // the post-pass gives no indices
    return CONV_EPI_OK;
}

conv_epi_status simt_reserve(conv_epi_handle h, const conv_epi_epilogue_desc &e) {
    if (!simt_gn_two_pass(e)) return ensure_gn_workspace(h, e.pool_k, e.groups, simt_gn_units(h->d, h->Ho, e.pool_k));
    const size_t need = (size_t)h->d.N * h->d.Cout * h->Ho * h->Wo * sizeof(float);  // y
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

int simt_gn_units(const conv_epi_desc &d, int Ho, int pool_k) {
    (void)d;
    return (Ho + pool_k - 1) / pool_k;
}

namespace {

// Channels-last input for the fp32 kernel, which reads NCHW: per image, the
// [H*W][Cin] plane transposed to [Cin][H*W] through a 32 x 33 shared tile
// (coalesced reads along the channels, coalesced writes along the
// positions).
// Blocks along x run over (image, 32-position tile), along y over 32-channel
// tiles.
__global__ void __launch_bounds__(256) nhwc_to_nchw(const float *__restrict__ x, float *__restrict__ y, int C, int HW) {
    __shared__ float tile[32][33];
    const unsigned tiles = (unsigned)(HW + 31) / 32;
    const int n = (int)(blockIdx.x / tiles);
    const int p0 = (int)(blockIdx.x % tiles) * 32, c0 = blockIdx.y * 32;
    const float *src = x + (size_t)n * HW * C;
    float *dst = y + (size_t)n * C * HW;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int p = p0 + r, c = c0 + threadIdx.x;
        if (p < HW && c < C) tile[r][threadIdx.x] = src[(size_t)p * C + c];
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int c = c0 + r, p = p0 + threadIdx.x;
        if (c < C && p < HW) dst[(size_t)c * HW + p] = tile[threadIdx.x][r];
    }
}

// The same for at most 128 channels, with more bytes per block: a block
// takes TP = (4096 / C) positions rounded down to a multiple of 32 (at least
// 32), whose TP * C values are one contiguous span of x, reads the span
// straight through (16 loads a thread in flight), and writes each channel's
// run of TP positions.  The shared copy is [TP][C + 1]: for even C both
// sides are free of bank conflicts.  (Below 32 channels a 32 x 32 tile would
// also be mostly empty.)
constexpr int kNarrowC = 128, kNarrowSpan = 4096, kNarrowThreads = 256;

__host__ __device__ inline int narrow_tp(int C) { return kNarrowSpan / C / 32 * 32; }

__global__ void __launch_bounds__(kNarrowThreads)
    nhwc_to_nchw_narrow(const float *__restrict__ x, float *__restrict__ y, int C, int HW) {
    __shared__ float tile[2 * kNarrowSpan];  // TP * (C + 1) = TP * C + TP <= 4096 + 4096
    const int TP = narrow_tp(C);
    const unsigned tiles = (unsigned)(HW + TP - 1) / TP;
    const int n = (int)(blockIdx.x / tiles);
    const int p0 = (int)(blockIdx.x % tiles) * TP;
    const int np = HW - p0 < TP ? HW - p0 : TP;
    const int span = np * C;
    const float *src = x + ((size_t)n * HW + p0) * C;
    float *dst = y + (size_t)n * C * HW + p0;
    float v[kNarrowSpan / kNarrowThreads];
#pragma unroll
    for (int k = 0; k < kNarrowSpan / kNarrowThreads; ++k) {
        const int e = threadIdx.x + k * kNarrowThreads;
        if (e < span) v[k] = src[e];
    }
#pragma unroll
    for (int k = 0; k < kNarrowSpan / kNarrowThreads; ++k) {
        const int e = threadIdx.x + k * kNarrowThreads;
        if (e < span) {
            const int p = e / C, c = e - p * C;
            tile[p * (C + 1) + c] = v[k];
        }
    }
    __syncthreads();
    for (int f = threadIdx.x; f < span; f += kNarrowThreads) {
        const int c = f / np, p = f - c * np;
        dst[(size_t)c * HW + p] = tile[p * (C + 1) + c];
    }
}

}  // namespace

// bytes of the packed filter for either channel count a thread may take
size_t simt_wpack_bytes(const conv_epi_desc &d) {
    const int Wo = d.W - 2;
    size_t most = 0;
    for (int co : {kCO, 8}) {
        const Layout L = layout_for(d, Wo, co);
        const size_t n = (size_t)((d.Cout + L.COP - 1) / L.COP) * L.COP * d.Cin * 9;
        if (n > most) most = n;
    }
    return most * sizeof(float);
}

conv_epi_status simt_forward_nchw(conv_epi_handle h, const float *x, const float *w, const float *b,
                                  const conv_epi_epilogue_desc &e, float *out, cudaStream_t s);

// channels-last input: first its NCHW copy in the handle's buffer
conv_epi_status simt_forward(conv_epi_handle h, const float *x, const float *w, const float *b,
                             const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    if (d.layout != CONV_EPI_LAYOUT_NHWC) return simt_forward_nchw(h, x, w, b, e, out, s);
    const size_t need = (size_t)d.N * d.Cin * d.H * d.W * sizeof(float);
    if (!h->xpad || h->xpad_bytes < need) return CONV_EPI_ERR_INVALID_ARG;  // conv_epi_create sizes it
    if ((size_t)d.H * d.W > 0x7fffffe0u) return CONV_EPI_ERR_UNSUPPORTED;
    const int HW = d.H * d.W;
    if (d.Cin <= kNarrowC) {
        const int TP = narrow_tp(d.Cin);
        const size_t gx = (size_t)((HW + TP - 1) / TP) * d.N;
        if (gx > 0x7fffffffu) return CONV_EPI_ERR_UNSUPPORTED;
        nhwc_to_nchw_narrow<<<(unsigned)gx, kNarrowThreads, 0, s>>>(x, h->xpad, d.Cin, HW);
    } else {
        const size_t gx = (size_t)((HW + 31) / 32) * d.N, gy = (size_t)(d.Cin + 31) / 32;
        if (gx > 0x7fffffffu || gy > 65535) return CONV_EPI_ERR_UNSUPPORTED;
        nhwc_to_nchw<<<dim3((unsigned)gx, (unsigned)gy), dim3(32, 8), 0, s>>>(x, h->xpad, d.Cin, HW);
    }
    CE_CUDA(cudaGetLastError());
    const conv_epi_status st = simt_forward_nchw(h, h->xpad, w, b, e, out, s);
    if (st == CONV_EPI_OK) h->last_launches += 1;
    return st;
}

conv_epi_status simt_forward_nchw(conv_epi_handle h, const float *x, const float *w, const float *b,
                                  const conv_epi_epilogue_desc &e, float *out, cudaStream_t s) {
    const conv_epi_desc &d = h->d;
    const Layout L = layout_for(d, h->Wo);
    SimtArgs a{};
    a.x = x, a.w = w, a.b = b;
    a.N = d.N, a.Cin = d.Cin, a.H = d.H, a.W = d.W, a.Cout = d.Cout, a.Ho = h->Ho, a.Wo = h->Wo;
    a.PG = L.PG, a.CS = L.CS, a.ntiles = L.ntiles;
    a.scalar = e.scalar, a.chan_scale = e.chan_scale, a.slope = e.lrelu_slope;
    a.groups = e.groups;
    a.out = out, a.idx = e.index_out;
    // several rows per CTA only where they reuse the staged filter (one
    // input-channel step and one output-channel pass); otherwise one row per
    // CTA keeps more CTAs in flight (measured: 4 rows cost C3/C4 3-4%)
    a.rpc = (d.Cin <= kCI && d.Cout <= L.COP) ? kRowsPerCta : 1;
    a.xrows = 3;
    a.ring = 0;
    // the min and per-channel chains with several rows per CTA and one pixel
    // tile keep the input rows in a ring of four slots (the layout unchanged,
    // the filter staged once, and the tiles plus the min chain's scratch still
    // two CTAs to an SM)
    Layout LL = L;
    if (e.kind != CONV_EPI_GN_SCALE_POOL_CLAMP && a.rpc > 1) {
        const Layout Lr = layout_for(d, h->Wo, kCO, 4);
        const int x4 = kCI * 4 * Lr.XW;
        const bool w_once = d.Cin <= kCI && d.Cout <= Lr.COP && 2 * Lr.CS * Lr.TW <= x4 && 2 * Lr.COP * Lr.PG <= x4;
        const size_t smem = (size_t)(x4 + kCI * 9 * Lr.COP + 2 * Lr.CS * Lr.TW) * sizeof(float);
        if (w_once && Lr.ntiles == 1 && Lr.CS == L.CS && smem <= kBandSmemLimit) {
            a.ring = 1, a.xrows = 4;
            LL = Lr;
            LL.smem = smem;
        }
    }
    const int packs = h->wpack ? 1 : 0;  // the filter-pack launch before the conv kernel
    conv_epi_status st;
    switch (e.kind) {
    case CONV_EPI_MIN_TANH2:
        a.units = (h->Ho + a.rpc - 1) / a.rpc;
        st = launch<CONV_EPI_MIN_TANH2, 1>(a, LL, d.N * a.units, s, h->wpack, h->wpack_bytes);
        break;
    case CONV_EPI_SCALE_MIN:
        a.units = (h->Ho + a.rpc - 1) / a.rpc;
        st = launch<CONV_EPI_SCALE_MIN, 1>(a, LL, d.N * a.units, s, h->wpack, h->wpack_bytes);
        break;
    case CONV_EPI_MUL_LRELU_GELU:
        a.units = (h->Ho + a.rpc - 1) / a.rpc;
        st = launch<CONV_EPI_MUL_LRELU_GELU, 1>(a, LL, d.N * a.units, s, h->wpack, h->wpack_bytes);
        break;
    case CONV_EPI_NONE:
        a.units = (h->Ho + a.rpc - 1) / a.rpc;
        st = launch<CONV_EPI_NONE, 1>(a, LL, d.N * a.units, s, h->wpack, h->wpack_bytes);
        break;
    case CONV_EPI_GN_SCALE_POOL_CLAMP: {
        if (simt_gn_two_pass(e)) {
            // the conv output into the handle's buffer, then the chain's post-pass
            if (!h->ybuf || h->ybuf_bytes < (size_t)d.N * d.Cout * h->Ho * h->Wo * sizeof(float))
                return CONV_EPI_ERR_INVALID_ARG;  // conv_epi_reserve sizes it
            conv_epi_epilogue_desc plain{};
            plain.kind = CONV_EPI_NONE;
            if ((st = simt_forward_nchw(h, x, w, b, plain, h->ybuf, s))) return st;
            const int conv_launches = h->last_launches;
            if ((st = postpass_forward(h, h->ybuf, e, out, s))) return st;
            h->last_launches += conv_launches;
            return CONV_EPI_OK;
        }
        a.units = simt_gn_units(d, h->Ho, e.pool_k);
        a.gn = h->gn;
        a.Hp = h->gn.Hp, a.Wp = h->gn.Wp;
        if (h->gn.units != a.units) return CONV_EPI_ERR_INVALID_ARG;
        constexpr int GN = CONV_EPI_GN_SCALE_POOL_CLAMP;
        const int grid = d.N * a.units;
        const int co = gn_co(d, h->Wo);
        // a band's input rows staged once where one input-channel step, one
        // channel pass and one pixel tile cover it, the layout stays the
        // same and two CTAs still fit an SM's shared memory
        {
            const Layout L3 = layout_for(d, h->Wo, co), Lb = layout_for(d, h->Wo, co, e.pool_k + 2);
            if (e.pool_k > 1 && d.Cin <= kCI && d.Cout <= Lb.COP && Lb.ntiles == 1 && Lb.CS == L3.CS &&
                Lb.smem <= kBandSmemLimit)
                a.xrows = e.pool_k + 2;
        }
        if (co == 8) {
            const Layout L8 = layout_for(d, h->Wo, 8, a.xrows);
            a.PG = L8.PG, a.CS = L8.CS, a.ntiles = L8.ntiles;
            if (e.pool_k == 4) st = launch<GN, 4, 8>(a, L8, grid, s, h->wpack, h->wpack_bytes);
            else if (e.pool_k == 2) st = launch<GN, 2, 8>(a, L8, grid, s, h->wpack, h->wpack_bytes);
            else st = launch<GN, 1, 8>(a, L8, grid, s, h->wpack, h->wpack_bytes);
        } else {
            const Layout L16 = layout_for(d, h->Wo, kCO, a.xrows);
            a.PG = L16.PG, a.CS = L16.CS, a.ntiles = L16.ntiles;
            if (e.pool_k == 4) st = launch<GN, 4>(a, L16, grid, s, h->wpack, h->wpack_bytes);
            else if (e.pool_k == 2) st = launch<GN, 2>(a, L16, grid, s, h->wpack, h->wpack_bytes);
            else st = launch<GN, 1>(a, L16, grid, s, h->wpack, h->wpack_bytes);
        }
        if (st) return st;
        h->last_launches = 1 + packs;
        st = gn_finalize(h, e, out, s, false);
        if (st == CONV_EPI_OK) h->last_launches = 2 + packs;
        return st;
    }
    default:
        return CONV_EPI_ERR_INVALID_ARG;
    }
    if (st == CONV_EPI_OK) h->last_launches = 1 + packs;
    return st;
}

}  // namespace conv_epi
