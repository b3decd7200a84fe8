// tl_kernels.cu -- sm_103a kernels and the device half of the C ABI.
//
// What runs here (Neutrino-1 pages):
//   * ternary weights {-1, 0, +1} with one scale per output row and the
//     signed sum "state times scale" (blog "Neutrino-1: quantization is a
//     training decision", "What's actually ternary");
//   * weights decoded inside the matrix kernel, never stored as fp16/fp32
//     (model page "Neutrino-1 8B", "Overview");
//   * single-stream decode is bound by bytes moved per token (blog, "Serving
//     it: the Neutrino Engine"), so the N <= 8 kernel is built to stream the
//     2-bit codes at HBM rate;
//   * speculative verify: up to seven drafted tokens checked in one batched
//     pass (wiki "Neutrino-1", "What is actually new"), hence N <= 8 columns
//     of one mma n8 tile.
//
// Kernel tl_mma_kernel (N <= 8, modes A and B):
//   Work.  K is cut into as few slices of at most kMaxSlice 128-column
//   blocks as it needs.  The launch's (16-row tile, block) units are ordered
//   slice by slice, then row tile by row tile; each slice has its own Pps
//   CTAs, and CTA c owns a contiguous range of Lc units of slice c / Pps, so
//   the CTAs of a slice stream the same number of bytes, each stages the
//   activations of one slice only, and a (row tile, slice) piece spans at
//   most two CTAs; a one-slice launch gives each CTA whole row tiles.  One
//   CTA of 16 warps per SM; the warps split the CTA's units into contiguous
//   ranges.
//   Weights.  Each warp streams its units with cp.async.bulk into its own
//   ring of shared-memory slots (up to 10 tiles per copy, completing on the
//   slot's mbarrier), running ahead across slices.  A TL2P v2 tile is in
//   mma.m16n8k16 A-fragment order and each 2-bit field holds 1 - w, so
//   register j of k-step m is (word >> 8*(m/4)) & (0x00030003 << 2*(m%4)):
//   a bf16x2 pair whose halves are (1 - w) * 2^(2q - 133), q = m%4 -- bf16
//   subnormals (or, for field 10 at q == 3, the smallest normal), exactly
//   linear in the field.  One AND per two weights, plus one shift per word.
//   Activations.  Staged per slice in shared memory in B-fragment order; the
//   k-steps of class q = m % 4 are multiplied by 2^(67 - 2q) (a bf16 product
//   by a power of two, exact), so every product is (1 - w) * x * 2^-66,
//   exact in fp32.
//   The staging also sums x over each half block (64 columns).  A tile's
//   k-steps 0..3 and 4..7 go to two accumulator chains, alternating, and the
//   next tile to two others; before its MMAs each chain is given minus its
//   half block's sum, so a chain holds -sum w x (scaled) and its rounding
//   tracks the result rather than sum x, whatever the mean of x.  The chains
//   are folded, with exact power-of-two factors, when a run of tiles ends.
//   Activations outside [2^-60, 2^61) in magnitude (mode A only) switch that
//   token's slice to a scale chosen from its largest exponent.  Columns
//   n >= N are zero and their results are discarded, so no lane is
//   predicated off.  The int8 mode that quantises inside the launch stages
//   each token's quantised integers the same way (kQ).
//   Reduction.  A warp that covers all of a row tile's units in a slice adds
//   its sum straight into the CTA's row accumulator (shared memory); rows
//   split between warps go through per-warp boundary slots that are added in
//   warp order after the slice.  A row tile whose pieces sit in several CTAs
//   is finished by whichever CTA completes it (workspace counter), adding the
//   pieces in a fixed order.  The plan never depends on N, and the power-of-
//   two scaling does not change any rounding, so every token's result is
//   bitwise independent of the batch.

#include "tl.h"
#include "tl_internal.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

namespace {

constexpr int kWarps = 16;            // warps per CTA of the N <= 8 kernel
constexpr int kCtasPerSm = 1;         // resident CTAs per SM (registers allow 1)
// CTAs per SM in a launch's grid.
constexpr int kGridPerSm = 1;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 2;             // bulk copies in flight per warp
// Tiles (512 B each) per bulk copy: 10 at one or two tokens, 8 at four and
// 6 at eight, as the staged activations (up to 64 KB) leave room.
__host__ __device__ constexpr int chunk_tiles(int nt) { return nt <= 2 ? 10 : nt == 4 ? 8 : 6; }
__host__ __device__ constexpr int ring_bytes(int nt) { return kWarps * kSlots * chunk_tiles(nt) * 512; }
constexpr int kNMax = 8;              // tokens per launch (mma n = 8)
constexpr int kMaxDevices = 64;
constexpr int kMaxSlice = 32;         // 128-column blocks per K slice (64 KB of X at 8 tokens)
constexpr int kMaxCtaRows = 32;       // row tiles one CTA may touch in one slice (kThreads / 16)
// 16-byte activation loads in flight per thread while staging a slice: all
// of a slice at once, up to 8 (4 at eight tokens, where more registers spill).
__host__ __device__ constexpr int stage_batch(int nt, bool mode_a) {
    return (nt * kMaxSlice * (mode_a ? 16 : 8) + kThreads - 1) / kThreads < (nt == 8 ? 4 : 8)
               ? (nt * kMaxSlice * (mode_a ? 16 : 8) + kThreads - 1) / kThreads
               : (nt == 8 ? 4 : 8);
}
constexpr long long kWaitLimit = 1ll << 31;   // SM cycles before a wait gives up
// Activations are staged times 2^kT: a k-step class q product is then
// (1 - w) * x * 2^(2q - 66), a normal fp32 number for |x| in [2^-60, 2^61).
constexpr int kT = 67;
constexpr int kWinLo = 127 - 60;      // bf16 exponent fields of the fixed-scale window
constexpr int kWinHi = 127 + 60;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes (or the hint expires) instead of spinning.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; false (and the status word set) when it gives up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *status) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (clock64() - t0 > kWaitLimit) {
            atomicExch(status, TL_DEVERR_TIMEOUT);
            return false;
        }
    }
    return true;
}
// One bulk copy global -> shared, completing `bytes` on the slot's mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------ work geometry
// Units are ordered slice by slice, then row tile, then block:
// u = sigma*R*KW + r*kw(sigma) + b, with kw(sigma) the slice's width (KW for
// every slice but the last, which is KWL wide).

// n / d for 0 <= n < 2^31 as (umulhi(n, m) + n) >> s (m, s from the host).
struct FastDiv {
    uint32_t m, s;
};
__device__ __forceinline__ int fdiv(int n, FastDiv d) {
    return (int)(((unsigned long long)__umulhi((uint32_t)n, d.m) + (uint32_t)n) >> d.s);
}

struct Slice {
    int sigma, kb0, kw;     // slice, its first block, its width in blocks
    int a0, a1;             // the CTA's units of the slice, slice-local
    int r_first, r_last;    // row tiles touched (r_last < r_first: none)
    int lo_first, hi_last;  // first block of r_first, one past the last block of r_last
};

// A warp's position: slice-local unit u of its range [u, uend) in slice
// sigma, at row tile r, block b (slice-local) of a slice kw blocks wide.
struct Cursor {
    int sigma, u, uend, r, b, kw, kb0;
};

// Kinds of step in a chain of launches run by one persistent kernel.
constexpr int kStepLinear = 0;   // a (grouped) ternary linear
constexpr int kStepQuant = 1;    // per-token activation quantisation (mode B chains)

// Everything below reads these launch constants.
struct GroupArgs {
    int kind;       // kStepLinear or kStepQuant
    int P;          // CTAs that take part (the plan's; chunks x tokens for a quantiser step)
    int kwr, rowsr; // shared-memory regions: slice width and row tiles they are sized for
    const char *packed[TL_MAX_GROUP];
    const float *scale[TL_MAX_GROUP];
    const int32_t *rowsum[TL_MAX_GROUP];
    void *Y[TL_MAX_GROUP];
    int M[TL_MAX_GROUP];
    int rt_off[TL_MAX_GROUP + 1];   // row-tile prefix over the group
    int G;
    int R;          // row tiles in the launch
    int KB;         // 128-column blocks
    int KW;         // blocks per K slice
    int KWL;        // blocks of the last slice
    int NS;         // slices
    int K;
    int U;          // units = R * KB
    int Pps;        // CTAs per slice: CTA c works in slice c / Pps only
    int Lc;         // units per CTA in a full slice (the slice's last CTAs may get fewer)
    int LcL;        // units per CTA in the last slice
    int rows;       // accumulator rows per CTA
    FastDiv dKW, dKWL;
    const void *X;  // bf16 [N][K] (mode A) or int8 [N][K] (mode B)
    const float *s;
    const int32_t *z;
    int N;
    int mode;
    int out;
    int xvec;       // X rows allow 16-byte loads (16-byte aligned, K a multiple of 8 / 16)
    float *part;    // pieces of row tiles finished across CTAs [R][NS][2][N][16] (NS > 1)
    unsigned long long *cnt;  // [R] blocks arrived (NS > 1); zero between launches
    unsigned long long *xslot;  // [R][N][16] exchange slots (NS == 1); zero between launches
    int *status;    // workspace status word
    // quantiser steps: X (bf16) -> qout (int8), sout, zout; symmetric if sym
    int8_t *qout;
    float *sout;
    int32_t *zout;
    int sym;
};

// Header of an encoded chain (device memory), followed by its steps.
struct ChainHeader {
    unsigned long long *cnt;    // [nsteps] CTAs done per step, over all passes so far
    unsigned long long *epoch;  // passes completed; [1] counts CTAs leaving the current pass
    const unsigned *gate;   // when not null, step 0 waits until *gate != 0
    long long wait_limit;   // SM cycles before a wait for a step's inputs gives up
    int nsteps;
    int lookahead;          // steps whose weights are prefetched into L2 ahead of use
};

__device__ __forceinline__ int slice_width(const GroupArgs &a, int sigma) {
    return sigma == a.NS - 1 ? a.KWL : a.KW;
}

__device__ __forceinline__ void slice_of(const GroupArgs &a, int cu0, int cu1, int sigma,
                                         Slice &p) {
    p.sigma = sigma;
    p.kb0 = sigma * a.KW;
    p.kw = slice_width(a, sigma);
    const FastDiv dv = sigma == a.NS - 1 ? a.dKWL : a.dKW;
    const int base = sigma * a.R * a.KW;
    p.a0 = max(cu0, base) - base;
    p.a1 = min(cu1, base + a.R * p.kw) - base;
    if (p.a1 > p.a0) {
        p.r_first = fdiv(p.a0, dv);
        p.r_last = fdiv(p.a1 - 1, dv);
        p.lo_first = p.a0 - p.r_first * p.kw;
        p.hi_last = p.a1 - p.r_last * p.kw;
    } else {
        p.r_first = 0; p.r_last = -1; p.lo_first = 0; p.hi_last = 0;
    }
}

// Blocks [lo, hi) of row tile r that the CTA covers in slice p.
__device__ __forceinline__ void row_span(const Slice &p, int r, int &lo, int &hi) {
    lo = r == p.r_first ? p.lo_first : 0;
    hi = r == p.r_last ? p.hi_last : p.kw;
}

// Whether the (row tile r, slice sigma) piece is cut by a CTA boundary (the
// slice's CTAs own consecutive ranges of lc units from the slice's start).
__device__ __forceinline__ bool piece_split(const GroupArgs &a, int r, int sigma) {
    const int kw = slice_width(a, sigma);
    const int lc = sigma == a.NS - 1 ? a.LcL : a.Lc;
    const int u0 = r * kw;
    return u0 / lc != (u0 + kw - 1) / lc;
}

// Move c to warp w's first unit in slice c.sigma or a later one before
// sig_end; false when the warp has no units left.
__device__ __forceinline__ bool cursor_enter(const GroupArgs &a, int cu0, int cu1, int sig_end,
                                             int w, Cursor &c) {
    for (; c.sigma < sig_end; ++c.sigma) {
        c.kb0 = c.sigma * a.KW;
        c.kw = slice_width(a, c.sigma);
        const int base = c.sigma * a.R * a.KW;
        const int a0 = max(cu0, base) - base, a1 = min(cu1, base + a.R * c.kw) - base;
        const int np = a1 - a0;
        if (np <= 0) continue;
        const int lw = (np + kWarps - 1) / kWarps;
        c.u = a0 + min(w * lw, np);
        c.uend = a0 + min(w * lw + lw, np);
        if (c.u < c.uend) {
            c.r = fdiv(c.u, c.sigma == a.NS - 1 ? a.dKWL : a.dKW);
            c.b = c.u - c.r * c.kw;
            return true;
        }
    }
    return false;
}

// Matrix of the group that holds row tile r, and r's first tile.
__device__ __forceinline__ const char *row_base(const GroupArgs &a, int r, int &gi) {
    gi = 0;
    while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
    return a.packed[gi] + (long long)(r - a.rt_off[gi]) * a.KB * 512;
}

// ------------------------------------------------------------ epilogue
// Y[n][m] from acc = sum_k w*x (mode A) or the exact integer sum_k w*q (mode
// B); sc = scale[m], rs = rowsum[m].
__device__ __forceinline__ void store_out(const GroupArgs &a, int gi, int m, int n, float acc,
                                          float sc, int rs, const float *ts, const int32_t *tz) {
    const int M = a.M[gi];
    float y;
    if (a.mode == TL_MODE_BF16) {
        y = __fmul_rn(acc, sc);
    } else {
        const int iacc = __float2int_rn(acc);
        if (a.out == TL_OUT_I32_RAW) {
            reinterpret_cast<int32_t *>(a.Y[gi])[(long long)n * M + m] = iacc;
            return;
        }
        const int corrected = iacc - tz[n] * rs;
        y = __fmul_rn(__fmul_rn((float)corrected, ts[n]), sc);
    }
    if (a.out == TL_OUT_F32)
        reinterpret_cast<float *>(a.Y[gi])[(long long)n * M + m] = y;
    else
        reinterpret_cast<__nv_bfloat16 *>(a.Y[gi])[(long long)n * M + m] = __float2bfloat16_rn(y);
}

// The 16 x N results of row tile r held as v[n * 16 + row], with the row
// tile's scales and row sums in sc[16], rs[16] and (integer modes) the
// tokens' steps and zero points in ts, tz.  One warp; lane (g, t) stores
// rows g, g+8 of tokens 2t, 2t+1.
__device__ __forceinline__ void store_row_tile(const GroupArgs &a, int r, const float *v,
                                               const float *sc, const int *rs, const float *ts,
                                               const int32_t *tz, int lane) {
    const int g = lane >> 2, t = lane & 3;
    int gi = 0;
    while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
    const int rl = r - a.rt_off[gi];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = g + 8 * h, m = rl * 16 + i, n = 2 * t + e;
            if (m < a.M[gi] && n < a.N) store_out(a, gi, m, n, v[n * 16 + i], sc[i], rs[i], ts, tz);
        }
}

// Row tile r of a one-slice launch whose blocks are split between two CTAs:
// each CTA swaps its piece of every element into the element's exchange slot
// (bit 32 set = occupied).  The CTA that finds the other piece there adds the
// two, stores the element and empties the slot; the other finds the slot
// empty and is done.  One atomic round trip, and the sum does not depend on
// which CTA comes second (a + b == b + a in floating point).
__device__ __forceinline__ void exchange_row_tile(const GroupArgs &a, int r, const float *v,
                                                  const float *sc, const int *rs, const float *ts,
                                                  const int32_t *tz, int lane) {
    const int g = lane >> 2, t = lane & 3;
    int gi = 0;
    while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
    const int rl = r - a.rt_off[gi];
    unsigned long long *slot = a.xslot + (long long)r * a.N * 16;
    // every swap in flight before any result is used
    unsigned long long old[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = g + 8 * h, n = 2 * t + e;
            old[h][e] = n < a.N ? atomicExch(slot + n * 16 + i,
                                             (1ull << 32) | __float_as_uint(v[n * 16 + i]))
                                : 0ull;
        }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = g + 8 * h, m = rl * 16 + i, n = 2 * t + e;
            if (old[h][e] >> 32) {
                slot[n * 16 + i] = 0ull;
                if (m < a.M[gi])
                    store_out(a, gi, m, n,
                              __fadd_rn(__uint_as_float((uint32_t)old[h][e]), v[n * 16 + i]),
                              sc[i], rs[i], ts, tz);
            }
        }
}

// One 128-column block of one 16-row tile: 8 MMAs (k-steps m = 0..7) over
// the lane's 16-byte slice of the tile (w) and the 4 B-fragment quarters (b),
// k-steps 0..3 into chain c0 and 4..7 into c1, alternating so that
// consecutive MMAs never share an accumulator.  Register j of k-step m is
// word j shifted right by 8*(m/4) and masked to the fields at bits 2*(m%4)
// and 16 + 2*(m%4).
__device__ __forceinline__ void tile_mma(float (&c0)[4], float (&c1)[4], const uint4 &w,
                                         const uint4 (&b)[4]) {
    const uint32_t hx = w.x >> 8, hy = w.y >> 8, hz = w.z >> 8, hw = w.w >> 8;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t F = 0x00030003u << (2 * p);
        const uint4 &q0 = b[p >> 1], &q1 = b[2 + (p >> 1)];
        mma_bf16_16816(c0, w.x & F, w.y & F, w.z & F, w.w & F, (p & 1) ? q0.z : q0.x,
                       (p & 1) ? q0.w : q0.y);
        mma_bf16_16816(c1, hx & F, hy & F, hz & F, hw & F, (p & 1) ? q1.z : q1.x,
                       (p & 1) ? q1.w : q1.y);
    }
}

// Position of the (block b, token n, half h) correction of a slice: the
// tokens 2t', 2t'+1 of both halves of a block are four consecutive floats,
// so lane (g, t) reads its tile's corrections with one 16-byte load (8 bytes
// at one token).
template <int NT>
__device__ __forceinline__ int xh_index(int b, int n, int h) {
    return NT == 1 ? b * 2 + h : ((b * (NT / 2) + (n >> 1)) * 2 + h) * 2 + (n & 1);
}
// One tile on chains c[2 par] (k-steps 0..3) and c[2 par + 1] (k-steps
// 4..7), each first given its half block's correction (xc: the lane's four
// floats, half 0 then half 1, tokens 2t', 2t'+1 each; two floats at one
// token, where only column 0 is kept).  The chains then hold
// sum (1 - w) x - sum x = -sum w x, scaled, and never grow with sum x.
template <int NT>
__device__ __forceinline__ void tile_corrected(float (&c)[4][4], int par, const uint4 &w,
                                               const uint4 (&b)[4], const float *xc) {
    float(&c0)[4] = c[2 * par];
    float(&c1)[4] = c[2 * par + 1];
    if (NT == 1) {
        const float2 cr = *reinterpret_cast<const float2 *>(xc);
        c0[0] = __fadd_rn(c0[0], cr.x);
        c0[2] = __fadd_rn(c0[2], cr.x);
        c1[0] = __fadd_rn(c1[0], cr.y);
        c1[2] = __fadd_rn(c1[2], cr.y);
    } else {
        const float4 cr = *reinterpret_cast<const float4 *>(xc);
        c0[0] = __fadd_rn(c0[0], cr.x);
        c0[1] = __fadd_rn(c0[1], cr.y);
        c0[2] = __fadd_rn(c0[2], cr.x);
        c0[3] = __fadd_rn(c0[3], cr.y);
        c1[0] = __fadd_rn(c1[0], cr.z);
        c1[1] = __fadd_rn(c1[1], cr.w);
        c1[2] = __fadd_rn(c1[2], cr.z);
        c1[3] = __fadd_rn(c1[3], cr.w);
    }
    tile_mma(c0, c1, w, b);
}

// -sum * 2^(T - 133), in two exact power-of-two factors: the correction, in
// chain units, for half a block whose activations sum to `sum` and are
// staged times 2^(T - 2q).
__device__ __forceinline__ float chain_units(float sum, int T) {
    const int d = T - 133, d1 = d / 2;
    return -__fmul_rn(__fmul_rn(sum, __int_as_float((d1 + 127) << 23)),
                      __int_as_float((d - d1 + 127) << 23));
}

// VPL consecutive activations of token n from column k0 (VPL = 8 bf16 in mode
// A, 16 int8 in mode B; k0 a multiple of VPL): one 16-byte load when X allows
// it, else element loads; columns >= K read as 0.  In a chain (kL2) the
// loads skip the SM's L1, since X may have been written by other SMs during
// the launch; a launch of its own reads X written by an earlier kernel and
// may share it through L1 with the SM's other CTA.
template <bool kL2>
__device__ __forceinline__ uint4 ldx(const uint4 *p) { return kL2 ? __ldcg(p) : __ldg(p); }
template <bool kL2>
__device__ __forceinline__ uint16_t ldx16(const uint16_t *p) { return kL2 ? __ldcg(p) : __ldg(p); }
template <bool kL2>
__device__ __forceinline__ uint8_t ldx8(const uint8_t *p) { return kL2 ? __ldcg(p) : __ldg(p); }
template <bool kModeA, bool kL2>
__device__ __forceinline__ uint4 load_group(const GroupArgs &a, int n, int k0) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (kModeA) {
        const uint16_t *x = reinterpret_cast<const uint16_t *>(a.X) + (long long)n * a.K + k0;
        if (a.xvec) {
            if (k0 < a.K) v = ldx<kL2>(reinterpret_cast<const uint4 *>(x));
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (k0 + e < a.K) w[e >> 1] |= (uint32_t)ldx16<kL2>(x + e) << (16 * (e & 1));
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        const uint8_t *x = reinterpret_cast<const uint8_t *>(a.X) + (long long)n * a.K + k0;
        if (a.xvec) {
            if (k0 < a.K) v = ldx<kL2>(reinterpret_cast<const uint4 *>(x));
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (k0 + e < a.K) w[e >> 2] |= (uint32_t)ldx8<kL2>(x + e) << (8 * (e & 3));
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    return v;
}

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16f(uint32_t h) { return __uint_as_float(h << 16); }
// x * 2^d for any bf16 x through fp32 (two exact power-of-two products).
__device__ __forceinline__ uint32_t scale_any(uint32_t h, int d) {
    const int d1 = d / 2, d2 = d - d1;
    const float f = __fmul_rn(__fmul_rn(bf16f(h), __int_as_float((d1 + 127) << 23)),
                              __int_as_float((d2 + 127) << 23));
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// dst[4 * tt] = w[tt] for tt = 0..3, written in the order tt = (it + q) % 4.
__device__ __forceinline__ void store_rotated(uint32_t *dst, const uint32_t (&w)[4], int q) {
    const bool r1 = q & 1, r2 = q & 2;
    const uint32_t a0 = r1 ? w[1] : w[0], a1 = r1 ? w[2] : w[1];
    const uint32_t a2 = r1 ? w[3] : w[2], a3 = r1 ? w[0] : w[3];
    const uint32_t b0 = r2 ? a2 : a0, b1 = r2 ? a3 : a1, b2 = r2 ? a0 : a2, b3 = r2 ? a1 : a3;
    dst[4 * (q & 3)] = b0;
    dst[4 * ((q + 1) & 3)] = b1;
    dst[4 * ((q + 2) & 3)] = b2;
    dst[4 * ((q + 3) & 3)] = b3;
}

// One staging group: activation group o (8 bf16 in mode A, 16 int8 in mode
// B, as one 16-byte word x) of token n in a block whose staged words start
// at blk.  Writes the group's words in B-fragment order, times 2^(kT - 2q)
// for k-step class q = m % 4 (the A operand of class q carries 2^(2q - 133),
// so every product is w-field * x * 2^(kT - 133)), and returns the group's
// sum in a fixed order and (mode A) the mask of halves outside the fixed
// window.  A zero x writes zeros.
// kQ: the group is 8 bf16 activations that are first quantised with the
// token's step s (r = 1/s) and zero point z, exactly as the quantiser
// kernel does; the codes are then staged and summed like mode B's.
template <bool kModeA, int NT, bool kQ = false>
__device__ __forceinline__ void stage_group(uint32_t *blk, int n, int o, const uint4 &x,
                                            float &sum, uint32_t &bad, const float *qs = nullptr,
                                            const float *qr = nullptr, const int *qz = nullptr,
                                            int sym = 0) {
    const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
    sum = 0.f;
    bad = 0u;
    if (kQ) {
        const int m = o >> 1, qd = m >> 1;
        const float f = __int_as_float((kT - 2 * (m & 3) + 127) << 23);
        const float sv = qs[n], rv = qr[n], zf = (float)qz[n], qlo = sym ? -127.f : -128.f;
        uint32_t *dst = blk + (qd * NT + n) * 16 + 2 * (m & 1) + (o & 1);
        uint32_t st[4];
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
            const float x0 = __uint_as_float(wd[tt] << 16), x1 = __uint_as_float(wd[tt] & 0xFFFF0000u);
            const float q0 = fminf(fmaxf(__fadd_rn(tl_internal::quant_round(x0, sv, rv), zf), qlo), 127.f);
            const float q1 = fminf(fmaxf(__fadd_rn(tl_internal::quant_round(x1, sv, rv), zf), qlo), 127.f);
            sum = __fadd_rn(sum, __fadd_rn(q0, q1));   // integers: exact
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(q0, f), __fmul_rn(q1, f));
            st[tt] = *reinterpret_cast<const uint32_t *>(&b2);
        }
        store_rotated(dst, st, qd);
    } else if (kModeA) {
        const int m = o >> 1, qd = m >> 1;
        // 2^(kT - 2q) in both halves: an exact bf16 product for values in the
        // window (and zero stays zero)
        const uint32_t e2 = (uint32_t)(kT - 2 * (m & 3) + 127) * 0x00800080u;
        const __nv_bfloat162 sc2 = *reinterpret_cast<const __nv_bfloat162 *>(&e2);
        uint32_t *dst = blk + (qd * NT + n) * 16 + 2 * (m & 1) + (o & 1);
        uint32_t st[4];
        // Per 16-bit half, with mag = |bits|: bit 15 of mag + kUp is set when
        // the exponent field is above kWinHi, bit 15 of kLo - mag when mag is
        // below the window, bit 15 of mag + 0x7FFF when mag is not zero (no
        // carry or borrow crosses the halves).
        constexpr uint32_t kUp = (0x8000u - ((uint32_t)(kWinHi + 1) << 7)) * 0x00010001u;
        constexpr uint32_t kLo = (0x8000u + ((uint32_t)kWinLo << 7) - 1u) * 0x00010001u;
        uint32_t flags = 0u;
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
            const uint32_t v = wd[tt];
            sum = __fadd_rn(__fadd_rn(sum, __uint_as_float(v << 16)),
                            __uint_as_float(v & 0xFFFF0000u));
            const uint32_t mag = v & 0x7FFF7FFFu;
            flags |= (mag + kUp) | ((kLo - mag) & (mag + 0x7FFF7FFFu));
            const __nv_bfloat162 p2 = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&v), sc2);
            st[tt] = *reinterpret_cast<const uint32_t *>(&p2);
        }
        bad = flags & 0x80008000u;
        // store word tt = (it + qd) % 4 at step it: the lanes of one block
        // quarter apart then write different banks
        store_rotated(dst, st, qd);
    } else {
        const int m = o, qd = m >> 1;
        uint32_t *dst = blk + (qd * NT + n) * 16 + 2 * (m & 1);
        const float two_t = __int_as_float((kT - 2 * (m & 3) + 127) << 23);
        int isum = 0;
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
            uint32_t st[4];
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                const uint32_t word = wd[2 * h8 + (tt >> 1)] >> (16 * (tt & 1));
                const int qlo = (int)(int8_t)(word & 0xFFu);
                const int qhi = (int)(int8_t)((word >> 8) & 0xFFu);
                isum += qlo + qhi;
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn((float)qlo, two_t),
                                                                __fmul_rn((float)qhi, two_t));
                st[tt] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            store_rotated(dst + h8, st, qd);
        }
        sum = (float)isum;
    }
}

// The activation groups of one slice: VPL activations per group, LB groups
// per 128-column block, N * kw * LB groups in all, taken SB * kThreads at a
// time starting at `base`.
template <bool kModeA, int SB, bool kL2>
__device__ __forceinline__ void stage_load(const GroupArgs &a, const Slice &P, int base,
                                           uint4 (&v)[SB]) {
    constexpr int VPL = kModeA ? 8 : 16;
    constexpr int LB = 128 / VPL;
    const int total = a.N * P.kw * LB;
    const FastDiv dv = P.sigma == a.NS - 1 ? a.dKWL : a.dKW;
#pragma unroll
    for (int i = 0; i < SB; ++i) {
        const int idx = base + i * kThreads + (int)threadIdx.x;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < total) {
            const int q = idx / LB, o = idx % LB;     // q = n * kw + jb
            const int n = fdiv(q, dv), jb = q - n * P.kw;
            v[i] = load_group<kModeA, kL2>(a, n, (P.kb0 + jb) * 128 + o * VPL);
        }
    }
}

// ------------------------------------------------------------ weight pipeline
// Each warp streams its units into a ring of kSlots shared-memory slots:
// lane 0 issues one bulk copy of up to CH tiles per slot, completing on the
// slot's mbarrier, and all lanes consume the slots in the same order.  In a
// chain of linears the producer runs on into the next step's units while the
// warp still works on the current step, so weights keep arriving across the
// wait for the step's inputs.
struct Pipe {
    uint32_t ring_w, bar_w;  // this warp's ring and barriers (shared-window addresses)
    int slot;                // next slot to consume
    uint32_t phases;         // parity to wait for, one bit per slot
    uint32_t inflight;       // (lane 0) slots with a copy in flight
    // (lane 0) the next chunk to copy: step pstep, cursor pc
    const GroupArgs *steps;
    int nsteps, pstep;
    int pcu0, pcu1, psig1;   // this CTA's units of step pstep
    Cursor pc;
    int pgi;
    const char *prow;
    bool pc_on;
};

// This CTA's units of a launch -- a contiguous range of one slice, none for
// CTAs past the plan's -- and the slices [sig0, sig1) it touches.
__device__ __forceinline__ void cta_units(const GroupArgs &a, int cta, int &cu0, int &cu1,
                                          int &sig0, int &sig1) {
    cu0 = cu1 = a.U;
    const int sig_c = cta / a.Pps, c_in = cta - sig_c * a.Pps;
    if (sig_c < a.NS) {
        const int su = a.R * slice_width(a, sig_c);
        const int lc = sig_c == a.NS - 1 ? a.LcL : a.Lc;
        const int base = sig_c * a.R * a.KW;
        const int off = (int)min((long long)c_in * lc, (long long)su);
        cu0 = base + off;
        cu1 = base + min(off + lc, su);
    }
    const int sunits = a.R * a.KW;
    sig0 = cu0 / sunits;
    sig1 = cu1 > cu0 ? (cu1 - 1) / sunits + 1 : sig0;
}

// Producer: move to the first linear step from p.pstep on in which this
// warp has units.
__device__ __forceinline__ void pipe_seek(Pipe &p, int cta, int warp) {
    for (; p.pstep < p.nsteps; ++p.pstep) {
        const GroupArgs &a = p.steps[p.pstep];
        if (a.kind != kStepLinear || cta >= a.P) continue;
        int sig0;
        cta_units(a, cta, p.pcu0, p.pcu1, sig0, p.psig1);
        p.pc.sigma = sig0;
        if (cursor_enter(a, p.pcu0, p.pcu1, p.psig1, warp, p.pc)) {
            p.prow = row_base(a, p.pc.r, p.pgi);
            p.pc_on = true;
            return;
        }
    }
    p.pc_on = false;
}

// Producer (lane 0, p.pc_on): copy the next chunk into `slot` and advance;
// `a` is the constants of step p.pstep.
template <int NT>
__device__ __forceinline__ void pipe_produce(Pipe &p, const GroupArgs &a, int slot, int cta,
                                             int warp) {
    constexpr int CH = chunk_tiles(NT);
    const int n = min(CH, min(p.pc.uend - p.pc.u, p.pc.kw - p.pc.b));
    bulk_load(p.ring_w + slot * (CH * 512), p.prow + (long long)(p.pc.kb0 + p.pc.b) * 512, n * 512,
              p.bar_w + 8u * slot);
    p.inflight |= 1u << slot;
    p.pc.u += n;
    p.pc.b += n;
    if (p.pc.b == p.pc.kw) {
        p.pc.b = 0;
        ++p.pc.r;
        if (p.pgi + 1 < a.G && p.pc.r == a.rt_off[p.pgi + 1]) p.prow = a.packed[++p.pgi];
        else p.prow += (long long)a.KB * 512;
    }
    if (p.pc.u == p.pc.uend) {
        ++p.pc.sigma;
        if (cursor_enter(a, p.pcu0, p.pcu1, p.psig1, warp, p.pc)) {
            p.prow = row_base(a, p.pc.r, p.pgi);
        } else {
            ++p.pstep;
            pipe_seek(p, cta, warp);
        }
    }
}

// Lane 0: bring this warp's tiles of one linear step into L2 with bulk
// prefetches of up to CH tiles (they return no data), from cursor q on.
template <int NT>
__device__ __forceinline__ void prefetch_from(const GroupArgs &a, Cursor q, int qg, const char *qr,
                                              int cu0, int cu1, int sig1, int warp) {
    constexpr int CH = chunk_tiles(NT);
    for (bool on = true; on;) {
        const int n = min(CH, min(q.uend - q.u, q.kw - q.b));
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qr + (long long)(q.kb0 + q.b) * 512),
                     "r"(n * 512)
                     : "memory");
        q.u += n;
        q.b += n;
        if (q.b == q.kw) {
            q.b = 0;
            ++q.r;
            if (qg + 1 < a.G && q.r == a.rt_off[qg + 1]) qr = a.packed[++qg];
            else qr += (long long)a.KB * 512;
        }
        if (q.u == q.uend) {
            ++q.sigma;
            on = cursor_enter(a, cu0, cu1, sig1, warp, q);
            if (on) qr = row_base(a, q.r, qg);
        }
    }
}

// All of this warp's tiles of a (later) step of a chain.
template <int NT>
__device__ __forceinline__ void prefetch_l2(const GroupArgs &a, int cta, int warp) {
    if (a.kind != kStepLinear || cta >= a.P) return;
    int cu0, cu1, sig0, sig1;
    cta_units(a, cta, cu0, cu1, sig0, sig1);
    Cursor q;
    q.sigma = sig0;
    if (!cursor_enter(a, cu0, cu1, sig1, warp, q)) return;
    int qg = 0;
    const char *qr = row_base(a, q.r, qg);
    prefetch_from<NT>(a, q, qg, qr, cu0, cu1, sig1, warp);
}

// The rest of this warp's tiles of the pipe's current step: those after
// the chunks its first copies took.
template <int NT>
__device__ __forceinline__ void prefetch_rest(const Pipe &p, const GroupArgs &a, int warp) {
    if (p.pc_on && p.pstep == 0)
        prefetch_from<NT>(a, p.pc, p.pgi, p.prow, p.pcu0, p.pcu1, p.psig1, warp);
}

// Lane 0, after a wait gave up: let the copies still in flight land
// (bounded) before the CTA leaves.
__device__ __forceinline__ void pipe_drain(const Pipe &p, int *status) {
    for (int k = 0; k < kSlots; ++k)
        if (p.inflight >> k & 1) mbar_wait(p.bar_w + 8u * k, (p.phases >> k) & 1u, status);
}

// Lane 0: barriers of this warp's ring, then the first kSlots copies.
template <int NT>
__device__ __forceinline__ void pipe_start(Pipe &p, int cta, int warp) {
    for (int k = 0; k < kSlots; ++k) mbar_init(p.bar_w + 8u * k, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    pipe_seek(p, cta, warp);
    for (int k = 0; k < kSlots && p.pc_on; ++k) pipe_produce<NT>(p, p.steps[p.pstep], k, cta, warp);
}

// Bounded wait of one thread until *word reaches `target` (64-bit), or,
// with `nonzero`, until the 32-bit word is non-zero; then an acquire fence
// (the polls are relaxed loads, so waiting CTAs order nothing until the
// value is seen).  Gives up, returning false, when another CTA has set the
// status word or after `limit` SM cycles (and then sets the status word).
__device__ __forceinline__ bool wait_word(const void *word, unsigned long long target, bool nonzero,
                                          long long limit, int *status) {
    const long long t0 = clock64();
    for (unsigned it = 0;; ++it) {
        bool ok;
        if (nonzero) {
            unsigned v;
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(word) : "memory");
            ok = v != 0u;
        } else {
            unsigned long long v;
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(word) : "memory");
            ok = v >= target;
        }
        if (ok) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
        if ((it & 15u) == 15u) {
            int st;
            asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(st) : "l"(status) : "memory");
            if (st != 0) return false;
            if (clock64() - t0 > limit) {
                atomicExch(status, TL_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Wait (thread 0) for step `step`'s inputs: the gate before step 0, else
// all prevP CTAs of step - 1 in this pass.  The counters only grow: after
// `epoch` completed passes, step i is done in this pass when its counter
// reaches (epoch + 1) * P_i.
__device__ __forceinline__ bool wait_inputs(const ChainHeader *ch, int step, unsigned long long epoch,
                                            unsigned prevP, int *status) {
    if (step == 0) return ch->gate == nullptr || wait_word(ch->gate, 0ull, true, ch->wait_limit, status);
    return wait_word(ch->cnt + step - 1, (epoch + 1) * prevP, false, ch->wait_limit, status);
}

// Count this CTA into step `step` (thread 0, after a barrier that follows
// the CTA's last write of the step): one release reduction, no reply awaited.
__device__ __forceinline__ void signal_step(const ChainHeader *ch, int step) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ch->cnt + step) : "memory");
}

// Leaving a pass (thread 0 of every CTA): the last CTA out advances the
// pass count, which the next launch reads at its start.
__device__ __forceinline__ void leave_pass(const ChainHeader *ch, unsigned long long epoch) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    if (atomicAdd(ch->epoch + 1, 1ull) + 1ull == (unsigned long long)gridDim.x) {
        ch->epoch[1] = 0ull;
        ch->epoch[0] = epoch + 1ull;
    }
}

// Per-CTA shared state of a linear step.
template <int NT>
struct StepSmem {
    float bslot[kWarps][2][16 * NT];   // boundary pieces of the current slice
    int bslot_row[kWarps][2];
    // per (block, token, half block): -(sum of x) * 2^(T - 133), added to the
    // half's chain once per tile (see xh_index)
    float xh[kMaxSlice * NT * 2];
    int texp[NT];                      // T per token: X is staged times 2^(T - 2q)
    int emax[NT];
    int redo;                          // tokens outside the fixed window (bit mask)
    int go;                            // the step's inputs are ready
    unsigned long long epoch;          // chain passes completed before this one
    float qs[NT], qr[NT];              // fused quantisation: each token's step and 1/step
    int qz[NT];                        // and zero point
};

// ------------------------------------------------------------ one linear step
// Fused quantisation, threads n < NT: token n's step, its reciprocal and
// its zero point from the per-warp minima and maxima in red[w][0 / 1][n]
// (each range includes 0), formed as the quantiser kernel forms them.
// Columns past the batch get step 1 and zero point 0, so they stage zeros.
template <int NT, int W>
__device__ __forceinline__ void quant_params(const float (&red)[W][2][16 * NT], int sym, float *qs,
                                             float *qr, int *qz) {
    if (threadIdx.x >= NT) return;
    const int n = threadIdx.x;
    float l = 0.f, h = 0.f;
    for (int w = 0; w < W; ++w) {
        l = fminf(l, red[w][0][n]);
        h = fmaxf(h, red[w][1][n]);
    }
    float sv;
    int zv;
    if (sym) {
        const float m = fmaxf(-l, h);   // max |x|, the row's range including 0
        sv = m == 0.f ? 1.f : __fdiv_rn(m, 127.f);
        zv = 0;
    } else if (h == l) {
        sv = 1.f;
        zv = 0;
    } else {
        sv = __fdiv_rn(__fsub_rn(h, l), 255.f);
        zv = -128 - (int)rintf(__fdiv_rn(l, sv));
    }
    qs[n] = sv;
    qr[n] = __frcp_rn(sv);
    qz[n] = zv;
}

// kModeA: bf16 activations (else int8 from the quantiser).  kQ (with
// !kModeA): bf16 activations quantised per token by the step itself, as the
// quantiser kernel would, then mode B's arithmetic.  NT: token columns
// staged (a power of two >= N).  kChain: the step is one of a chain
// run by one persistent launch; it waits for the prevP CTAs of step - 1
// (the chain's counters) instead of for the previous kernel.  Returns, the
// same in every thread of the CTA, whether every wait succeeded.
template <bool kModeA, int NT, bool kChain, bool kQ = false>
__device__ __forceinline__ bool run_step(const GroupArgs &a, int cta, uint8_t *smem,
                                         StepSmem<NT> &sh, Pipe &pipe, const ChainHeader *ch,
                                         int step, unsigned prevP) {
    constexpr int CH = chunk_tiles(NT);         // tiles per bulk copy
    constexpr int SLOT = CH * 512;
    constexpr int XQ = NT * 4;                  // uint4 per 32-column quarter
    constexpr int XB = 4 * XQ;                  // uint4 per 128-column block
    constexpr int RV = 16 * NT;                 // floats per row-tile result
    constexpr bool kBf = kModeA || kQ;          // X is bf16
    constexpr int VPL = kBf ? 8 : 16;           // activations per staging group
    constexpr int LB = 128 / VPL;               // staging groups per block
    constexpr int HB = LB / 2;                  // staging groups per half block
    constexpr int XHB = 2 * NT;                 // correction floats per block
    constexpr int SB = stage_batch(NT, kBf);    // staging loads in flight per thread
    constexpr bool kAsyncX = NT >= 4;           // stage X with cp.async (when X allows 16-byte copies)
    // dynamic shared memory, at offsets fixed for every step of a launch
    uint8_t *ring = smem;                                                // [kWarps][kSlots][SLOT]
    uint4 *xs = reinterpret_cast<uint4 *>(smem + ring_bytes(NT));      // one slice of X
    float *acc = reinterpret_cast<float *>(smem + ring_bytes(NT) + a.kwr * XB * 16);  // [rows][RV]
    float *scl = acc + a.rowsr * RV;                                     // [rows][16] scales
    int *rsm = reinterpret_cast<int *>(scl + a.rowsr * 16);              // [rows][16] row sums
    auto &bslot = sh.bslot;
    auto &bslot_row = sh.bslot_row;
    float *xh = sh.xh;
    int *texp = sh.texp;
    int *emax = sh.emax;
    int &redo = sh.redo;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int N = a.N;
    // this CTA's units: range c_in of its slice (none past the last slice)
    int cu0, cu1, sig0, sig1;
    cta_units(a, cta, cu0, cu1, sig0, sig1);
    uint32_t *xw = reinterpret_cast<uint32_t *>(xs);
    const uint32_t xs_s = smem_u32(xs);

    // this CTA's scales (and row sums) of its first slice, one per thread
    Slice P;
    slice_of(a, cu0, cu1, sig0, P);
    float sc_pre = 0.f;
    int rs_pre = 0;
    {
        const int rho = threadIdx.x >> 4, i = threadIdx.x & 15;
        if (rho <= P.r_last - P.r_first) {
            int gi;
            row_base(a, P.r_first + rho, gi);
            const int m = (P.r_first + rho - a.rt_off[gi]) * 16 + i;
            if (m < a.M[gi]) {
                sc_pre = __ldg(a.scale[gi] + m);
                if (!kModeA) rs_pre = __ldg(a.rowsum[gi] + m);
            }
        }
    }
    if (threadIdx.x < kWarps * 2) (&bslot_row[0][0])[threadIdx.x] = -1;
    if (threadIdx.x == 0) redo = 0;
    if (threadIdx.x < NT) emax[threadIdx.x] = 0;
    for (int i = threadIdx.x; i < a.rows * RV; i += kThreads) acc[i] = 0.f;
    if (N < NT) {  // the columns past the batch stay zero in every slice
        for (int i = threadIdx.x; i < a.kwr * 64 * NT; i += kThreads)
            if (((i >> 4) % NT) >= N) xw[i] = 0u;
        for (int i = threadIdx.x; i < kMaxSlice * NT * 2; i += kThreads) xh[i] = 0.f;
    }
    // Warm L2 (and the address translation) for this CTA's activations; a
    // prefetch returns no data, so it may run before the previous kernel has
    // written them.  One 128-byte line per thread per step, addresses inside
    // each row's columns [k_lo, k_hi).
    if (sig1 > sig0) {
        constexpr int EB = kBf ? 2 : 1;
        const long long k_lo = (long long)sig0 * a.KW * 128;
        const long long k_hi = min((long long)a.K, (long long)sig1 * a.KW * 128);
        const int lines = (int)((k_hi - k_lo) * EB + 127) / 128;
        for (int i = threadIdx.x; i < N * lines; i += kThreads) {
            const int n = i / lines, l = i - n * lines;
            const char *p = reinterpret_cast<const char *>(a.X) + ((long long)n * a.K + k_lo) * EB + l * 128;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
    __syncthreads();

    // Now the activations, written by the previous kernel or step.
    if (!kChain) {
        griddep_wait();
    } else {
        if (threadIdx.x == 0) sh.go = wait_inputs(ch, step, sh.epoch, prevP, a.status);
        __syncthreads();
        if (!sh.go) return false;
    }
    // the token scales the epilogue of an integer mode uses
    const float *ts = kQ ? sh.qs : a.s;
    const int32_t *tz = kQ ? sh.qz : a.z;
    uint4 xv[SB];
    bool xv_loaded = false;
    // fused quantisation with one slice copied whole by cp.async: the range
    // comes from the copied slice (below) instead of a pass of its own
    const bool q_late = kQ && kAsyncX && a.xvec && a.NS == 1;
    if (kQ && !q_late) {
        // Fused quantisation: every CTA reduces each token's whole row to its
        // minimum and maximum (widened to include 0; exact in any order, so
        // every CTA derives the same step and zero point) and forms them as
        // the quantiser kernel does; padding past K is staged as the
        // quantised zero, whose products with the padded weights cancel in
        // the chains' integer sums.
        // R rows' worth of loads per token in flight per thread (eight in all)
        constexpr int R = NT >= 8 ? 1 : 8 / NT;
        float lo[NT], hi[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) lo[n] = hi[n] = 0.f;
        const uint16_t *x0 = reinterpret_cast<const uint16_t *>(a.X);
        if (a.NS == 1 && !(kAsyncX && a.xvec) && N * P.kw * LB <= kThreads * SB) {
            // One slice, staged from registers in one batch: that batch is
            // every token's whole row, so it gives the minimum and maximum.
            stage_load<kBf, SB, kChain>(a, P, 0, xv);
            xv_loaded = true;
            const int total = N * P.kw * LB;
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                const int idx = i * kThreads + (int)threadIdx.x;
                if (idx >= total) break;
                const int n = fdiv(idx / LB, a.dKWL);
                const uint32_t w4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
                float l = 0.f, h = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float e0 = __uint_as_float(w4[j] << 16), e1 = __uint_as_float(w4[j] & 0xFFFF0000u);
                    l = fminf(l, fminf(e0, e1));
                    h = fmaxf(h, fmaxf(e0, e1));
                }
#pragma unroll
                for (int nn = 0; nn < NT; ++nn)
                    if (nn == n) {
                        lo[nn] = fminf(lo[nn], l);
                        hi[nn] = fmaxf(hi[nn], h);
                    }
            }
        } else if (a.xvec) {
            const int nv = a.K / 8;
            for (int i0 = threadIdx.x; i0 < nv; i0 += kThreads * R) {
                uint4 u[R][NT];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const int i = i0 + r * kThreads;
                        u[r][n] = (n < N && i < nv)
                                      ? ldx<kChain>(reinterpret_cast<const uint4 *>(x0 + (long long)n * a.K) + i)
                                      : make_uint4(0u, 0u, 0u, 0u);   // zero: inside every range
                    }
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const uint32_t w4[4] = {u[r][n].x, u[r][n].y, u[r][n].z, u[r][n].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float e0 = __uint_as_float(w4[j] << 16),
                                        e1 = __uint_as_float(w4[j] & 0xFFFF0000u);
                            lo[n] = fminf(lo[n], fminf(e0, e1));
                            hi[n] = fmaxf(hi[n], fmaxf(e0, e1));
                        }
                    }
            }
        } else {
            for (int k0 = threadIdx.x; k0 < a.K; k0 += kThreads * R) {
                uint32_t u[R][NT];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const int k = k0 + r * kThreads;
                        u[r][n] = (n < N && k < a.K) ? (uint32_t)ldx16<kChain>(x0 + (long long)n * a.K + k) : 0u;
                    }
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const float e = __uint_as_float(u[r][n] << 16);
                        lo[n] = fminf(lo[n], e);
                        hi[n] = fmaxf(hi[n], e);
                    }
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                lo[n] = fminf(lo[n], __shfl_xor_sync(0xffffffffu, lo[n], off));
                hi[n] = fmaxf(hi[n], __shfl_xor_sync(0xffffffffu, hi[n], off));
            }
            if (lane == 0) {
                bslot[warp][0][n] = lo[n];       // the boundary slots are free until the main loop
                bslot[warp][1][n] = hi[n];
            }
        }
        __syncthreads();
        quant_params<NT>(bslot, a.sym, sh.qs, sh.qr, sh.qz);
        __syncthreads();
    }
    if (!(kAsyncX && a.xvec) && !xv_loaded) stage_load<kBf, SB, kChain>(a, P, 0, xv);

    Cursor cc;
    cc.sigma = sig0;
    bool cc_on = cursor_enter(a, cu0, cu1, sig1, warp, cc);
    int &slot = pipe.slot;
    uint32_t &phases = pipe.phases;             // parity bit per slot
    const uint32_t bar_w = pipe.bar_w;
    bool ok = true;
    float c[4][4];

    for (int sigma = sig0; sigma < sig1; ++sigma) {
        if (sigma != sig0) slice_of(a, cu0, cu1, sigma, P);
        const int nrows = P.r_last - P.r_first + 1;
        // ---- stage X for the slice in B-fragment order, times 2^kT, and sum
        // it per block.  Word ((j*4 + qd)*NT + n)*16 + 4*tt + w holds
        // x[n][k], x[n][k+1] for m = 2qd + w/2, k = (kb0 + j)*128 + 16*m +
        // 2*tt + 8*(w%2); columns n >= N stay zero.  A thread takes VPL
        // consecutive activations at a time (one 16-byte load when X allows
        // it); the LB threads of a block sum it in a fixed order, the same
        // for either kind of load.
        {
            const int total = N * P.kw * LB;
            const FastDiv dv = sigma == a.NS - 1 ? a.dKWL : a.dKW;
            if (kAsyncX && a.xvec) {
                // Four or more tokens: every 16 bytes of the slice's rows are
                // copied at once (cp.async, zero past K) into their block's own
                // region, row n at byte n * RB; then each warp rewrites its
                // blocks in place, group by group as below.
                constexpr int EB = kBf ? 2 : 1;
                constexpr int RB = 128 * EB;               // bytes of one token's block row
                constexpr int CPR = RB / 16;                // 16-byte copies per block row
                const int nch = N * P.kw * CPR;
                for (int i = threadIdx.x; i < nch; i += kThreads) {
                    const int c = i % CPR, q = i / CPR;     // q = n * kw + jb
                    const int n = fdiv(q, dv), jb = q - n * P.kw;
                    const int k0 = (P.kb0 + jb) * 128 + c * (16 / EB);
                    const uint32_t full = k0 < a.K ? 16u : 0u;
                    const char *src = reinterpret_cast<const char *>(a.X) +
                                      ((long long)n * a.K + (full ? k0 : 0)) * EB;
                    const uint32_t dst = xs_s + (uint32_t)(jb * (NT * 256) + n * RB + c * 16);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                                 "r"(full)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
                __syncthreads();
                if (q_late) {
                    // Every token's whole row is in the slice: thread t reads
                    // token (t / 16) % NT only (kThreads is a multiple of 16 NT),
                    // each half warp reduces its token, and warp w leaves its two
                    // tokens' ranges (zero elsewhere) in the boundary slots.
                    static_assert(kThreads % (16 * NT) == 0, "one token per thread");
                    const int n = (threadIdx.x >> 4) % NT;
                    float l = 0.f, h = 0.f;
                    if (n < N) {
                        for (int u = threadIdx.x; u < P.kw * NT * 16; u += kThreads) {
                            const uint4 v = xs[u];
                            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float e0 = __uint_as_float(w4[j] << 16),
                                            e1 = __uint_as_float(w4[j] & 0xFFFF0000u);
                                l = fminf(l, fminf(e0, e1));
                                h = fmaxf(h, fmaxf(e0, e1));
                            }
                        }
                    }
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) {
                        l = fminf(l, __shfl_xor_sync(0xffffffffu, l, off));
                        h = fmaxf(h, __shfl_xor_sync(0xffffffffu, h, off));
                    }
                    if (lane < NT) bslot[warp][0][lane] = bslot[warp][1][lane] = 0.f;
                    __syncwarp();
                    if ((lane & 15) == 0) {
                        bslot[warp][0][n] = l;
                        bslot[warp][1][n] = h;
                    }
                    __syncthreads();
                    quant_params<NT>(bslot, a.sym, sh.qs, sh.qr, sh.qz);
                    __syncthreads();
                }
                constexpr int J = NT * LB / 32 > 0 ? NT * LB / 32 : 1;   // groups per lane in one block
                for (int jb = warp; jb < P.kw; jb += kWarps) {
                    uint32_t *blk = xw + jb * NT * 64;
                    uint4 v[J];
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const int g = lane + 32 * j, n = g / LB, o = g % LB;
                        v[j] = n < N ? *reinterpret_cast<const uint4 *>(blk + n * (RB / 4) + o * 4)
                                     : make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const int g = lane + 32 * j, n = g / LB, o = g % LB;
                        float sum;
                        uint32_t bad;
                        stage_group<kModeA, NT, kQ>(blk, n, o, v[j], sum, bad, sh.qs, sh.qr, sh.qz, a.sym);
#pragma unroll
                        for (int off = HB / 2; off > 0; off >>= 1)
                            sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, off));
                        if (n < N && (o % HB) == 0) xh[xh_index<NT>(jb, n, o / HB)] = chain_units(sum, kT);
                        if (kModeA && n < N && bad) atomicOr(&redo, 1 << n);
                    }
                }
            } else
            for (int base = 0; base < total; base += kThreads * SB) {
                if (sigma != sig0 || base != 0) stage_load<kBf, SB, kChain>(a, P, base, xv);
#pragma unroll
                for (int i = 0; i < SB; ++i) {
                    if (base + i * kThreads >= total) break;   // uniform over the block
                    const int idx = base + i * kThreads + (int)threadIdx.x;
                    const bool valid = idx < total;
                    const int q = idx / LB, o = idx % LB;
                    const int n = valid ? fdiv(q, dv) : 0, jb = q - n * P.kw;
                    float sum = 0.f;
                    uint32_t bad = 0u;
                    if (valid)
                        stage_group<kModeA, NT, kQ>(xw + jb * NT * 64, n, o, xv[i], sum, bad, sh.qs, sh.qr,
                                                    sh.qz, a.sym);
#pragma unroll
                    for (int off = HB / 2; off > 0; off >>= 1)
                        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, off));
                    if (valid && (o % HB) == 0) xh[xh_index<NT>(jb, n, o / HB)] = chain_units(sum, kT);
                    if (kModeA && valid && bad) atomicOr(&redo, 1 << n);
                }
            }
            // this slice's scales and row sums (one per thread)
            if (sigma == sig0) {
                if ((int)(threadIdx.x >> 4) < a.rows) {
                    scl[threadIdx.x] = sc_pre;
                    if (!kModeA) rsm[threadIdx.x] = rs_pre;
                }
            } else {
                const int rho = threadIdx.x >> 4, i = threadIdx.x & 15;
                float sc = 0.f;
                int rs = 0;
                if (rho < nrows) {
                    int gi;
                    row_base(a, P.r_first + rho, gi);
                    const int m = (P.r_first + rho - a.rt_off[gi]) * 16 + i;
                    if (m < a.M[gi]) {
                        sc = __ldg(a.scale[gi] + m);
                        if (!kModeA) rs = __ldg(a.rowsum[gi] + m);
                    }
                }
                if (rho < a.rows) {
                    scl[threadIdx.x] = sc;
                    if (!kModeA) rsm[threadIdx.x] = rs;
                }
            }
        }
        if (threadIdx.x < NT) texp[threadIdx.x] = kT;
        __syncthreads();

        if (kModeA && redo != 0) {
            // Rare: some token has activations outside the fixed window.  Its
            // scale follows its largest exponent field E in the slice: 2^(254 - E)
            // keeps every staged value finite; values more than 2^120 below the
            // largest may lose their contribution.
            const int mask = redo;
            const int klo = P.kb0 * 128, khi = min((P.kb0 + P.kw) * 128, a.K);
            for (int n = 0; n < N; ++n) {
                if (!(mask >> n & 1)) continue;
                const uint16_t *x = reinterpret_cast<const uint16_t *>(a.X) + (long long)n * a.K;
                uint32_t e = 0;
                for (int k = klo + threadIdx.x; k < khi; k += kThreads)
                    e = max(e, ((uint32_t)__ldcg(x + k) >> 7) & 0xFFu);
                e = __reduce_max_sync(0xffffffffu, e);
                if (lane == 0) atomicMax(&emax[n], (int)e);
            }
            __syncthreads();
            if (threadIdx.x < NT && (mask >> threadIdx.x & 1)) texp[threadIdx.x] = 254 - emax[threadIdx.x];
            for (int idx = threadIdx.x; idx < P.kw * 64 * NT; idx += kThreads) {
                const int n = (idx >> 4) % NT;
                if (!(mask >> n & 1)) continue;
                const int w = idx & 3, tt = (idx >> 2) & 3, rest = (idx >> 4) / NT;
                const int qd = rest & 3, j = rest >> 2;
                const int m = 2 * qd + (w >> 1);
                const int k = (P.kb0 + j) * 128 + 16 * m + 2 * tt + 8 * (w & 1);
                const uint16_t *x = reinterpret_cast<const uint16_t *>(a.X) + (long long)n * a.K;
                const uint32_t lo = k < a.K ? __ldcg(x + k) : 0u, hi = k + 1 < a.K ? __ldcg(x + k + 1) : 0u;
                const int d = 254 - emax[n] - 2 * (m & 3);
                xw[idx] = scale_any(lo, d) | (scale_any(hi, d) << 16);
            }
            // and the token's corrections at its new scale: one warp per
            // (token, block, half), 64 activations summed in a fixed order
            for (int p = warp; p < N * P.kw * 2; p += kWarps) {
                const int h = p & 1, j = (p >> 1) % P.kw, n = (p >> 1) / P.kw;
                if (!(mask >> n & 1)) continue;
                const uint16_t *x = reinterpret_cast<const uint16_t *>(a.X) + (long long)n * a.K;
                const int k = (P.kb0 + j) * 128 + 64 * h + 2 * lane;
                float sm = __fadd_rn(k < a.K ? bf16f(__ldcg(x + k)) : 0.f,
                                     k + 1 < a.K ? bf16f(__ldcg(x + k + 1)) : 0.f);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, off));
                if (lane == 0) xh[xh_index<NT>(j, n, h)] = chain_units(sm, 254 - emax[n]);
            }
            __syncthreads();
            if (threadIdx.x == 0) redo = 0;
            if (threadIdx.x < NT) emax[threadIdx.x] = 0;
        }

        // this lane's tokens 2t, 2t+1: the chains hold sum (1 - w) x 2^(T - 133)
        // minus the corrections sum x 2^(T - 133), i.e. -sum w x 2^(T - 133);
        // undo 2^(T - 133) with two exact factors
        int tx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) tx[e] = texp[(2 * t + e) % NT];
        const float *xhl = xh + (NT == 1 ? 0 : xh_index<NT>(0, 2 * (t % (NT > 1 ? NT / 2 : 1)), 0));

        // ---- this warp's units of the slice
        int run_lo = cc.b, nslot = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
        while (ok && cc_on && cc.sigma == sigma) {
            const int n = min(CH, min(cc.uend - cc.u, cc.kw - cc.b));
            const bool got = __all_sync(0xffffffffu,
                                        mbar_wait(bar_w + 8u * slot, (phases >> slot) & 1u, a.status));
            if (!got) { ok = false; break; }
            phases ^= 1u << slot;
            const uint4 *tiles = reinterpret_cast<const uint4 *>(ring + warp * (kSlots * SLOT) + slot * SLOT) + lane;
            const uint4 *xb = xs + cc.b * XB + (g % NT) * 4 + t;
            const float *xc = xhl + cc.b * XHB;
            if (n == CH) {
                // full chunk: load tile i+1 while tile i is multiplied
                uint4 w = tiles[0];
                uint4 bq[4];
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) bq[qd] = xb[qd * XQ];
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    uint4 wn = w, bn[4] = {bq[0], bq[1], bq[2], bq[3]};
                    if (i + 1 < CH) {
                        wn = tiles[(i + 1) * 32];
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd) bn[qd] = xb[(i + 1) * XB + qd * XQ];
                    }
                    tile_corrected<NT>(c, i & 1, w, bq, xc + i * XHB);
                    w = wn;
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) bq[qd] = bn[qd];
                }
            } else {
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    if (i >= n) break;
                    const uint4 w = tiles[i * 32];
                    uint4 bq[4];
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) bq[qd] = xb[i * XB + qd * XQ];
                    tile_corrected<NT>(c, i & 1, w, bq, xc + i * XHB);
                }
            }
            // end of a run of one row tile: this chunk ends the row or the warp's range
            if (cc.b + n == cc.kw || cc.u + n == cc.uend) {
                // lane (g, t) holds rows g, g+8 of tokens 2t, 2t+1: v[2h + e]
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float sm = __fadd_rn(__fadd_rn(c[0][q], c[1][q]), __fadd_rn(c[2][q], c[3][q]));
                    const int d = 133 - tx[q & 1], d1 = d / 2;
                    v[q] = -__fmul_rn(__fmul_rn(sm, __int_as_float((d1 + 127) << 23)),
                                      __int_as_float((d - d1 + 127) << 23));
                }
                int lo, hi;
                row_span(P, cc.r, lo, hi);
                const int rho = cc.r - P.r_first;
                if (run_lo == lo && cc.b + n == hi) {
                    // the whole row tile of this slice: no other warp touches it
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            if (2 * t + e < NT) acc[rho * RV + (2 * t + e) * 16 + g + 8 * h] += v[2 * h + e];
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            if (2 * t + e < NT) bslot[warp][nslot][(2 * t + e) * 16 + g + 8 * h] = v[2 * h + e];
                    if (lane == 0) bslot_row[warp][nslot] = rho;
                    ++nslot;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
                run_lo = cc.b + n < cc.kw ? cc.b + n : -1;   // next run starts a row
            }
            // refill this slot with the chunk kSlots ahead
            __syncwarp();
            if (lane == 0) {
                pipe.inflight &= ~(1u << slot);
                if (pipe.pc_on) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    pipe_produce<NT>(pipe, kChain ? pipe.steps[pipe.pstep] : a, slot, cta, warp);
                }
            }
            cc.u += n;
            cc.b += n;
            if (cc.b == cc.kw) { cc.b = 0; ++cc.r; }
            if (cc.u == cc.uend) {
                ++cc.sigma;
                cc_on = cursor_enter(a, cu0, cu1, sig1, warp, cc);
            }
            if (run_lo < 0) run_lo = cc.b;
            slot ^= 1;
        }
        __syncthreads();
        // ---- boundary pieces of the slice, added in warp order (one thread per element)
        for (int i = threadIdx.x; i < nrows * RV; i += kThreads) {
            const int rho = i / RV, e = i % RV;
            float v = acc[i];
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (bslot_row[w][k] == rho) v += bslot[w][k][e];
            acc[i] = v;
        }
        __syncthreads();
        if (threadIdx.x < kWarps * 2) (&bslot_row[0][0])[threadIdx.x] = -1;

        // ---- the slice's rows: sum_k w*x over the CTA's blocks of row tile r
        // is (sum of x over those blocks) - 2^P * S.  A row tile wholly inside
        // this CTA and slice goes straight to Y; otherwise the piece goes to
        // the workspace and whoever completes the row tile adds all pieces.
        if (ok) {
            for (int rho = warp; rho < nrows; rho += kWarps) {
                const int r = P.r_first + rho;
                int lo, hi;
                row_span(P, r, lo, hi);
                float *v = acc + rho * RV;
                if (a.NS == 1 && lo == 0 && hi == P.kw) {
                    store_row_tile(a, r, v, scl + rho * 16, rsm + rho * 16, ts, tz, lane);
                } else if (a.NS == 1) {
                    exchange_row_tile(a, r, v, scl + rho * 16, rsm + rho * 16, ts, tz, lane);
                } else {
                    const int half = lo == 0 ? 0 : 1;   // 0: holds the slice's first block
                    float *dst = a.part + (((long long)r * a.NS + sigma) * 2 + half) * N * 16;
                    for (int e = lane; e < N * 16; e += 32) __stcg(dst + e, v[e]);
                    __syncwarp();
                    unsigned long long now = 0ull;
                    if (lane == 0) {
                        asm volatile("fence.acq_rel.gpu;" ::: "memory");
                        now = atomicAdd(a.cnt + r, (unsigned long long)(hi - lo)) + (unsigned long long)(hi - lo);
                    }
                    now = __shfl_sync(0xffffffffu, now, 0);
                    if (now == (unsigned long long)a.KB) {
                        asm volatile("fence.acq_rel.gpu;" ::: "memory");
                        // all pieces, slice by slice, the half with the slice's first
                        // block first; kPS slices' loads in flight at a time
                        constexpr int kE = (16 * NT + 31) / 32;   // elements per lane
                        constexpr int kPS = NT >= 8 ? 2 : 4;       // slices per batch of loads
                        float y[kE];
#pragma unroll
                        for (int j = 0; j < kE; ++j) y[j] = 0.f;
                        for (int s0 = 0; s0 < a.NS; s0 += kPS) {
                            float pv[kPS][2][kE];
#pragma unroll
                            for (int ds = 0; ds < kPS; ++ds) {
                                const int s2 = s0 + ds;
                                const bool have = s2 < a.NS;
                                const bool split = have && piece_split(a, r, s2);
                                const float *pc2 = a.part + ((long long)r * a.NS + (have ? s2 : 0)) * 2 * N * 16;
#pragma unroll
                                for (int j = 0; j < kE; ++j) {
                                    const int e = lane + 32 * j;
                                    pv[ds][0][j] = have && e < N * 16 ? __ldcg(pc2 + e) : 0.f;
                                    pv[ds][1][j] = split && e < N * 16 ? __ldcg(pc2 + N * 16 + e) : 0.f;
                                }
                            }
#pragma unroll
                            for (int ds = 0; ds < kPS; ++ds) {
                                if (s0 + ds >= a.NS) break;
                                const bool split = piece_split(a, r, s0 + ds);
#pragma unroll
                                for (int j = 0; j < kE; ++j) {
                                    y[j] = __fadd_rn(y[j], pv[ds][0][j]);
                                    if (split) y[j] = __fadd_rn(y[j], pv[ds][1][j]);
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < kE; ++j)
                            if (lane + 32 * j < N * 16) v[lane + 32 * j] = y[j];
                        __syncwarp();
                        store_row_tile(a, r, v, scl + rho * 16, rsm + rho * 16, ts, tz, lane);
                        if (lane == 0) a.cnt[r] = 0ull;
                    }
                }
                __syncwarp();
                for (int e = lane; e < RV; e += 32) v[e] = 0.f;   // ready for the next slice
            }
        }
        // (the next slice's staging barrier orders these reads of xh, acc
        // and scl before they are rewritten)
    }
    return __syncthreads_and(ok) != 0;
}


// ------------------------------------------------------------ kernels
// One (grouped) linear per launch; kQ quantises bf16 X per token itself.
template <bool kModeA, int NT, bool kQ = false>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
tl_mma_kernel(const __grid_constant__ GroupArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(16) StepSmem<NT> sh;
    __shared__ __align__(8) unsigned long long bars[kWarps][kSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The dependent launch may be scheduled at once; it only streams weights
    // until this grid has finished.
    griddep_launch();
    Pipe pipe;
    pipe.ring_w = smem_u32(smem) + warp * (kSlots * chunk_tiles(NT) * 512);
    pipe.bar_w = smem_u32(&bars[warp][0]);
    pipe.slot = 0;
    pipe.phases = 0;
    pipe.inflight = 0;
    pipe.steps = &a;
    pipe.nsteps = 1;
    pipe.pstep = 0;
    // Weights do not depend on the previous kernel: each warp's lane 0 starts
    // its first copies, and brings the rest of its tiles into L2, before the
    // launch waits for it.
    if (lane == 0) {
        pipe_start<NT>(pipe, blockIdx.x, warp);
        prefetch_rest<NT>(pipe, a, warp);
    }
    const bool ok = run_step<kModeA, NT, false, kQ>(a, blockIdx.x, smem, sh, pipe, nullptr, 0, 0u);
    if (!ok && lane == 0) pipe_drain(pipe, a.status);
}

using KernelFn = void (*)(GroupArgs);

KernelFn kernel_for(int mode, int nt) {
    const bool A = mode == TL_MODE_BF16;
    if (mode == TL_MODE_I8_FUSED) switch (nt) {
            case 1: return tl_mma_kernel<false, 1, true>;
            case 2: return tl_mma_kernel<false, 2, true>;
            case 4: return tl_mma_kernel<false, 4, true>;
            default: return tl_mma_kernel<false, 8, true>;
        }
    switch (nt) {
        case 1: return A ? tl_mma_kernel<true, 1> : tl_mma_kernel<false, 1>;
        case 2: return A ? tl_mma_kernel<true, 2> : tl_mma_kernel<false, 2>;
        case 4: return A ? tl_mma_kernel<true, 4> : tl_mma_kernel<false, 4>;
        default: return A ? tl_mma_kernel<true, 8> : tl_mma_kernel<false, 8>;
    }
}

inline int padded_tokens(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

// ------------------------------------------------------------------ quant
// Per-token activation quantisation as a grid of (K chunk, token) CTAs.
// Every CTA of a token reduces the token's whole row to its minimum and
// maximum (exact and independent of order, so all of them derive the same s
// and z), then quantises its own chunk.  q = rint(x / s) needs the correctly
// rounded quotient only where it decides the rounding: x * (1/s) is within
// three units in the last place of fl(x / s), so it gives the same integer
// unless it lies that close to a half-integer (or is not finite), and only
// then is the IEEE division taken.
constexpr int kQThreads = 256;
constexpr int kQChunk = 4096;          // activations quantised per CTA
constexpr int kQHeld = 8;              // 16-byte groups a thread keeps in registers
// A launch of its own whose whole row fits in registers takes one CTA per
// token (the CTA quantises all of the row); otherwise one CTA per chunk.
__host__ __device__ __forceinline__ bool quant_held(int vec, int K) {
    return vec && K / 8 <= kQHeld * kQThreads;
}

// Token n, chunk c (kQT threads).  kLaunch: a launch of its own, which
// waits for the previous kernel on the stream and lets the next one start.
template <bool kLaunch, int kQT = kQThreads, bool kBfOut = false>
__device__ __forceinline__ void quant_chunk(const uint16_t *__restrict__ X, int K, int vec,
                                            void *__restrict__ Q, float *__restrict__ s_out,
                                            int32_t *__restrict__ z_out, int symmetric, int n,
                                            int c) {
    const int k0 = c * kQChunk;
    const uint16_t *x = X + (long long)n * K;
    int8_t *q = static_cast<int8_t *>(Q) + (long long)n * K;
    __nv_bfloat16 *qb = static_cast<__nv_bfloat16 *>(Q) + (long long)n * K;   // (kBfOut)
    // the previous kernel on the stream may still be writing X
    if (kLaunch) griddep_wait();
    float lo = 0.f, hi = 0.f;
    // A launch of its own whose row fits in registers (thread i holds the
    // 16-byte groups i, i + kQT, ...) is the token's only CTA: it quantises
    // the whole row from them instead of reading it again.
    const bool held = kLaunch && kQT == kQThreads && quant_held(vec, K);
    uint4 hv[kLaunch ? kQHeld : 1];
    if (held) {
        const uint4 *xv = reinterpret_cast<const uint4 *>(x);
#pragma unroll
        for (int j = 0; j < (kLaunch ? kQHeld : 1); ++j) {
            const int i = threadIdx.x + j * kQT;
            hv[j] = i < K / 8 ? __ldcg(xv + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < (kLaunch ? kQHeld : 1); ++j) {
            // groups past K hold zeros, which the range includes anyway
            const uint32_t w[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = __uint_as_float(w[e] << 16), b = __uint_as_float(w[e] & 0xFFFF0000u);
                if (symmetric) {
                    hi = fmaxf(hi, fmaxf(fabsf(a), fabsf(b)));
                } else {
                    lo = fminf(lo, fminf(a, b));
                    hi = fmaxf(hi, fmaxf(a, b));
                }
            }
        }
    } else if (vec) {
        const uint4 *xv = reinterpret_cast<const uint4 *>(x);
        for (int i = threadIdx.x; i < K / 8; i += kQT) {
            const uint4 u = __ldcg(xv + i);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
                if (symmetric) {
                    hi = fmaxf(hi, fmaxf(fabsf(a), fabsf(b)));
                } else {
                    lo = fminf(lo, fminf(a, b));
                    hi = fmaxf(hi, fmaxf(a, b));
                }
            }
        }
    } else {
        for (int k = threadIdx.x; k < K; k += kQT) {
            const float v = __uint_as_float((uint32_t)__ldcg(x + k) << 16);
            if (symmetric) {
                hi = fmaxf(hi, fabsf(v));
            } else {
                lo = fminf(lo, v);
                hi = fmaxf(hi, v);
            }
        }
    }
    __shared__ float slo[kQT / 32], shi[kQT / 32];
    __shared__ float s_sh;
    __shared__ int z_sh;
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    const int wid = threadIdx.x >> 5, ln = threadIdx.x & 31;
    if (ln == 0) { slo[wid] = lo; shi[wid] = hi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kQT / 32; ++w) {
            lo = fminf(lo, slo[w]);
            hi = fmaxf(hi, shi[w]);
        }
        float s;
        int z;
        if (symmetric) {
            s = hi == 0.f ? 1.f : __fdiv_rn(hi, 127.f);
            z = 0;
        } else if (hi == lo) {
            s = 1.f;
            z = 0;
        } else {
            s = __fdiv_rn(__fsub_rn(hi, lo), 255.f);
            z = -128 - (int)rintf(__fdiv_rn(lo, s));
        }
        s_sh = s;
        z_sh = z;
        if (c == 0) {
            s_out[n] = s;
            z_out[n] = z;
        }
    }
    __syncthreads();
    // the next kernel may start its prologue; it waits for this grid before
    // reading Q, s and z
    if (kLaunch) griddep_launch();
    const float s = s_sh;
    const float r = __frcp_rn(s);
    const float zf = (float)z_sh;
    const float qlo = symmetric ? -127.f : -128.f;
    const int k1 = min(K, k0 + kQChunk);
    auto qv = [&](float v) {
        return fminf(fmaxf(__fadd_rn(tl_internal::quant_round(v, s, r), zf), qlo), 127.f);
    };
    auto one = [&](float v) { return (uint32_t)(uint8_t)(int8_t)(int)qv(v); };
    if (held) {
#pragma unroll
        for (int j = 0; j < (kLaunch ? kQHeld : 1); ++j) {
            const int i = threadIdx.x + j * kQT;
            if (i >= K / 8) continue;
            const uint32_t w[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
            if (kBfOut) {
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(qv(__uint_as_float(w[e] << 16)),
                                                                    qv(__uint_as_float(w[e] & 0xFFFF0000u)));
                    o[e] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                reinterpret_cast<uint4 *>(qb)[i] = make_uint4(o[0], o[1], o[2], o[3]);
            } else {
                uint32_t o[2] = {0u, 0u};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t lo8 = one(__uint_as_float(w[e] << 16));
                    const uint32_t hi8 = one(__uint_as_float(w[e] & 0xFFFF0000u));
                    o[e >> 1] |= (lo8 | (hi8 << 8)) << (16 * (e & 1));
                }
                reinterpret_cast<uint2 *>(q)[i] = make_uint2(o[0], o[1]);
            }
        }
        return;
    }
    if (kBfOut) {
        // the integers as bf16 (exact): 8 per 16-byte store
        if (vec) {
            const uint4 *xv = reinterpret_cast<const uint4 *>(x);
            for (int i = k0 / 8 + threadIdx.x; i < k1 / 8; i += kQT) {
                const uint4 u = __ldcg(xv + i);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(qv(__uint_as_float(w[j] << 16)),
                                                                    qv(__uint_as_float(w[j] & 0xFFFF0000u)));
                    o[j] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                reinterpret_cast<uint4 *>(qb)[i] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        } else {
            for (int k = k0 + threadIdx.x; k < k1; k += kQT)
                qb[k] = __float2bfloat16_rn(qv(__uint_as_float((uint32_t)__ldcg(x + k) << 16)));
        }
        return;
    }
    if (vec) {
        // 8 activations per step: one 16-byte load, one 8-byte store
        const uint4 *xv = reinterpret_cast<const uint4 *>(x);
        for (int i = k0 / 8 + threadIdx.x; i < k1 / 8; i += kQT) {
            const uint4 u = __ldcg(xv + i);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t o[2] = {0u, 0u};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t lo8 = one(__uint_as_float(w[j] << 16));
                const uint32_t hi8 = one(__uint_as_float(w[j] & 0xFFFF0000u));
                o[j >> 1] |= (lo8 | (hi8 << 8)) << (16 * (j & 1));
            }
            reinterpret_cast<uint2 *>(q)[i] = make_uint2(o[0], o[1]);
        }
    } else {
        for (int k = k0 + threadIdx.x; k < k1; k += kQT)
            q[k] = (int8_t)one(__uint_as_float((uint32_t)__ldcg(x + k) << 16));
    }
}

template <bool kBfOut>
__global__ void __launch_bounds__(kQThreads)
tl_quant_kernel(const uint16_t *__restrict__ X, int K, int vec, void *__restrict__ Q,
                float *__restrict__ s_out, int32_t *__restrict__ z_out, int symmetric) {
    quant_chunk<true, kQThreads, kBfOut>(X, K, vec, Q, s_out, z_out, symmetric, blockIdx.y, blockIdx.x);
}

// ------------------------------------------------------------------ chains
// A chain of linears (and, in mode B, quantiser steps) in one persistent
// launch: every CTA works through the steps in order, waiting before each
// for the previous step's CTAs to have finished (a release/acquire counter
// per step, bounded waits), while its warps' weight pipelines run ahead into
// later steps and prefetch their weights into L2.  The CTA that completes a
// step's counter clears the previous step's, and the last step's, so the
// counters are zero again when the launch ends.
template <bool kModeA, int NT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
tl_chain_kernel(const ChainHeader *__restrict__ ch, const GroupArgs *__restrict__ steps) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(16) StepSmem<NT> sh;
    __shared__ __align__(8) unsigned long long bars[kWarps][kSlots];
    __shared__ __align__(16) GroupArgs sa;      // the current step's constants
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, cta = blockIdx.x;
    const int nsteps = ch->nsteps, ahead = ch->lookahead;
    Pipe pipe;
    pipe.ring_w = smem_u32(smem) + warp * (kSlots * chunk_tiles(NT) * 512);
    pipe.bar_w = smem_u32(&bars[warp][0]);
    pipe.slot = 0;
    pipe.phases = 0;
    pipe.inflight = 0;
    pipe.steps = steps;
    pipe.nsteps = nsteps;
    pipe.pstep = 0;
    if (lane == 0) {
        pipe_start<NT>(pipe, cta, warp);
        for (int k = 0; k < ahead && k < nsteps; ++k) prefetch_l2<NT>(steps[k], cta, warp);
    }
    if (threadIdx.x == 0) {
        unsigned long long e;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(e) : "l"(ch->epoch) : "memory");
        sh.epoch = e;
    }
    bool ok = true;
    int *status = nullptr;
    for (int step = 0; step < nsteps; ++step) {
        if (lane == 0 && step + ahead < nsteps) prefetch_l2<NT>(steps[step + ahead], cta, warp);
        __syncthreads();                         // everyone is done with the last step's constants
        for (int i = threadIdx.x; i < (int)(sizeof(GroupArgs) / 4); i += kThreads)
            reinterpret_cast<uint32_t *>(&sa)[i] = reinterpret_cast<const uint32_t *>(steps + step)[i];
        __syncthreads();
        status = sa.status;
        if (cta >= sa.P) continue;
        const unsigned prevP = step > 0 ? (unsigned)steps[step - 1].P : 0u;
        if (sa.kind == kStepLinear) {
            ok = run_step<kModeA, NT, true>(sa, cta, smem, sh, pipe, ch, step, prevP);
        } else {
            if (threadIdx.x == 0) sh.go = wait_inputs(ch, step, sh.epoch, prevP, sa.status);
            __syncthreads();
            ok = sh.go != 0;
            if (ok) {
                const int chunks = (sa.K + kQChunk - 1) / kQChunk;
                quant_chunk<false, kThreads>(reinterpret_cast<const uint16_t *>(sa.X), sa.K, sa.xvec, sa.qout,
                                   sa.sout, sa.zout, sa.sym, cta / chunks, cta % chunks);
            }
        }
        if (!ok) break;
        // the step's results are written: count this CTA in
        __syncthreads();
        if (threadIdx.x == 0) signal_step(ch, step);
    }
    if (!ok && lane == 0) pipe_drain(pipe, status);
    __syncthreads();
    if (threadIdx.x == 0) leave_pass(ch, sh.epoch);
}

using ChainFn = void (*)(const ChainHeader *, const GroupArgs *);

ChainFn chain_kernel_for(int mode, int nt) {
    const bool A = mode == TL_MODE_BF16;
    switch (nt) {
        case 1: return A ? tl_chain_kernel<true, 1> : tl_chain_kernel<false, 1>;
        case 2: return A ? tl_chain_kernel<true, 2> : tl_chain_kernel<false, 2>;
        case 4: return A ? tl_chain_kernel<true, 4> : tl_chain_kernel<false, 4>;
        default: return A ? tl_chain_kernel<true, 8> : tl_chain_kernel<false, 8>;
    }
}

// ------------------------------------------------------------------ host side

struct DeviceInfo {
    std::atomic<int> init;   // 0 = unknown, 1 = ok, -1 = unsupported
    int sms;                 // written before init is set to 1
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;      // serialises first-time set-up across host threads

// Dynamic shared memory: weight ring, one slice of X, row accumulators, and
// the rows' scales and row sums.
constexpr size_t dyn_smem(int nt, int kw, int rows) {
    return (size_t)ring_bytes(nt) + (size_t)kw * 128 * nt * 2 + (size_t)rows * 16 * nt * 4 +
           (size_t)rows * 16 * 8;
}

// Attributes of the current device, looked up (and the kernels' shared
// memory limits raised) once per device; host threads may race to do it.
tl_status init_device(int dev, DeviceInfo &d) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TL_ERR_CUDA;
    if (major != 10 || minor != 3) {
        d.init.store(-1, std::memory_order_release);
        return TL_OK;
    }
    for (int mode = 0; mode < 3; ++mode)
        for (int nt = 1; nt <= 8; nt *= 2)
            if (cudaFuncSetAttribute(kernel_for(mode, nt),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)dyn_smem(nt, kMaxSlice, kMaxCtaRows)) != cudaSuccess ||
                (mode < 2 && cudaFuncSetAttribute(chain_kernel_for(mode, nt),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)dyn_smem(nt, kMaxSlice, kMaxCtaRows)) != cudaSuccess))
                return TL_ERR_CUDA;
    tl_status pst = tl_internal::prefill_init_device();
    if (pst != TL_OK) return pst;
    pst = tl_internal::head_init_device();
    if (pst != TL_OK) return pst;
    pst = tl_internal::fused_init_device();
    if (pst != TL_OK) return pst;
    pst = tl_internal::blockscale_init_device();
    if (pst != TL_OK) return pst;
    d.sms = sms;
    d.init.store(1, std::memory_order_release);
    return TL_OK;
}

tl_status device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TL_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TL_ERR_UNSUPPORTED;
    DeviceInfo &d = g_dev[dev];
    if (d.init.load(std::memory_order_acquire) == 0) {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (d.init.load(std::memory_order_acquire) == 0) {
            const tl_status st = init_device(dev, d);
            if (st != TL_OK) return st;
        }
    }
    if (d.init.load(std::memory_order_acquire) < 0) return TL_ERR_UNSUPPORTED;
    *out = &d;
    return TL_OK;
}

struct Plan {
    int R, KB, KW, KWL, NS, P, Pps, Lc, LcL, rows;
    long long U;
    size_t smem;       // dynamic shared memory for the given N
    size_t cnt_bytes;  // arrival counters (front of the workspace, after the status word)
    size_t front;      // status word, counters and exchange slots: zero between calls
    size_t back;       // partial sums of row tiles across slices (scratch)
    size_t ws_bytes;   // workspace for the given N
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// m = ceil(2^(32+l) / d) - 2^32 with l = ceil(log2 d): then for every
// 32-bit n, floor(n / d) = (umulhi(n, m) + n) >> l (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994).
FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const unsigned long long big = 1ull << (32 + l);
    FastDiv f;
    f.m = (uint32_t)((big + d - 1) / d - (1ull << 32));
    f.s = l;
    return f;
}

// The plan depends on the shapes and the SM count only, never on N, so every
// token is summed in the same order whatever the batch.
tl_status make_plan(const int *Ms, int G, int K, int N, int sms, Plan *p) {
    p->R = 0;
    for (int g = 0; g < G; ++g) p->R += (int)ceil_div(Ms[g], 16);
    p->KB = (int)ceil_div(K, 128);
    p->U = (long long)p->R * p->KB;
    if (p->U >= (1ll << 30)) return TL_ERR_SHAPE;
    // Slices: as few as kMaxSlice allows.  Each slice has its own Pps CTAs,
    // so no CTA crosses a slice boundary; each CTA gets at least KW - 1
    // units (a (row tile, slice) piece then spans at most two CTAs) and at
    // most kMaxCtaRows - 2 row tiles' worth.
    const long long slots = (long long)sms * kGridPerSm;   // CTA slots on the GPU
    p->NS = (int)ceil_div(p->KB, kMaxSlice);
    p->KW = (int)ceil_div(p->KB, p->NS);
    p->NS = (int)ceil_div(p->KB, p->KW);
    p->KWL = p->KB - (p->NS - 1) * p->KW;             // the last slice's width
    const long long su = (long long)p->R * p->KW, suL = (long long)p->R * p->KWL;
    long long pps = std::max<long long>(1, slots / p->NS);    // no CTA beyond the slots
    pps = std::min<long long>(pps, p->KW > 1 ? std::max<long long>(1, su / (p->KW - 1)) : su);
    pps = std::max<long long>(pps, ceil_div(p->R, kMaxCtaRows - 2));
    pps = std::max<long long>(1, pps);
    // One slice: whole row tiles per CTA (the grid may leave a few SMs
    // idle), so that no row tile is split between two CTAs and no CTA waits
    // on another's exchange slot.
    long long Lc = 0, LcL = 0;
    if (p->NS == 1) {
        const long long rpc = ceil_div(p->R, pps);   // row tiles per CTA
        pps = ceil_div(p->R, rpc);
        Lc = LcL = rpc * p->KW;
    } else {
        Lc = ceil_div(su, pps);
        LcL = ceil_div(suL, pps);
    }
    if ((p->KW > 1 && Lc < p->KW - 1) || (p->KWL > 1 && LcL < p->KWL - 1)) return TL_ERR_SHAPE;
    auto rows_for = [](long long L, long long kw) { return ceil_div(L + kw - 1, kw) + 1; };
    const long long rows = std::max(rows_for(Lc, p->KW), rows_for(LcL, p->KWL));
    if ((long long)p->NS * pps > (1ll << 31) - 1) return TL_ERR_SHAPE;
    p->Pps = (int)pps;
    p->P = (int)(p->NS * pps);
    p->Lc = (int)Lc;
    p->LcL = (int)LcL;
    p->rows = (int)std::min<long long>(rows, p->R);
    if (p->rows > kMaxCtaRows) return TL_ERR_SHAPE;
    const int nt = padded_tokens(std::min(std::max(N, 1), kNMax));
    const int n = std::min(std::max(N, 1), kNMax);
    p->smem = dyn_smem(nt, p->KW, p->rows);
    using tl_internal::round256;
    p->cnt_bytes = round256((size_t)p->R * 8);
    const size_t slot_bytes = p->NS == 1 ? round256((size_t)p->R * n * 16 * 8) : 0;
    p->front = tl_internal::kStatusBytes + p->cnt_bytes + slot_bytes;
    p->back = p->NS > 1 ? (size_t)p->R * p->NS * 2 * 16 * n * 4 : 0;
    p->ws_bytes = tl_internal::workspace_need(p->front, p->back);
    return TL_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
tl_status check_weights(const tl_weight *Ws, int G, int mode) {
    if (!Ws) return TL_ERR_NULL;
    if (G < 1 || G > TL_MAX_GROUP) return TL_ERR_SHAPE;
    for (int g = 0; g < G; ++g) {
        const tl_weight &w = Ws[g];
        if (!w.packed || !w.scale) return TL_ERR_NULL;
        if (mode != TL_MODE_BF16 && !w.rowsum) return TL_ERR_NULL;
        if (w.layout != TL_LAYOUT_TL2P_V2) return TL_ERR_UNSUPPORTED;
        if (w.M < 1 || w.K < 1 || w.M > TL_MAX_M || w.K > TL_MAX_K) return TL_ERR_SHAPE;
        if (w.K != Ws[0].K) return TL_ERR_SHAPE;
        if (!aligned(w.packed, 16) || !aligned(w.scale, 4)) return TL_ERR_ALIGN;
        if (mode != TL_MODE_BF16 && !aligned(w.rowsum, 4)) return TL_ERR_ALIGN;
    }
    return TL_OK;
}

size_t workspace_bytes_for(const tl_weight *Ws, int G, int N, int sms) {
    int Ms[TL_MAX_GROUP];
    for (int g = 0; g < G; ++g) Ms[g] = Ws[g].M;
    const int K = Ws[0].K;
    Plan p;
    if (make_plan(Ms, G, K, N, sms, &p) != TL_OK) return 0;
    if (tl_internal::prefill_supported(N, K))
        return std::max({tl_internal::prefill_workspace_bytes(Ws, G, N, K, TL_MODE_BF16, sms),
                         tl_internal::prefill_workspace_bytes(Ws, G, N, K, TL_MODE_I8, sms),
                         tl_internal::prefill_workspace_bytes(Ws, G, N, K, TL_MODE_I8_FUSED, sms)});
    return p.ws_bytes;
}

// Launch constants of one (grouped) linear over tokens [n0, n0 + n) with
// plan p; the workspace pieces are given by the caller.
void fill_linear(GroupArgs &a, const tl_weight *Ws, int G, const void *X, const float *s,
                 const int32_t *z, void *const *Ys, int n0, int n, int mode, int out,
                 const Plan &p, int *status, void *cnt, void *xslot, void *part) {
    std::memset(&a, 0, sizeof a);
    a.kind = kStepLinear;
    a.G = G;
    a.rt_off[0] = 0;
    const int K = Ws[0].K;
    for (int g = 0; g < G; ++g) {
        a.packed[g] = reinterpret_cast<const char *>(Ws[g].packed);
        a.scale[g] = Ws[g].scale;
        a.rowsum[g] = Ws[g].rowsum;
        a.M[g] = Ws[g].M;
        const size_t esz = out == TL_OUT_BF16 ? 2 : 4;
        a.Y[g] = static_cast<char *>(Ys[g]) + (size_t)n0 * Ws[g].M * esz;
        a.rt_off[g + 1] = a.rt_off[g] + (int)ceil_div(Ws[g].M, 16);
    }
    a.R = p.R; a.KB = p.KB; a.KW = p.KW; a.KWL = p.KWL; a.NS = p.NS; a.K = K; a.U = (int)p.U;
    a.Pps = p.Pps; a.Lc = p.Lc; a.LcL = p.LcL; a.rows = p.rows; a.P = p.P;
    a.kwr = p.KW; a.rowsr = p.rows;
    a.dKW = make_fastdiv((uint32_t)p.KW);
    a.dKWL = make_fastdiv((uint32_t)p.KWL);
    const size_t xsz = mode == TL_MODE_I8 ? 1 : 2;
    a.X = static_cast<const char *>(X) + (size_t)n0 * K * xsz;
    a.s = s ? s + n0 : nullptr;
    a.z = z ? z + n0 : nullptr;
    a.N = n; a.mode = mode; a.out = out;
    a.xvec = aligned(a.X, 16) && (K % (mode == TL_MODE_I8 ? 16 : 8)) == 0;
    a.cnt = static_cast<unsigned long long *>(cnt);
    a.xslot = static_cast<unsigned long long *>(xslot);
    a.part = static_cast<float *>(part);
    a.status = status;
}

tl_status launch_chunk(const tl_weight *Ws, int G, const void *X, const float *s,
                       const int32_t *z, void *const *Ys, int n0, int n, int mode, int out,
                       void *ws, size_t ws_bytes, unsigned flags, cudaStream_t stream,
                       const DeviceInfo &dev) {
    int Ms[TL_MAX_GROUP];
    for (int g = 0; g < G; ++g) Ms[g] = Ws[g].M;
    Plan p;
    const tl_status pst = make_plan(Ms, G, Ws[0].K, n, dev.sms, &p);
    if (pst != TL_OK) return pst;
    if (!ws || ws_bytes < p.ws_bytes) return TL_ERR_WORKSPACE;
    char *wsb = static_cast<char *>(ws) + tl_internal::kStatusBytes;
    GroupArgs a;
    fill_linear(a, Ws, G, X, s, z, Ys, n0, n, mode, out, p, static_cast<int *>(ws), wsb,
                wsb + p.cnt_bytes,
                static_cast<char *>(ws) + tl_internal::scratch_offset(ws_bytes, p.back));
    a.sym = mode == TL_MODE_I8_FUSED && (flags & TL_FLAG_SYMMETRIC) ? 1 : 0;

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & TL_FLAG_PDL) ? 1 : 0;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, kernel_for(mode, padded_tokens(n)), a);
    if (le != cudaSuccess) return TL_ERR_CUDA;
    return TL_OK;
}


// ------------------------------------------------------------------ chains (host)
constexpr uint32_t kChainMagic = 0x544C4348u;   // "TLCH"
constexpr size_t kChainHead = 256;              // image bytes before the steps
constexpr int kChainLookahead = 3;              // steps prefetched into L2 ahead of use

// The image's first bytes: the device-side header, then what tl_chain_run
// reads on the host.
struct ChainHostHead {
    ChainHeader hdr;
    uint32_t magic;
    int32_t grid, smem, nt, mode, total;
};
static_assert(sizeof(ChainHostHead) <= kChainHead, "chain head");
static_assert(sizeof(GroupArgs) % 4 == 0, "steps are copied as words");

// Workspace of a chain: status word, per-step counters, the row-tile
// counters and exchange slots every linear step shares (all zero between
// launches), then scratch: split-K pieces and, in mode B, the quantised
// activations of the current step.
struct ChainLayout {
    size_t epoch_off, steps_off, cnt_off, xslot_off, part_off, q_off, s_off, z_off, bytes, front;
    int kwr, rowsr, grid, total;
};

tl_status chain_layout(const tl_chain_step *st, int nsteps, int N, int mode, int sms,
                       ChainLayout *L) {
    using tl_internal::round256;
    size_t cnt_b = 0, xslot_b = 0, part_b = 0;
    int kmax = 0;
    L->kwr = 1;
    L->rowsr = 1;
    L->grid = 1;
    for (int i = 0; i < nsteps; ++i) {
        int Ms[TL_MAX_GROUP];
        for (int g = 0; g < st[i].G; ++g) Ms[g] = st[i].Ws[g].M;
        Plan p;
        const tl_status ps = make_plan(Ms, st[i].G, st[i].Ws[0].K, N, sms, &p);
        if (ps != TL_OK) return ps;
        cnt_b = std::max(cnt_b, p.cnt_bytes);
        if (p.NS == 1) xslot_b = std::max(xslot_b, round256((size_t)p.R * N * 16 * 8));
        part_b = std::max(part_b, round256(p.back));
        L->kwr = std::max(L->kwr, p.KW);
        L->rowsr = std::max(L->rowsr, p.rows);
        L->grid = std::max(L->grid, p.P);
        kmax = std::max(kmax, st[i].Ws[0].K);
        if (mode == TL_MODE_I8)
            L->grid = std::max(L->grid, (int)ceil_div(st[i].Ws[0].K, kQChunk) * N);
    }
    L->total = mode == TL_MODE_I8 ? 2 * nsteps : nsteps;
    L->epoch_off = tl_internal::kStatusBytes;
    L->steps_off = L->epoch_off + 256;
    L->cnt_off = L->steps_off + round256((size_t)L->total * 8);
    L->xslot_off = L->cnt_off + cnt_b;
    L->front = L->xslot_off + xslot_b;
    L->part_off = L->front;
    L->q_off = L->part_off + part_b;
    L->s_off = L->q_off + (mode == TL_MODE_I8 ? round256((size_t)N * kmax) : 0);
    L->z_off = L->s_off + (mode == TL_MODE_I8 ? 256 : 0);
    L->bytes = L->z_off + (mode == TL_MODE_I8 ? 256 : 0);
    return TL_OK;
}

tl_status check_chain(const tl_chain_step *st, int nsteps, int N, int mode, int out) {
    if (!st) return TL_ERR_NULL;
    if (nsteps < 1 || nsteps > TL_MAX_CHAIN || N < 1 || N > kNMax) return TL_ERR_SHAPE;
    if (mode != TL_MODE_BF16 && mode != TL_MODE_I8) return TL_ERR_MODE;
    if (out != TL_OUT_F32 && out != TL_OUT_BF16 && out != TL_OUT_I32_RAW) return TL_ERR_MODE;
    if (out == TL_OUT_I32_RAW && mode != TL_MODE_I8) return TL_ERR_MODE;
    for (int i = 0; i < nsteps; ++i) {
        const tl_status ws = check_weights(st[i].Ws, st[i].G, mode);
        if (ws != TL_OK) return ws;
        if (!st[i].X || !st[i].Ys) return TL_ERR_NULL;
        if (!aligned(st[i].X, 2)) return TL_ERR_ALIGN;
        for (int g = 0; g < st[i].G; ++g) {
            if (!st[i].Ys[g]) return TL_ERR_NULL;
            if (!aligned(st[i].Ys[g], out == TL_OUT_BF16 ? 2 : 4)) return TL_ERR_ALIGN;
        }
    }
    return TL_OK;
}

}  // namespace

namespace tl_internal {

tl_status device_sms(int *sms) {
    DeviceInfo *dev = nullptr;
    const tl_status st = device_info(&dev);
    if (st != TL_OK) return st;
    *sms = dev->sms;
    return TL_OK;
}

tl_status decode_scratch_bytes(const tl_weight *Ws, int G, size_t *need, size_t *zeroed) {
    DeviceInfo *dev = nullptr;
    const tl_status st = device_info(&dev);
    if (st != TL_OK) return st;
    int Ms[TL_MAX_GROUP];
    for (int g = 0; g < G; ++g) Ms[g] = Ws[g].M;
    Plan p;
    const tl_status pst = make_plan(Ms, G, Ws[0].K, kNMax, dev->sms, &p);  // chunks <= 8 tokens
    if (pst != TL_OK) return pst;
    *need = p.ws_bytes;
    *zeroed = p.front;
    return TL_OK;
}

tl_status launch_quant(const void *X_bf16, int N, int K, void *Q, bool bf16_out, float *s,
                       int32_t *z, int symmetric, cudaStream_t stream) {
    // 16-byte rows: vector loads of X, 8-byte (int8) or 16-byte (bf16) stores of Q
    const int vec = aligned(X_bf16, 16) && aligned(Q, bf16_out ? 16 : 8) && (K % 8) == 0;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(quant_held(vec, K) ? 1u : (unsigned)((K + kQChunk - 1) / kQChunk), (unsigned)N);
    cfg.blockDim = dim3(kQThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le =
        bf16_out ? cudaLaunchKernelEx(&cfg, tl_quant_kernel<true>, static_cast<const uint16_t *>(X_bf16), K,
                                      vec, Q, s, z, symmetric ? 1 : 0)
                 : cudaLaunchKernelEx(&cfg, tl_quant_kernel<false>, static_cast<const uint16_t *>(X_bf16), K,
                                      vec, Q, s, z, symmetric ? 1 : 0);
    return le == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

tl_status launch_decode(const tl_weight *Ws, int G, const void *X, const float *s,
                        const int32_t *z, void *const *Ys, int N, int mode, int out, void *ws,
                        size_t ws_bytes, unsigned flags, cudaStream_t stream) {
    DeviceInfo *dev = nullptr;
    tl_status st = device_info(&dev);
    if (st != TL_OK) return st;
    for (int n0 = 0; n0 < N; n0 += kNMax) {
        const int n = N - n0 < kNMax ? N - n0 : kNMax;
        st = launch_chunk(Ws, G, X, s, z, Ys, n0, n, mode, out, ws, ws_bytes, flags, stream,
                          *dev);
        if (st != TL_OK) return st;
    }
    return TL_OK;
}

}  // namespace tl_internal

extern "C" {

size_t tl_workspace_bytes(const tl_weight *Ws, int G, int N) {
    if (!Ws || G < 1 || G > TL_MAX_GROUP || N < 1) return 0;
    DeviceInfo *dev = nullptr;
    int sms = 148;
    if (device_info(&dev) == TL_OK) sms = dev->sms;
    for (int g = 0; g < G; ++g)
        if (Ws[g].M < 1 || Ws[g].K < 1 || Ws[g].K != Ws[0].K) return 0;
    return workspace_bytes_for(Ws, G, N, sms);
}

tl_status tl_decode_plan(const tl_weight *Ws, int G, int N, int sms, int32_t *plan) {
    if (!Ws || !plan) return TL_ERR_NULL;
    if (G < 1 || G > TL_MAX_GROUP || N < 1 || sms < 1) return TL_ERR_SHAPE;
    int Ms[TL_MAX_GROUP];
    for (int g = 0; g < G; ++g) {
        if (Ws[g].M < 1 || Ws[g].K < 1 || Ws[g].M > TL_MAX_M || Ws[g].K > TL_MAX_K ||
            Ws[g].K != Ws[0].K)
            return TL_ERR_SHAPE;
        Ms[g] = Ws[g].M;
    }
    const int n = std::min(N, kNMax);
    Plan p;
    const tl_status st = make_plan(Ms, G, Ws[0].K, n, sms, &p);
    if (st != TL_OK) return st;
    const int32_t v[TL_PLAN_FIELDS] = {p.R,  p.KB, p.NS,   p.KW,   p.KWL,
                                       p.Pps, p.P, p.Lc,   p.LcL,  p.rows,
                                       kWarps, chunk_tiles(padded_tokens(n)), kGridPerSm, kMaxCtaRows};
    for (int i = 0; i < TL_PLAN_FIELDS; ++i) plan[i] = v[i];
    return TL_OK;
}

tl_status tl_quantize_act(const void *X_bf16, int N, int K, int8_t *Q, float *s, int32_t *z,
                          int symmetric, void *stream) {
    if (!X_bf16 || !Q || !s || !z) return TL_ERR_NULL;
    if (N < 1 || K < 1 || K > TL_MAX_K) return TL_ERR_SHAPE;
    if (!aligned(X_bf16, 2) || !aligned(s, 4) || !aligned(z, 4)) return TL_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    const tl_status st = device_info(&dev);
    if (st != TL_OK) return st;
    if (N > 65535) return TL_ERR_SHAPE;
    return tl_internal::launch_quant(X_bf16, N, K, Q, false, s, z, symmetric,
                                     static_cast<cudaStream_t>(stream));
}

tl_status tl_linear_group(const tl_weight *Ws, int G, const void *X, const float *s,
                          const int32_t *z, void *const *Ys, int N, int mode, int out_dtype,
                          void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream) {
    if (mode != TL_MODE_BF16 && mode != TL_MODE_I8 && mode != TL_MODE_I8_FUSED) return TL_ERR_MODE;
    tl_status st = check_weights(Ws, G, mode);
    if (st != TL_OK) return st;
    if (out_dtype != TL_OUT_F32 && out_dtype != TL_OUT_BF16 && out_dtype != TL_OUT_I32_RAW)
        return TL_ERR_MODE;
    if (out_dtype == TL_OUT_I32_RAW && mode != TL_MODE_I8) return TL_ERR_MODE;
    if (!X || !Ys) return TL_ERR_NULL;
    if (N < 1) return TL_ERR_SHAPE;
    if (mode == TL_MODE_I8 && (!s || !z)) return TL_ERR_NULL;
    if (mode != TL_MODE_I8 && !aligned(X, 2)) return TL_ERR_ALIGN;
    if (mode == TL_MODE_I8 && (!aligned(s, 4) || !aligned(z, 4))) return TL_ERR_ALIGN;
    for (int g = 0; g < G; ++g) {
        if (!Ys[g]) return TL_ERR_NULL;
        if (!aligned(Ys[g], out_dtype == TL_OUT_BF16 ? 2 : 4)) return TL_ERR_ALIGN;
    }
    if (!workspace) return TL_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TL_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != TL_OK) return st;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (tl_internal::prefill_supported(N, Ws[0].K)) {
        if (mode == TL_MODE_BF16 && !aligned(X, 16)) return TL_ERR_ALIGN;
        return tl_internal::launch_prefill(Ws, G, X, s, z, Ys, N, mode, out_dtype, workspace,
                                           workspace_bytes, flags, cs);
    }
    for (int n0 = 0; n0 < N; n0 += kNMax) {
        const int n = N - n0 < kNMax ? N - n0 : kNMax;
        st = launch_chunk(Ws, G, X, s, z, Ys, n0, n, mode, out_dtype, workspace,
                          workspace_bytes, flags, cs, *dev);
        if (st != TL_OK) return st;
    }
    return TL_OK;
}

size_t tl_chain_image_bytes(int nsteps, int mode) {
    if (nsteps < 1 || nsteps > TL_MAX_CHAIN) return 0;
    const size_t total = mode == TL_MODE_I8 ? 2 * (size_t)nsteps : (size_t)nsteps;
    return kChainHead + total * sizeof(GroupArgs);
}

size_t tl_chain_workspace_bytes(const tl_chain_step *steps, int nsteps, int N, int mode) {
    if (check_chain(steps, nsteps, N, mode, TL_OUT_F32) != TL_OK) return 0;
    DeviceInfo *dev = nullptr;
    int sms = 148;
    if (device_info(&dev) == TL_OK) sms = dev->sms;
    ChainLayout L;
    if (chain_layout(steps, nsteps, N, mode, sms, &L) != TL_OK) return 0;
    return L.bytes;
}

tl_status tl_chain_encode(const tl_chain_step *steps, int nsteps, int N, int mode, int out_dtype,
                          const unsigned *gate, long long wait_limit, void *workspace,
                          size_t workspace_bytes, void *image, size_t image_bytes) {
    tl_status st = check_chain(steps, nsteps, N, mode, out_dtype);
    if (st != TL_OK) return st;
    if (!image) return TL_ERR_NULL;
    if (image_bytes < tl_chain_image_bytes(nsteps, mode)) return TL_ERR_SHAPE;
    if (!workspace) return TL_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TL_ERR_ALIGN;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != TL_OK) return st;
    ChainLayout L;
    st = chain_layout(steps, nsteps, N, mode, dev->sms, &L);
    if (st != TL_OK) return st;
    if (workspace_bytes < L.bytes) return TL_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    char *img = static_cast<char *>(image);
    std::memset(img, 0, tl_chain_image_bytes(nsteps, mode));
    GroupArgs *sa = reinterpret_cast<GroupArgs *>(img + kChainHead);
    int8_t *Q = reinterpret_cast<int8_t *>(ws + L.q_off);
    float *qs = reinterpret_cast<float *>(ws + L.s_off);
    int32_t *qz = reinterpret_cast<int32_t *>(ws + L.z_off);
    int k = 0;
    for (int i = 0; i < nsteps; ++i) {
        const tl_chain_step &c = steps[i];
        const int K = c.Ws[0].K;
        int Ms[TL_MAX_GROUP];
        for (int g = 0; g < c.G; ++g) Ms[g] = c.Ws[g].M;
        Plan p;
        st = make_plan(Ms, c.G, K, N, dev->sms, &p);
        if (st != TL_OK) return st;
        const void *X = c.X;
        if (mode == TL_MODE_I8) {
            // the step's activations, quantised per token by the chain itself
            GroupArgs &q = sa[k++];
            std::memset(&q, 0, sizeof q);
            q.kind = kStepQuant;
            q.K = K;
            q.N = N;
            q.X = c.X;
            q.xvec = aligned(c.X, 16) && (K % 8) == 0;
            q.qout = Q;
            q.sout = qs;
            q.zout = qz;
            q.P = (int)ceil_div(K, kQChunk) * N;
            q.status = reinterpret_cast<int *>(ws);
            X = Q;
        }
        GroupArgs &a = sa[k++];
        fill_linear(a, c.Ws, c.G, X, mode == TL_MODE_I8 ? qs : nullptr,
                    mode == TL_MODE_I8 ? qz : nullptr, c.Ys, 0, N, mode, out_dtype, p,
                    reinterpret_cast<int *>(ws), ws + L.cnt_off, ws + L.xslot_off,
                    ws + L.part_off);
    }
    for (int i = 0; i < L.total; ++i) {
        sa[i].kwr = L.kwr;
        sa[i].rowsr = L.rowsr;
    }
    const int nt = padded_tokens(N);
    const size_t smem = dyn_smem(nt, L.kwr, L.rowsr);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_kernel_for(mode, nt), kThreads,
                                                      smem) != cudaSuccess)
        return TL_ERR_CUDA;
    if ((long long)per_sm * dev->sms < L.grid) return TL_ERR_UNSUPPORTED;
    ChainHostHead &h = *reinterpret_cast<ChainHostHead *>(img);
    h.hdr.cnt = reinterpret_cast<unsigned long long *>(ws + L.steps_off);
    h.hdr.epoch = reinterpret_cast<unsigned long long *>(ws + L.epoch_off);
    h.hdr.gate = gate;
    h.hdr.wait_limit = wait_limit > 0 ? wait_limit : kWaitLimit;
    h.hdr.nsteps = L.total;
    h.hdr.lookahead = kChainLookahead;
    h.magic = kChainMagic;
    h.grid = L.grid;
    h.smem = (int32_t)smem;
    h.nt = nt;
    h.mode = mode;
    h.total = L.total;
    return TL_OK;
}

tl_status tl_chain_run(const void *image, const void *image_device, void *stream) {
    if (!image || !image_device) return TL_ERR_NULL;
    if (!aligned(image_device, 16)) return TL_ERR_ALIGN;
    ChainHostHead h;
    std::memcpy(&h, image, sizeof h);
    if (h.magic != kChainMagic) return TL_ERR_BAD_VALUE;
    DeviceInfo *dev = nullptr;
    const tl_status st = device_info(&dev);
    if (st != TL_OK) return st;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)h.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)h.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once, or no launch
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const char *dimg = static_cast<const char *>(image_device);
    const cudaError_t le = cudaLaunchKernelEx(
        &cfg, chain_kernel_for(h.mode, h.nt), reinterpret_cast<const ChainHeader *>(dimg),
        reinterpret_cast<const GroupArgs *>(dimg + kChainHead));
    return le == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

tl_status tl_linear(const tl_weight *W, const void *X, const float *s, const int32_t *z, void *Y,
                    int N, int mode, int out_dtype, void *workspace, size_t workspace_bytes,
                    unsigned flags, void *stream) {
    void *Ys[1] = {Y};
    return tl_linear_group(W, 1, X, s, z, Ys, N, mode, out_dtype, workspace, workspace_bytes,
                           flags, stream);
}

}  // extern "C"
