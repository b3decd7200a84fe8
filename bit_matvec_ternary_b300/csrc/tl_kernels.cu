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
//   most two CTAs.  The 8 warps split the CTA's units into contiguous ranges.
//   Weights.  Each warp streams its units with cp.async.bulk into its own
//   ring of shared-memory slots (up to 8 tiles per copy, completing on the
//   slot's mbarrier), running ahead across slices.  A TL2P v2 tile is in
//   mma.m16n8k16 A-fragment order and each 2-bit field holds 1 - w, so
//   register j of k-step m is (word >> 8*(m/4)) & (0x00030003 << 2*(m%4)):
//   a bf16x2 pair whose halves are (1 - w) * 2^(2q - 133), q = m%4 -- bf16
//   subnormals (or, for field 10 at q == 3, the smallest normal), exactly
//   linear in the field.  One AND per two weights, plus one shift per word.
//   Activations.  Staged per slice in shared memory in B-fragment order,
//   multiplied by 2^67 (an exponent add, exact), so a class-q product is
//   (1 - w) * x * 2^(2q - 66), exact in fp32; the tensor cores form the sums,
//   one accumulator chain per class, and each chain is rescaled exactly when
//   a run of tiles is folded.  The staging also sums x per 128-column block,
//   and a row's result is (sum of x over its blocks) - sum (1 - w) x.
//   Activations outside [2^-60, 2^61) in magnitude (mode A only) switch that
//   token's slice to a scale chosen from its largest exponent.  Columns
//   n >= N are zero and their results are discarded, so no lane is
//   predicated off.
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
#include <cstring>

namespace {

constexpr int kWarps = 8;             // warps per CTA of the N <= 8 kernel
constexpr int kCtasPerSm = 2;         // resident CTAs per SM (registers and shared memory allow 2)
// CTAs per SM in a launch's grid.
constexpr int kGridPerSm = 2;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 2;             // bulk copies in flight per warp
// Tiles (512 B each) per bulk copy: 8, or 4 at eight tokens, where the
// staged activations take 64 KB (two CTAs still fit in one SM's shared
// memory for plans of up to 8 row tiles per CTA).
__host__ __device__ constexpr int chunk_tiles(int nt) { return nt <= 4 ? 8 : 4; }
__host__ __device__ constexpr int ring_bytes(int nt) { return kWarps * kSlots * chunk_tiles(nt) * 512; }
constexpr int kNMax = 8;              // tokens per launch (mma n = 8)
constexpr int kMaxDevices = 64;
constexpr int kMaxSlice = 32;         // 128-column blocks per K slice (64 KB of X at 8 tokens)
constexpr int kMaxCtaRows = 16;       // row tiles one CTA may touch in one slice
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

// Everything below reads these launch constants.
struct GroupArgs {
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
                                          float sc, int rs) {
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
        const int corrected = iacc - a.z[n] * rs;
        y = __fmul_rn(__fmul_rn((float)corrected, a.s[n]), sc);
    }
    if (a.out == TL_OUT_F32)
        reinterpret_cast<float *>(a.Y[gi])[(long long)n * M + m] = y;
    else
        reinterpret_cast<__nv_bfloat16 *>(a.Y[gi])[(long long)n * M + m] = __float2bfloat16_rn(y);
}

// The 16 x N results of row tile r held as v[n * 16 + row], with the row
// tile's scales and row sums in sc[16], rs[16].  One warp; lane (g, t)
// stores rows g, g+8 of tokens 2t, 2t+1.
__device__ __forceinline__ void store_row_tile(const GroupArgs &a, int r, const float *v,
                                               const float *sc, const int *rs, int lane) {
    const int g = lane >> 2, t = lane & 3;
    int gi = 0;
    while (gi + 1 < a.G && a.rt_off[gi + 1] <= r) ++gi;
    const int rl = r - a.rt_off[gi];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = g + 8 * h, m = rl * 16 + i, n = 2 * t + e;
            if (m < a.M[gi] && n < a.N) store_out(a, gi, m, n, v[n * 16 + i], sc[i], rs[i]);
        }
}

// Row tile r of a one-slice launch whose blocks are split between two CTAs:
// each CTA swaps its piece of every element into the element's exchange slot
// (bit 32 set = occupied).  The CTA that finds the other piece there adds the
// two, stores the element and empties the slot; the other finds the slot
// empty and is done.  One atomic round trip, and the sum does not depend on
// which CTA comes second (a + b == b + a in floating point).
__device__ __forceinline__ void exchange_row_tile(const GroupArgs &a, int r, const float *v,
                                                  const float *sc, const int *rs, int lane) {
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
                              sc[i], rs[i]);
            }
        }
}

// One 128-column block of one 16-row tile: 8 MMAs (k-steps m = 0..7) over
// the lane's 16-byte slice of the tile (w) and the 4 B-fragment quarters (b).
// Register j of k-step m is word j shifted right by 8*(m/4) and masked to the
// fields at bits 2*(m%4) and 16 + 2*(m%4).
__device__ __forceinline__ void tile_mma(float (&c)[4][4], const uint4 &w, const uint4 (&b)[4]) {
    const uint32_t hx = w.x >> 8, hy = w.y >> 8, hz = w.z >> 8, hw = w.w >> 8;
    // four independent accumulator chains; consecutive MMAs never share one
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t F = 0x00030003u << (2 * (m & 3));
        const uint32_t a0 = (m < 4 ? w.x : hx) & F, a1 = (m < 4 ? w.y : hy) & F;
        const uint32_t a2 = (m < 4 ? w.z : hz) & F, a3 = (m < 4 ? w.w : hw) & F;
        const uint4 &q = b[m >> 1];
        mma_bf16_16816(c[m & 3], a0, a1, a2, a3, (m & 1) ? q.z : q.x, (m & 1) ? q.w : q.y);
    }
}

// VPL consecutive activations of token n from column k0 (VPL = 8 bf16 in mode
// A, 16 int8 in mode B; k0 a multiple of VPL): one 16-byte load when X allows
// it, else element loads; columns >= K read as 0.
template <bool kModeA>
__device__ __forceinline__ uint4 load_group(const GroupArgs &a, int n, int k0) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (kModeA) {
        const uint16_t *x = reinterpret_cast<const uint16_t *>(a.X) + (long long)n * a.K + k0;
        if (a.xvec) {
            if (k0 < a.K) v = __ldg(reinterpret_cast<const uint4 *>(x));
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (k0 + e < a.K) w[e >> 1] |= (uint32_t)x[e] << (16 * (e & 1));
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        const uint8_t *x = reinterpret_cast<const uint8_t *>(a.X) + (long long)n * a.K + k0;
        if (a.xvec) {
            if (k0 < a.K) v = __ldg(reinterpret_cast<const uint4 *>(x));
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (k0 + e < a.K) w[e >> 2] |= (uint32_t)x[e] << (8 * (e & 3));
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
// at blk.  Writes the group's words in B-fragment order, times 2^kT, and
// returns the group's sum in a fixed order and (mode A) the mask of halves
// outside the fixed window.  A zero x writes zeros.
template <bool kModeA, int NT>
__device__ __forceinline__ void stage_group(uint32_t *blk, int n, int o, const uint4 &x,
                                            float &sum, uint32_t &bad) {
    const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
    sum = 0.f;
    bad = 0u;
    if (kModeA) {
        const int m = o >> 1, qd = m >> 1;
        uint32_t *dst = blk + (qd * NT + n) * 16 + 2 * (m & 1) + (o & 1);
        uint32_t st[4];
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
            const uint32_t v = wd[tt];
            sum = __fadd_rn(__fadd_rn(sum, __uint_as_float(v << 16)),
                            __uint_as_float(v & 0xFFFF0000u));
            // per half: nonzero, and exponent outside [kWinLo, kWinHi]
            const uint32_t nz = __vcmpne2(v & 0x7FFF7FFFu, 0u);
            const uint32_t off = __vsub2(v & 0x7F807F80u, (uint32_t)kWinLo * 0x00800080u);
            bad |= __vcmpgtu2(off, (uint32_t)(kWinHi - kWinLo) * 0x00800080u) & nz;
            st[tt] = v + ((uint32_t)kT * 0x00800080u & nz);
        }
        // store word tt = (it + qd) % 4 at step it: the lanes of one block
        // quarter apart then write different banks
        store_rotated(dst, st, qd);
    } else {
        const int m = o, qd = m >> 1;
        uint32_t *dst = blk + (qd * NT + n) * 16 + 2 * (m & 1);
        const float two_t = __int_as_float((kT + 127) << 23);
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
template <bool kModeA, int SB>
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
            v[i] = load_group<kModeA>(a, n, (P.kb0 + jb) * 128 + o * VPL);
        }
    }
}

// Kernel launch helpers shared with the host side.
// ------------------------------------------------------------ kernel
// kModeA: bf16 activations (else int8 from the quantiser).  NT: token
// columns staged (a power of two >= N).
template <bool kModeA, int NT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
tl_mma_kernel(const __grid_constant__ GroupArgs a) {
    constexpr int CH = chunk_tiles(NT);         // tiles per bulk copy
    constexpr int SLOT = CH * 512;
    constexpr int XQ = NT * 4;                  // uint4 per 32-column quarter
    constexpr int XB = 4 * XQ;                  // uint4 per 128-column block
    constexpr int RV = 16 * NT;                 // floats per row-tile result
    constexpr int VPL = kModeA ? 8 : 16;        // activations per staging group
    constexpr int LB = 128 / VPL;               // staging groups per block
    constexpr int SB = stage_batch(NT, kModeA); // staging loads in flight per thread
    constexpr bool kAsyncX = NT >= 4;           // stage X with cp.async (when X allows 16-byte copies)
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;                                                // [kWarps][kSlots][SLOT]
    uint4 *xs = reinterpret_cast<uint4 *>(smem + ring_bytes(NT));      // one slice of X
    float *acc = reinterpret_cast<float *>(smem + ring_bytes(NT) + a.KW * XB * 16);  // [rows][RV]
    float *scl = acc + a.rows * RV;                                      // [rows][16] scales
    int *rsm = reinterpret_cast<int *>(scl + a.rows * 16);               // [rows][16] row sums
    __shared__ float bslot[kWarps][2][RV];      // boundary pieces of the current slice
    __shared__ int bslot_row[kWarps][2];
    __shared__ float osum[kMaxSlice][NT];       // sum of x per block of the slice
    __shared__ float opre[kMaxSlice + 1][NT];   // prefix sums of osum
    __shared__ int texp[NT];                    // T per token: X is staged times 2^T
    __shared__ int redo;                        // tokens outside the fixed window (bit mask)
    __shared__ int emax[NT];
    __shared__ __align__(8) unsigned long long bars[kWarps][kSlots];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int N = a.N;
    // this CTA's units: range c_in of its slice (none past the last slice)
    int cu0 = a.U, cu1 = a.U;
    {
        const int sig_c = (int)blockIdx.x / a.Pps, c_in = (int)blockIdx.x - sig_c * a.Pps;
        if (sig_c < a.NS) {
            const int su = a.R * slice_width(a, sig_c);
            const int lc = sig_c == a.NS - 1 ? a.LcL : a.Lc;
            const int base = sig_c * a.R * a.KW;
            const int off = (int)min((long long)c_in * lc, (long long)su);
            cu0 = base + off;
            cu1 = base + min(off + lc, su);
        }
    }
    const int sunits = a.R * a.KW;
    const int sig0 = cu0 / sunits;
    const int sig1 = cu1 > cu0 ? (cu1 - 1) / sunits + 1 : sig0;
    uint32_t *xw = reinterpret_cast<uint32_t *>(xs);
    const uint32_t xs_s = smem_u32(xs);

    // The dependent launch may be scheduled at once; it only streams weights
    // until this grid has finished.
    griddep_launch();

    // Weights do not depend on the previous kernel: each warp's lane 0 sets up
    // its ring and starts its first copies before waiting for it.  The
    // producer then runs kSlots chunks ahead of the warp's consumer, across
    // slices.
    const uint32_t ring_w = smem_u32(ring) + warp * (kSlots * SLOT);
    const uint32_t bar_w = smem_u32(&bars[warp][0]);
    Cursor pc;
    pc.sigma = sig0;
    bool pc_on = cursor_enter(a, cu0, cu1, sig1, warp, pc);
    int pgi = 0;
    const char *prow = pc_on ? row_base(a, pc.r, pgi) : nullptr;
    auto produce = [&](int slot_) {
        const int n = min(CH, min(pc.uend - pc.u, pc.kw - pc.b));
        bulk_load(ring_w + slot_ * SLOT, prow + (long long)(pc.kb0 + pc.b) * 512, n * 512,
                  bar_w + 8u * slot_);
        pc.u += n;
        pc.b += n;
        if (pc.b == pc.kw) {
            pc.b = 0;
            ++pc.r;
            if (pgi + 1 < a.G && pc.r == a.rt_off[pgi + 1]) prow = a.packed[++pgi];
            else prow += (long long)a.KB * 512;
        }
        if (pc.u == pc.uend) {
            ++pc.sigma;
            pc_on = cursor_enter(a, cu0, cu1, sig1, warp, pc);
            if (pc_on) prow = row_base(a, pc.r, pgi);
        }
    };
    if (lane == 0) {
        for (int k = 0; k < kSlots; ++k) mbar_init(bar_w + 8u * k, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int k = 0; k < kSlots && pc_on; ++k) produce(k);
        // and the rest of this warp's tiles into L2, while the previous
        // launch may still be running
        if (pc_on) {
            Cursor q = pc;
            int qg = pgi;
            const char *qr = prow;
            for (bool on = true; on;) {
                const int n = min(CH, min(q.uend - q.u, q.kw - q.b));
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 qr + (long long)(q.kb0 + q.b) * 512),
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
    }
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
    if (N < NT)   // the columns past the batch stay zero in every slice
        for (int i = threadIdx.x; i < a.KW * 64 * NT; i += kThreads)
            if (((i >> 4) % NT) >= N) xw[i] = 0u;
    // Warm L2 (and the address translation) for this CTA's activations; a
    // prefetch returns no data, so it may run before the previous kernel has
    // written them.  One 128-byte line per thread per step, addresses inside
    // each row's columns [k_lo, k_hi).
    if (sig1 > sig0) {
        constexpr int EB = kModeA ? 2 : 1;
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

    // Now the activations, written by the previous kernel.
    griddep_wait();
    uint4 xv[SB];
    if (!(kAsyncX && a.xvec)) stage_load<kModeA, SB>(a, P, 0, xv);

    Cursor cc;
    cc.sigma = sig0;
    bool cc_on = cursor_enter(a, cu0, cu1, sig1, warp, cc);
    int slot = 0;
    uint32_t phases = 0;                        // parity bit per slot
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
                constexpr int EB = kModeA ? 2 : 1;
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
                        stage_group<kModeA, NT>(blk, n, o, v[j], sum, bad);
#pragma unroll
                        for (int off = LB / 2; off > 0; off >>= 1)
                            sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, off));
                        if (n < N && o == 0) osum[jb][n] = sum;
                        if (kModeA && n < N && bad) atomicOr(&redo, 1 << n);
                    }
                }
            } else
            for (int base = 0; base < total; base += kThreads * SB) {
                if (sigma != sig0 || base != 0) stage_load<kModeA, SB>(a, P, base, xv);
#pragma unroll
                for (int i = 0; i < SB; ++i) {
                    if (base + i * kThreads >= total) break;   // uniform over the block
                    const int idx = base + i * kThreads + (int)threadIdx.x;
                    const bool valid = idx < total;
                    const int q = idx / LB, o = idx % LB;
                    const int n = valid ? fdiv(q, dv) : 0, jb = q - n * P.kw;
                    float sum = 0.f;
                    uint32_t bad = 0u;
                    if (valid) stage_group<kModeA, NT>(xw + jb * NT * 64, n, o, xv[i], sum, bad);
#pragma unroll
                    for (int off = LB / 2; off > 0; off >>= 1)
                        sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, off));
                    if (valid && (lane % LB) == 0) osum[jb][n] = sum;
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
                for (int k = klo + threadIdx.x; k < khi; k += kThreads) e = max(e, ((uint32_t)x[k] >> 7) & 0xFFu);
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
                const uint32_t lo = k < a.K ? x[k] : 0u, hi = k + 1 < a.K ? x[k + 1] : 0u;
                const int d = 254 - emax[n];
                xw[idx] = scale_any(lo, d) | (scale_any(hi, d) << 16);
            }
            __syncthreads();
            if (threadIdx.x == 0) redo = 0;
            if (threadIdx.x < NT) emax[threadIdx.x] = 0;
        }

        // prefix sums of the block sums, one warp per token column
        if (warp < NT) {
            const int n = warp;
            float v0 = lane < P.kw ? osum[lane][n] : 0.f;
            float v1 = lane + 32 < P.kw ? osum[lane + 32][n] : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, v0, off);
                const float y1 = __shfl_up_sync(0xffffffffu, v1, off);
                if (lane >= off) { v0 = __fadd_rn(v0, y0); v1 = __fadd_rn(v1, y1); }
            }
            v1 = __fadd_rn(v1, __shfl_sync(0xffffffffu, v0, 31));
            if (lane == 0) opre[0][n] = 0.f;
            if (lane < P.kw) opre[lane + 1][n] = v0;
            if (lane + 32 < P.kw) opre[lane + 33][n] = v1;
        }
        // this lane's tokens 2t, 2t+1: chain q holds the products of k-step
        // class q, (1 - w) x 2^(2q - 133 + T); undo 2^(2q - 133 + T) with two
        // exact factors each
        int tx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) tx[e] = texp[min(2 * t + e, NT - 1)];

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
                    tile_mma(c, w, bq);
                    w = wn;
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) bq[qd] = bn[qd];
                }
            } else {
                for (int i = 0; i < n; ++i) {
                    const uint4 w = tiles[i * 32];
                    uint4 bq[4];
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) bq[qd] = xb[i * XB + qd * XQ];
                    tile_mma(c, w, bq);
                }
            }
            // end of a run of one row tile: this chunk ends the row or the warp's range
            if (cc.b + n == cc.kw || cc.u + n == cc.uend) {
                // lane (g, t) holds rows g, g+8 of tokens 2t, 2t+1: v[2h + e]
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float s = 0.f;
#pragma unroll
                    for (int cl = 0; cl < 4; ++cl) {
                        const int d = 133 - tx[q & 1] - 2 * cl, d1 = d / 2;
                        s = __fadd_rn(s, __fmul_rn(__fmul_rn(c[cl][q], __int_as_float((d1 + 127) << 23)),
                                                   __int_as_float((d - d1 + 127) << 23)));
                    }
                    v[q] = s;
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
            if (lane == 0 && pc_on) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                produce(slot);
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
                for (int e = lane; e < N * 16; e += 32) {
                    const int n = e >> 4;
                    v[e] = __fsub_rn(__fsub_rn(opre[hi][n], opre[lo][n]), v[e]);
                }
                __syncwarp();
                if (a.NS == 1 && lo == 0 && hi == P.kw) {
                    store_row_tile(a, r, v, scl + rho * 16, rsm + rho * 16, lane);
                } else if (a.NS == 1) {
                    exchange_row_tile(a, r, v, scl + rho * 16, rsm + rho * 16, lane);
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
                        store_row_tile(a, r, v, scl + rho * 16, rsm + rho * 16, lane);
                        if (lane == 0) a.cnt[r] = 0ull;
                    }
                }
                __syncwarp();
                for (int e = lane; e < RV; e += 32) v[e] = 0.f;   // ready for the next slice
            }
        }
        // (the next slice's staging barrier orders these reads of opre, acc
        // and scl before they are rewritten)
    }
    if (!ok) {
        // a copy never landed: drain what is still in flight (bounded), then leave
        for (int k = 0; k < kSlots; ++k) mbar_wait(bar_w + 8u * k, (phases >> k) & 1u, a.status);
    }
}

using KernelFn = void (*)(GroupArgs);

KernelFn kernel_for(int mode, int nt) {
    const bool A = mode == TL_MODE_BF16;
    switch (nt) {
        case 1: return A ? tl_mma_kernel<true, 1> : tl_mma_kernel<false, 1>;
        case 2: return A ? tl_mma_kernel<true, 2> : tl_mma_kernel<false, 2>;
        case 4: return A ? tl_mma_kernel<true, 4> : tl_mma_kernel<false, 4>;
        default: return A ? tl_mma_kernel<true, 8> : tl_mma_kernel<false, 8>;
    }
}

inline int padded_tokens(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

// ------------------------------------------------------------------ quant
__global__ void __launch_bounds__(256)
tl_quant_kernel(const uint16_t *__restrict__ X, int K, int8_t *__restrict__ Q,
                float *__restrict__ s_out, int32_t *__restrict__ z_out, int symmetric) {
    const int n = blockIdx.x;
    const uint16_t *x = X + (long long)n * K;
    int8_t *q = Q + (long long)n * K;
    float lo = 0.f, hi = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float v = __uint_as_float((uint32_t)x[k] << 16);
        if (symmetric) {
            hi = fmaxf(hi, fabsf(v));
        } else {
            lo = fminf(lo, v);
            hi = fmaxf(hi, v);
        }
    }
    __shared__ float slo[32], shi[32];
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
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
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
        s_out[n] = s;
        z_out[n] = z;
    }
    __syncthreads();
    const float s = s_sh;
    const float zf = (float)z_sh;
    const float qlo = symmetric ? -127.f : -128.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float v = __uint_as_float((uint32_t)x[k] << 16);
        float r = __fadd_rn(rintf(__fdiv_rn(v, s)), zf);
        r = fminf(fmaxf(r, qlo), 127.f);
        q[k] = (int8_t)(int)r;
    }
}

// ------------------------------------------------------------------ host side

struct DeviceInfo {
    int init;     // 0 = unknown, 1 = ok, -1 = unsupported
    int sms;
};
DeviceInfo g_dev[kMaxDevices];

// Dynamic shared memory: weight ring, one slice of X, row accumulators, and
// the rows' scales and row sums.
constexpr size_t dyn_smem(int nt, int kw, int rows) {
    return (size_t)ring_bytes(nt) + (size_t)kw * 128 * nt * 2 + (size_t)rows * 16 * nt * 4 +
           (size_t)rows * 16 * 8;
}

tl_status device_info(DeviceInfo **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TL_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TL_ERR_UNSUPPORTED;
    DeviceInfo &d = g_dev[dev];
    if (d.init == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TL_ERR_CUDA;
        if (major != 10 || minor != 3) {
            d.init = -1;
        } else {
            for (int mode = 0; mode < 2; ++mode)
                for (int nt = 1; nt <= 8; nt *= 2)
                    if (cudaFuncSetAttribute(kernel_for(mode, nt),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dyn_smem(nt, kMaxSlice, kMaxCtaRows)) != cudaSuccess)
                        return TL_ERR_CUDA;
            const tl_status pst = tl_internal::prefill_init_device();
            if (pst != TL_OK) return pst;
            d.sms = sms;
            d.init = 1;
        }
    }
    if (d.init < 0) return TL_ERR_UNSUPPORTED;
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
    const long long Lc = ceil_div(su, pps), LcL = ceil_div(suL, pps);
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
        if (mode == TL_MODE_I8 && !w.rowsum) return TL_ERR_NULL;
        if (w.layout != TL_LAYOUT_TL2P_V2) return TL_ERR_UNSUPPORTED;
        if (w.M < 1 || w.K < 1 || w.M > TL_MAX_M || w.K > TL_MAX_K) return TL_ERR_SHAPE;
        if (w.K != Ws[0].K) return TL_ERR_SHAPE;
        if (!aligned(w.packed, 16) || !aligned(w.scale, 4)) return TL_ERR_ALIGN;
        if (mode == TL_MODE_I8 && !aligned(w.rowsum, 4)) return TL_ERR_ALIGN;
    }
    return TL_OK;
}

size_t workspace_bytes_for(const tl_weight *Ws, int G, int N, int sms) {
    int Ms[TL_MAX_GROUP];
    for (int g = 0; g < G; ++g) Ms[g] = Ws[g].M;
    const int K = Ws[0].K;
    if (tl_internal::prefill_supported(N, K))
        return std::max(tl_internal::prefill_workspace_bytes(Ws, G, N, K, TL_MODE_BF16, sms),
                        tl_internal::prefill_workspace_bytes(Ws, G, N, K, TL_MODE_I8, sms));
    Plan p;
    if (make_plan(Ms, G, K, N, sms, &p) != TL_OK) return 0;
    return p.ws_bytes;
}

tl_status launch_chunk(const tl_weight *Ws, int G, const void *X, const float *s,
                       const int32_t *z, void *const *Ys, int n0, int n, int mode, int out,
                       void *ws, size_t ws_bytes, unsigned flags, cudaStream_t stream,
                       const DeviceInfo &dev) {
    GroupArgs a;
    std::memset(&a, 0, sizeof a);
    int Ms[TL_MAX_GROUP];
    a.G = G;
    a.rt_off[0] = 0;
    const int K = Ws[0].K;
    for (int g = 0; g < G; ++g) {
        a.packed[g] = reinterpret_cast<const char *>(Ws[g].packed);
        a.scale[g] = Ws[g].scale;
        a.rowsum[g] = Ws[g].rowsum;
        a.M[g] = Ms[g] = Ws[g].M;
        const size_t esz = out == TL_OUT_BF16 ? 2 : 4;
        a.Y[g] = static_cast<char *>(Ys[g]) + (size_t)n0 * Ws[g].M * esz;
        a.rt_off[g + 1] = a.rt_off[g] + (int)ceil_div(Ws[g].M, 16);
    }
    Plan p;
    const tl_status pst = make_plan(Ms, G, K, n, dev.sms, &p);
    if (pst != TL_OK) return pst;
    if (!ws || ws_bytes < p.ws_bytes) return TL_ERR_WORKSPACE;
    a.R = p.R; a.KB = p.KB; a.KW = p.KW; a.KWL = p.KWL; a.NS = p.NS; a.K = K; a.U = (int)p.U;
    a.Pps = p.Pps; a.Lc = p.Lc; a.LcL = p.LcL; a.rows = p.rows;
    a.dKW = make_fastdiv((uint32_t)p.KW);
    a.dKWL = make_fastdiv((uint32_t)p.KWL);
    const size_t xsz = mode == TL_MODE_BF16 ? 2 : 1;
    a.X = static_cast<const char *>(X) + (size_t)n0 * K * xsz;
    a.s = s ? s + n0 : nullptr;
    a.z = z ? z + n0 : nullptr;
    a.N = n; a.mode = mode; a.out = out;
    a.xvec = aligned(a.X, 16) && (K % (mode == TL_MODE_BF16 ? 8 : 16)) == 0;
    char *wsb = static_cast<char *>(ws) + tl_internal::kStatusBytes;
    a.cnt = reinterpret_cast<unsigned long long *>(wsb);
    a.xslot = reinterpret_cast<unsigned long long *>(wsb + p.cnt_bytes);
    a.part = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                       tl_internal::scratch_offset(ws_bytes, p.back));
    a.status = static_cast<int *>(ws);

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

}  // namespace

namespace tl_internal {

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
    tl_quant_kernel<<<N, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(X_bf16), K, Q, s, z, symmetric ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

tl_status tl_linear_group(const tl_weight *Ws, int G, const void *X, const float *s,
                          const int32_t *z, void *const *Ys, int N, int mode, int out_dtype,
                          void *workspace, size_t workspace_bytes, unsigned flags,
                          void *stream) {
    tl_status st = check_weights(Ws, G, mode);
    if (st != TL_OK) return st;
    if (mode != TL_MODE_BF16 && mode != TL_MODE_I8) return TL_ERR_MODE;
    if (out_dtype != TL_OUT_F32 && out_dtype != TL_OUT_BF16 && out_dtype != TL_OUT_I32_RAW)
        return TL_ERR_MODE;
    if (out_dtype == TL_OUT_I32_RAW && mode != TL_MODE_I8) return TL_ERR_MODE;
    if (!X || !Ys) return TL_ERR_NULL;
    if (N < 1) return TL_ERR_SHAPE;
    if (mode == TL_MODE_I8 && (!s || !z)) return TL_ERR_NULL;
    if (mode == TL_MODE_BF16 && !aligned(X, 2)) return TL_ERR_ALIGN;
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

tl_status tl_linear(const tl_weight *W, const void *X, const float *s, const int32_t *z, void *Y,
                    int N, int mode, int out_dtype, void *workspace, size_t workspace_bytes,
                    unsigned flags, void *stream) {
    void *Ys[1] = {Y};
    return tl_linear_group(W, 1, X, s, z, Ys, N, mode, out_dtype, workspace, workspace_bytes,
                           flags, stream);
}

}  // extern "C"
